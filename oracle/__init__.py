"""Plain CPU oracle for the batch-invariant NVFP4 W4A4 MoE expert forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path (``nvfp4_moe_expert_gb300``) and imports nothing
from it; both sides are fed by the seeded generators in ``moe_synth``.

The oracle is a slow, literal restatement of what the source pages define:

* page "miniTE diagnoses and narrows the cross-engine execution gap of NVFP4
  RL" (onedev.kr/papers/1404), section "How it differs" (무엇과 다른가): the
  two-level NVFP4 format (E2M1 codes, 16-element E4M3 block scales, FP32 outer
  scales g = max|row| / (6*448)), round-to-nearest-even with no Hadamard and no
  stochastic rounding, the FP32 epilogue multiplying g^x*g^w before the BF16
  cast, and the router probability applied to the SwiGLU activation before FC2;
* the same page, section "How to use it" (어떻게 쓰나): sort + amax, then pad and
  quantise; FC2 maxima taken from the producer of the router-weighted
  activation;
* page "Finishing RL training faster: bitwise consistency, high performance,
  agent-driven" (spke.com/ko/ai/article/3192), section 4.4 "Expert GEMM: two
  layouts, same row result": SiLU(gate)*up in FP32 with one rounding of the
  product; section 4.5 "Cross-GPU reduction": the expert outputs are summed in
  FP32 in top-k slot order; sections 2 and 4.1 (router step, ``router.py``):
  one FP32-output router GEMM for every batch size and a top-k whose ties and
  order are fixed;
* the miniTE page again, sections "How it differs" and its results paragraph
  (``backward.py``): the straight-through backward, BF16 GEMMs on the saved
  BF16 originals, measured by gradient relative L2 against an FP32 reference.

Floating point: FP64 where the contract does not fix the precision (GEMM
accumulation, SiLU), IEEE FP32 (numpy float32, correctly rounded, no FMA
contraction) where it does.

Parity status of each function is stated in its module header; every public
function here is pinned by ``tests/test_oracle_*.py``.
"""

from .formats import (  # noqa: F401
    E2M1_VALUES,
    bf16_bits_to_f32,
    round_to_bf16_bits,
    e2m1_encode,
    e2m1_decode,
    e4m3_encode,
    e4m3_decode,
)
from .quant import (  # noqa: F401
    quantize_rows, dequantize_rows, pack_nibbles, unpack_nibbles, OUTER_DIVISOR,
)
from .router import router_logits_f64, topk_order, topk_probs, router_topk  # noqa: F401
from .backward import moe_backward_ste, forward_saved_activations, silu_and_derivative  # noqa: F401
from .moe import (  # noqa: F401
    route_sort,
    qgemm_f64,
    epilogue_f64,
    dense_swiglu_mlp_f64,
    swiglu_prob,
    combine_slots,
    moe_forward,
    MoEWeightsQ,
    quantize_weights,
)

"""Pins for the oracle's STE backward (oracle/backward.py).  CPU only.

* central finite differences of the unquantised layer (tiny shapes, every
  input element): with the forward's own saved values the STE backward is the
  exact gradient, so a dropped term, a wrong sign or a transposed operand
  anywhere shows;
* float64 torch autograd of the layer written out with torch ops (larger
  shapes; an independent way to the same gradient);
* special cases fixed by the definition: p = 0 (no gradient through FC1),
  h = 0 (no FC2 weight gradient), an expert with no pairs, k = 1 with one
  expert (the dense SwiGLU MLP);
* the BF16-stage variant: every rounded tensor holds BF16 values and stays
  within the rounding bound of the exact gradient.
"""

import numpy as np
import pytest

import moe_synth as S
from oracle import backward as B
from oracle import formats as F


def _case(T, H, I, E, k, seed, empty_expert=None):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    w1 = rng.standard_normal((E, 2 * I, H)) * 0.5
    w2 = rng.standard_normal((E, H, I)) * 0.5
    experts = [e for e in range(E) if e != empty_expert]
    ids = np.stack([rng.choice(experts, k, replace=False) for _ in range(T)])
    p = rng.uniform(0.1, 1.0, (T, k))
    dout = rng.standard_normal((T, H))
    return dout, x, ids, p, w1, w2


def _loss(dout, x, ids, p, w1, w2):
    out, _, _ = B.forward_saved_activations(x, ids, p, w1, w2)
    return float(np.sum(dout * out))


def _grads(dout, x, ids, p, w1, w2, **kw):
    _, gu, h = B.forward_saved_activations(x, ids, p, w1, w2)
    return B.moe_backward_ste(dout, x, ids, p, w1, w2, gu, h, **kw)


def _fd(f, arr, eps=1e-6):
    g = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + eps
        fp = f()
        arr[i] = old - eps
        fm = f()
        arr[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


@pytest.mark.parametrize("T,H,I,E,k,seed", [(3, 5, 4, 3, 2, 0), (4, 6, 3, 4, 3, 1), (2, 4, 2, 1, 1, 2)])
def test_finite_differences(T, H, I, E, k, seed):
    dout, x, ids, p, w1, w2 = _case(T, H, I, E, k, seed)
    g = _grads(dout, x, ids, p, w1, w2)
    f = lambda: _loss(dout, x, ids, p, w1, w2)   # noqa: E731  (reads the arrays the FD perturbs)
    for name, arr in (("dx", x), ("dw1", w1), ("dw2", w2), ("dprob", p)):
        fd = _fd(f, arr)
        err = np.abs(g[name] - fd).max()
        assert err <= 1e-7 * max(1.0, np.abs(fd).max()), (name, err)


def test_torch_autograd():
    torch = pytest.importorskip("torch")
    T, H, I, E, k = 24, 16, 8, 6, 3
    dout, x, ids, p, w1, w2 = _case(T, H, I, E, k, seed=5, empty_expert=2)
    tx, tw1, tw2, tp = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (x, w1, w2, p))
    out = torch.zeros(T, H, dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            g = tw1[e] @ tx[t]
            a, u = g[:I], g[I:]
            hh = a * torch.sigmoid(a) * u * tp[t, j]
            out = out.index_add(0, torch.tensor([t]), (tw2[e] @ hh)[None])
    (out * torch.tensor(dout)).sum().backward()
    g = _grads(dout, x, ids, p, w1, w2)
    for name, ta in (("dx", tx), ("dw1", tw1), ("dw2", tw2), ("dprob", tp)):
        ref = ta.grad.numpy()
        assert np.abs(g[name] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max()), name
    # and the oracle's unquantised forward is the same layer
    got, _, _ = B.forward_saved_activations(x, ids, p, w1, w2)
    assert np.abs(got - out.detach().numpy()).max() <= 1e-12 * np.abs(got).max()


def test_special_cases():
    T, H, I, E, k = 10, 8, 4, 5, 2
    dout, x, ids, p, w1, w2 = _case(T, H, I, E, k, seed=7, empty_expert=3)
    _, gu, h = B.forward_saved_activations(x, ids, p, w1, w2)
    # an expert with no pairs gets exactly zero weight gradients
    g = B.moe_backward_ste(dout, x, ids, p, w1, w2, gu, h)
    assert np.all(g["dw1"][3] == 0) and np.all(g["dw2"][3] == 0)
    # p = 0: nothing flows through SwiGLU into FC1, but dp and dW2 (from the saved h) remain
    g0 = B.moe_backward_ste(dout, x, ids, np.zeros_like(p), w1, w2, gu, h)
    assert np.all(g0["dx"] == 0) and np.all(g0["dw1"] == 0)
    assert np.array_equal(g0["dprob"], g["dprob"]) and np.array_equal(g0["dw2"], g["dw2"])
    # h = 0 saved: no FC2 weight gradient, everything else unchanged
    gh = B.moe_backward_ste(dout, x, ids, p, w1, w2, gu, np.zeros_like(h))
    assert np.all(gh["dw2"] == 0) and np.array_equal(gh["dx"], g["dx"])
    # dOut = 0: every gradient is zero
    gz = B.moe_backward_ste(np.zeros_like(dout), x, ids, p, w1, w2, gu, h)
    assert all(np.all(gz[n] == 0) for n in ("dx", "dw1", "dw2", "dprob"))


def test_dense_mlp_case():
    # one expert, top-1, p = 1: the gradient of the dense SwiGLU MLP, written out by hand
    rng = np.random.default_rng(3)
    T, H, I = 6, 8, 5
    x = rng.standard_normal((T, H))
    w1 = rng.standard_normal((1, 2 * I, H))
    w2 = rng.standard_normal((1, H, I))
    dout = rng.standard_normal((T, H))
    ids = np.zeros((T, 1), np.int64)
    p = np.ones((T, 1))
    g = _grads(dout, x, ids, p, w1, w2)
    a = x @ w1[0, :I].T
    u = x @ w1[0, I:].T
    sig = 1 / (1 + np.exp(-a))
    dh = dout @ w2[0]
    da = dh * u * (sig + a * sig * (1 - sig))
    du = dh * a * sig
    assert np.allclose(g["dx"], np.concatenate([da, du], 1) @ w1[0], rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dw2"][0], dout.T @ (a * sig * u), rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dw1"][0], np.concatenate([da, du], 1).T @ x, rtol=1e-12, atol=1e-12)


def test_bf16_stages_bound():
    cfg = S.LayerConfig("bwd_pin", H=64, I=32, E=4, k=2, T=40, seed=9)
    xb = S.make_x(cfg)
    w1b, w2b = S.make_weights(cfg)
    ids, p = S.make_routing(cfg)
    db = S.make_grad_out(cfg)
    x, w1, w2, dout = (F.bf16_bits_to_f32(a).astype(np.float64) for a in (xb, w1b, w2b, db))
    _, gu, h = B.forward_saved_activations(x, ids, p, w1, w2)
    ex = B.moe_backward_ste(dout, x, ids, p, w1, w2, gu, h)
    st = B.moe_backward_ste(dout, x, ids, p, w1, w2, gu, h, bf16_stages=True)
    for name in ("dh", "dgu", "dx_slots", "dx"):
        v = st[name]
        assert np.array_equal(v, B._bf16(v)), name          # BF16 values
    # each BF16 stage adds at most a relative 2^-8 per element (rms about 2^-9/sqrt(3));
    # dX passes four of them
    u = 2.0 ** -9 / np.sqrt(3)
    for name, stages in (("dh", 1), ("dgu", 2), ("dx", 4), ("dw1", 2), ("dprob", 1)):
        rel = np.linalg.norm(st[name] - ex[name]) / np.linalg.norm(ex[name])
        assert 0 < rel <= 2 * np.sqrt(stages) * u, (name, rel)
    assert np.array_equal(st["dw2"], ex["dw2"])               # dW2 needs no rounded tensor


def test_silu_derivative_closed_forms():
    # sigma(0) = 1/2; sigma(ln 3) = 3/4; sigma(-ln 3) = 1/4; the limits 0 and 1
    a = np.array([0.0, np.log(3.0), -np.log(3.0), 40.0, -40.0])
    silu, d = B.silu_and_derivative(a)
    want_silu = np.array([0.0, 0.75 * np.log(3.0), -0.25 * np.log(3.0), 40.0, 0.0])
    want_d = np.array([0.5, 0.75 * (1 + 0.25 * np.log(3.0)), 0.25 * (1 - 0.75 * np.log(3.0)), 1.0, 0.0])
    assert np.allclose(silu, want_silu, rtol=1e-15, atol=1e-15)
    assert np.allclose(d, want_d, rtol=1e-15, atol=1e-15)
    # and the derivative is the slope of silu
    x = np.linspace(-8, 8, 161)
    eps = 1e-6
    fd = (B.silu_and_derivative(x + eps)[0] - B.silu_and_derivative(x - eps)[0]) / (2 * eps)
    assert np.abs(B.silu_and_derivative(x)[1] - fd).max() < 1e-8

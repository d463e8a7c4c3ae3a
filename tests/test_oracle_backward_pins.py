"""Pins of the oracle's training backward against what the pages and calculus fix.

The attention gradient is tied to (a) central finite differences of the pinned
forward oracle, (b) PyTorch autograd of a dense masked softmax attention whose
mask is the glossary's W=4 table (window rows) and the causal triangle (routed
rows), and (c) closed forms and conservation laws of softmax attention.  The
router gradient is tied to autograd of the report's straight-through gate
written literally, sigma = 1(sigmoid(R) > 0.5) + sigmoid(R) - sg(sigmoid(R)),
with the adaptive weight gamma held fixed (a coefficient, like NLL).
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _case(seed, B=1, N=13, Hq=4, Hkv=2, d=8, frac=0.4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N, Hq, d))
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    do = rng.standard_normal((B, N, Hq, d))
    gate = (rng.random((B, N)) < frac).astype(np.uint8)
    return q, k, v, do, gate


# --------------------------------------------------------------------------
# (a) finite differences of the forward oracle
# --------------------------------------------------------------------------
@pytest.mark.parametrize("W", [1, 4, 30])
def test_gradient_matches_finite_differences(W):
    q, k, v, do, gate = _case(11 + W)
    scale = 0.31

    def loss(q_, k_, v_):
        return float((oracle.prefill(q_, k_, v_, gate, W, scale) * do).sum())

    dq, dk, dv = oracle.prefill_backward(q, k, v, gate, do, W, scale)
    h = 1e-5
    for which, (arr, grad) in enumerate(((q, dq), (k, dk), (v, dv))):
        for idx in np.ndindex(arr.shape):
            args_p, args_m = [q, k, v], [q, k, v]
            a_p, a_m = arr.copy(), arr.copy()
            a_p[idx] += h
            a_m[idx] -= h
            args_p[which], args_m[which] = a_p, a_m
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) < 1e-8 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


# --------------------------------------------------------------------------
# (b) autograd of a dense masked attention built from the glossary's table
# --------------------------------------------------------------------------
def _golden_window_mask():
    rows, W, N = [], None, None
    with open(os.path.join(GOLDEN, "swa_w4_n7_mask.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("# W"):
                W = int(line.split()[2])
            elif line.startswith("# N"):
                N = int(line.split()[2])
            elif line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return W, N, np.array(rows, dtype=bool)


def _dense_grads(q, k, v, do, mask, scale):
    """Autograd of softmax(scale QK^T masked) V per (b, head); mask [B,N,N]."""
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kk = kt.repeat_interleave(G, dim=2)
    vv = vt.repeat_interleave(G, dim=2)
    s = torch.einsum("bihc,bjhc->bhij", qt, kk) * scale
    s = s.masked_fill(~torch.tensor(mask)[:, None], float("-inf"))
    o = torch.einsum("bhij,bjhc->bihc", torch.softmax(s, dim=-1), vv)
    (o * torch.tensor(do)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def test_gradient_matches_autograd_on_w4_table():
    W, N, table = _golden_window_mask()
    q, k, v, do, gate = _case(5, B=2, N=N, Hq=4, Hkv=2, d=6, frac=0.5)
    causal = np.tril(np.ones((N, N), dtype=bool))
    mask = np.where(gate[:, :, None] != 0, causal[None], table[None])
    ref = _dense_grads(q, k, v, do, mask, 0.4)
    got = oracle.prefill_backward(q, k, v, gate, do, W, 0.4)
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g, r, rtol=0, atol=1e-12)


def test_gradient_matches_autograd_larger_window():
    N, W = 37, 6
    q, k, v, do, gate = _case(6, B=1, N=N, Hq=6, Hkv=3, d=5, frac=0.3)
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    window = (j <= i) & (j > i - W)
    mask = np.where(gate[:, :, None] != 0, (j <= i)[None], window[None])
    ref = _dense_grads(q, k, v, do, mask, 0.2)
    got = oracle.prefill_backward(q, k, v, gate, do, W, 0.2)
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g, r, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# (c) closed forms and conservation laws
# --------------------------------------------------------------------------
def test_window_one_gradient_closed_form():
    """W=1, window rows: o_i = v_i, so dV = dO summed over the head group and
    dQ = dK = 0 exactly."""
    q, k, v, do, _ = _case(7, B=2, N=9, Hq=4, Hkv=2, d=8)
    gate = np.zeros((2, 9), np.uint8)
    dq, dk, dv = oracle.prefill_backward(q, k, v, gate, do, 1, 0.5)
    assert not dq.any() and not dk.any()
    np.testing.assert_array_equal(dv, do.reshape(2, 9, 2, 2, 8).sum(axis=3))


def test_constant_values_give_no_score_gradient():
    """Every v_j equal: the output is that vector whatever the weights, so
    dQ and dK vanish."""
    q, k, _, do, gate = _case(8)
    v = np.broadcast_to(_rand((1, 1, 2, 8), 9), (1, 13, 2, 8)).copy()
    dq, dk, _ = oracle.prefill_backward(q, k, v, gate, do, 4, 0.7)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


def test_conservation_laws():
    """Softmax weights sum to 1 per row: sum_j dV_j = sum_i dO_i (per head
    group), and sum_j dS_ij = 0 per row, so sum_j dK_j = 0."""
    q, k, v, do, gate = _case(10, B=2, N=21, Hq=6, Hkv=2, d=7)
    dq, dk, dv = oracle.prefill_backward(q, k, v, gate, do, 5, 0.3)
    np.testing.assert_allclose(dv.sum(axis=1), do.reshape(2, 21, 2, 3, 7).sum(axis=(1, 3)),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, rtol=0, atol=1e-12)


def test_window_ge_n_equals_full_gradient():
    """The glossary's FAQ: W = N is causal attention, so gates make no
    difference to the gradient either."""
    q, k, v, do, gate = _case(12, N=11)
    a = oracle.prefill_backward(q, k, v, np.zeros_like(gate), do, 11, 0.3)
    b = oracle.prefill_backward(q, k, v, np.ones_like(gate), do, 11, 0.3)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_sampled_rows_and_keys_match_full():
    q, k, v, do, gate = _case(13, B=2, N=17, Hq=4, Hkv=2, d=6)
    dq, dk, dv = oracle.prefill_backward(q, k, v, gate, do, 3, 0.4)
    rows = [(0, 0, 0), (1, 16, 3), (0, 9, 2), (1, 4, 1)]
    got = oracle.prefill_backward_rows(q, k, v, gate, do, 3, 0.4, rows)
    np.testing.assert_allclose(got, np.stack([dq[b, i, h] for b, i, h in rows]), atol=1e-13)
    keys = [(0, 0, 0), (1, 16, 1), (0, 7, 1), (1, 2, 0)]
    gk, gv = oracle.prefill_backward_keys(q, k, v, gate, do, 3, 0.4, keys)
    np.testing.assert_allclose(gk, np.stack([dk[b, j, h] for b, j, h in keys]), atol=1e-13)
    np.testing.assert_allclose(gv, np.stack([dv[b, j, h] for b, j, h in keys]), atol=1e-13)


# --------------------------------------------------------------------------
# Router backward: the straight-through gate and the regulariser
# --------------------------------------------------------------------------
def _ste_autograd(h, w, b, o_full, o_swa, do, gamma, d_reg):
    ht, wt, bt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (h, w, [b]))
    r = ht @ wt + bt
    soft = torch.sigmoid(r)
    sigma = (soft > 0.5).double() + soft - soft.detach()
    of, os_ = torch.tensor(o_full), torch.tensor(o_swa)
    o = sigma[:, None] * of + (1 - sigma[:, None]) * os_
    reg = torch.tensor(gamma) * torch.nn.functional.softplus(r)
    r.retain_grad()
    ((o * torch.tensor(do)).sum() + (torch.tensor(d_reg) * reg).sum()).backward()
    return r.grad.numpy(), ht.grad.numpy(), wt.grad.numpy(), float(bt.grad[0])


def test_route_backward_matches_straight_through_autograd():
    rng = np.random.default_rng(21)
    T, D, HD = 23, 16, 12
    h = rng.standard_normal((T, D))
    w = rng.standard_normal(D) / 4
    b = 0.1
    o_full, o_swa, do = (rng.standard_normal((T, HD)) for _ in range(3))
    gamma = rng.random(T) * 1e-2
    d_reg = rng.standard_normal(T)
    logits = h @ w + b
    ref = _ste_autograd(h, w, b, o_full, o_swa, do, gamma, d_reg)
    got = oracle.route_backward(logits, o_full, o_swa, do, gamma, d_reg, h, w)
    np.testing.assert_allclose(got["d_logits"], ref[0], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(got["dh"], ref[1], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(got["dw"], ref[2], rtol=1e-12, atol=1e-15)
    assert abs(got["db"] - ref[3]) < 1e-12 * max(1.0, abs(ref[3]))


def test_route_backward_inside_window_is_regulariser_only():
    """For t < W both branches visit [0, t], so o_FULL = o_SWA and the
    straight-through term vanishes: d_logit = d_reg * gamma * sigmoid(logit).
    At logit 0 with NLL = mse = 0, gamma = 1e-3 / 0.1 = 1e-2 and sigmoid = 1/2."""
    rng = np.random.default_rng(22)
    B, N, Hq, Hkv, d, W = 1, 10, 2, 2, 4, 16
    q = rng.standard_normal((B, N, Hq, d))
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    logits = np.zeros((B, N))
    nll = np.zeros((B, N))
    out = oracle.dual(q, k, v, logits, nll, W, 0.5)
    np.testing.assert_array_equal(out["o_full"], out["o_swa"])
    do = rng.standard_normal((B * N, Hq * d))
    d_reg = rng.standard_normal(B * N)
    got = oracle.route_backward(logits.ravel(), out["o_full"].reshape(B * N, -1),
                                out["o_swa"].reshape(B * N, -1), do, out["gamma"].ravel(), d_reg)
    assert np.all(out["gamma"] == 1e-2)
    np.testing.assert_allclose(got["d_logits"], d_reg * 5e-3, rtol=1e-15, atol=0)


def test_route_backward_without_regulariser():
    """No regulariser gradient: d_logit = s(1-s) <dO, o_FULL - o_SWA>, which at
    logit 0 is a quarter of the inner product."""
    rng = np.random.default_rng(23)
    of, os_, do = (rng.standard_normal((5, 7)) for _ in range(3))
    got = oracle.route_backward(np.zeros(5), of, os_, do, np.ones(5))
    np.testing.assert_allclose(got["d_logits"], 0.25 * (do * (of - os_)).sum(axis=1),
                               rtol=1e-15)

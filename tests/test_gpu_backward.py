"""GPU parity of the training backward (swiattn_prefill_backward,
swiattn_route_backward) against the fp64 oracle, through the C ABI.

Tolerances.  fp32 paths: max-abs 1e-4 (scaled by max(1, max|ref|)), as for the
forward.  bf16 paths, derived from the arithmetic: the gradients are stored
as bf16 (a relative rounding error of up to 2^-8 = 3.9e-3 per element, about
1.4e-3 on average), and the kernels round P and dS to bf16 before the
tensor-core contractions, with D_i = dO_i.O_i taken from the bf16 output.  The
bound is max|err| <= 1e-2 * max|ref| (about 2.5 bf16 steps at the largest
element) and mean|err| <= 4e-3 * mean|ref| (about one step on average).
The router backward feeds on bf16 branch outputs whose difference
o_FULL - o_SWA cancels leading bits, and rounds dh once more: mean bound
6e-3 * mean|ref| there.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swiattn_inputs as inp

pytestmark = pytest.mark.gpu

REL_MAX, REL_MEAN, ROUTE_REL_MEAN, F32_TOL = 1e-2, 4e-3, 6e-3, 1e-4


@pytest.fixture(scope="module")
def swa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_router_gb300 as m
    return m


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def assert_rel_close(got, ref, what, rel_mean=REL_MEAN):
    g, r = f64(got).reshape(np.shape(ref)), np.asarray(ref)
    err = np.abs(g - r)
    assert err.max() <= REL_MAX * np.abs(r).max(), (what, err.max(), np.abs(r).max())
    assert err.mean() <= rel_mean * np.abs(r).mean(), (what, err.mean(), np.abs(r).mean())


def assert_f32_close(got, ref, what):
    r = np.asarray(ref)
    err = np.abs(f64(got).reshape(r.shape) - r)
    assert err.max() <= F32_TOL * max(1.0, np.abs(r).max()), (what, err.max())


def make_case(B, N, Hq, Hkv, d, dtype, seed, frac=None, gates=None):
    g = inp._gen(seed)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, d, dtype, g)
    if gates is not None:
        gate = gates
    elif frac in (0, 1):
        gate = torch.full((B, N), int(frac), dtype=torch.uint8)
    else:
        gate = torch.stack([inp.run_gates(N, frac, g) for _ in range(B)])
    do = inp.output_grad((B, N, Hq, d), dtype, seed + 1000)
    return q, k, v, gate, do


def gpu_backward(swa, q, k, v, gate, do, W):
    qd, kd, vd, gd, dod = (t.cuda() for t in (q, k, v, gate, do))
    o, lse = swa.prefill(qd, kd, vd, gd, W, want_lse=True)
    grads = swa.prefill_backward(qd, kd, vd, gd, o, lse, dod, W)
    assert swa.get_device_error() == 0
    return grads


def oracle_backward(q, k, v, gate, do, W):
    d = q.shape[-1]
    return oracle.prefill_backward(f64(q), f64(k), f64(v), gate.numpy(), f64(do), W,
                                   1.0 / math.sqrt(d))


# (B, N, Hq, Hkv, W, gates): several tiles, ragged tails, GQA, every gate mix.
BF16_CASES = [
    (1, 1000, 4, 2, 256, 0.3),     # ragged N, GQA 2, routed runs
    (2, 777, 2, 2, 100, 0.13),     # batch 2, W not a multiple of the tile
    (1, 300, 2, 1, 64, 1),         # every row routed
    (1, 300, 2, 2, 64, 0),         # pure sliding window
    (1, 100, 2, 2, 1000, 0.5),     # N < one tile, W >= N
    (1, 129, 4, 4, 128, 0.5),      # one row past a tile
    (1, 2048, 16, 4, 1024, 0.5),   # the dual-branch head layout, W = 1024
]


@pytest.mark.parametrize("B,N,Hq,Hkv,W,frac", BF16_CASES)
def test_backward_bf16_matches_oracle(swa, B, N, Hq, Hkv, W, frac):
    q, k, v, gate, do = make_case(B, N, Hq, Hkv, 128, torch.bfloat16, seed=N + W, frac=frac)
    dq, dk, dv = gpu_backward(swa, q, k, v, gate, do, W)
    rq, rk, rv = oracle_backward(q, k, v, gate, do, W)
    assert_rel_close(dq, rq, "dq")
    assert_rel_close(dk, rk, "dk")
    assert_rel_close(dv, rv, "dv")


@pytest.mark.parametrize("N,Hq,Hkv,d,W,frac", [(256, 2, 2, 64, 32, 0.13), (300, 4, 2, 128, 50, 0.3),
                                                (130, 2, 1, 64, 1, 0.5)])
def test_backward_fp32_matches_oracle(swa, N, Hq, Hkv, d, W, frac):
    q, k, v, gate, do = make_case(1, N, Hq, Hkv, d, torch.float32, seed=7 + N, frac=frac)
    dq, dk, dv = gpu_backward(swa, q, k, v, gate, do, W)
    rq, rk, rv = oracle_backward(q, k, v, gate, do, W)
    assert_f32_close(dq, rq, "dq")
    assert_f32_close(dk, rk, "dk")
    assert_f32_close(dv, rv, "dv")


def test_backward_tiny_fp32_config(swa):
    """The tiny fp32 workload (N=256, H=2, d=64, W=32, Bernoulli(0.13) gates)."""
    c = inp.tiny_fp32(seed=0)
    do = inp.output_grad(c["q"].shape, torch.float32, 1)
    dq, dk, dv = gpu_backward(swa, c["q"], c["k"], c["v"], c["gate"], do, c["W"])
    rq, rk, rv = oracle_backward(c["q"], c["k"], c["v"], c["gate"], do, c["W"])
    assert_f32_close(dq, rq, "dq")
    assert_f32_close(dk, rk, "dk")
    assert_f32_close(dv, rv, "dv")


def test_backward_window_one_bf16(swa):
    """W = 1, window rows, one query head per KV head: each row attends to
    itself with weight exactly 1 after bf16 rounding, so dv equals dO bit for
    bit; dq and dk are sums of near-cancelling terms (dP_ii - D_i)."""
    q, k, v, gate, do = make_case(1, 333, 2, 2, 128, torch.bfloat16, seed=3, frac=0)
    dq, dk, dv = gpu_backward(swa, q, k, v, gate, do, 1)
    assert torch.equal(dv.cpu(), do)
    assert dq.abs().max().item() < 1e-3 and dk.abs().max().item() < 1e-3


def test_backward_deterministic(swa):
    q, k, v, gate, do = make_case(1, 1500, 4, 2, 128, torch.bfloat16, seed=9, frac=0.2)
    qd, kd, vd, gd, dod = (t.cuda() for t in (q, k, v, gate, do))
    o, lse = swa.prefill(qd, kd, vd, gd, 256, want_lse=True)
    a = swa.prefill_backward(qd, kd, vd, gd, o, lse, dod, 256)
    b = swa.prefill_backward(qd, kd, vd, gd, o, lse, dod, 256)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def _sampled_check(swa, q, k, v, gate, do, W, rows, keys):
    dq, dk, dv = gpu_backward(swa, q, k, v, gate, do, W)
    d = q.shape[-1]
    args = (f64(q), f64(k), f64(v), gate.numpy(), f64(do), W, 1.0 / math.sqrt(d))
    rq = oracle.prefill_backward_rows(*args, rows)
    gq = torch.stack([dq[b, i, h] for b, i, h in rows])
    assert_rel_close(gq, rq, "dq rows")
    rk, rv = oracle.prefill_backward_keys(*args, keys)
    assert_rel_close(torch.stack([dk[b, j, h] for b, j, h in keys]), rk, "dk keys")
    assert_rel_close(torch.stack([dv[b, j, h] for b, j, h in keys]), rv, "dv keys")


def test_backward_dual_8k_sampled(swa):
    """Full-size training workload: B=2, N=8192, GQA 16/4, W=1024, gates from
    the router logits (logit > 0, about half the tokens), dO ~ N(0,1)."""
    c = inp.dual_8k(seed=0)
    gate = (c["logits"] > 0).to(torch.uint8)
    do = inp.output_grad(c["q"].shape, torch.bfloat16, 1)
    rng = np.random.default_rng(0)
    N, W = c["N"], c["W"]
    rows = [(0, 0, 0), (1, N - 1, 15), (0, W - 1, 3), (1, W, 4)]
    rows += [(int(rng.integers(2)), int(rng.integers(N)), int(rng.integers(16))) for _ in range(28)]
    keys = [(0, 0, 0), (1, N - 1, 3), (0, 4000, 1), (1, int(rng.integers(N)), 2)]
    _sampled_check(swa, c["q"], c["k"], c["v"], gate, do, W, rows, keys)


def test_backward_prefill_32k_sampled(swa):
    """Long-context prefill workload (N=32768, H=16, routed fraction 0.13)."""
    c = inp.prefill_32k(frac=0.13, seed=0)
    do = inp.output_grad(c["q"].shape, torch.bfloat16, 2)
    rng = np.random.default_rng(1)
    N = c["N"]
    routed = np.nonzero(c["gate"].numpy()[0])[0]
    rows = [(0, 0, 0), (0, N - 1, 15), (0, int(routed[-1]), 7)]
    rows += [(0, int(rng.integers(N)), int(rng.integers(16))) for _ in range(13)]
    keys = [(0, 0, 0), (0, N - 1, 9), (0, 20000, 3)]
    _sampled_check(swa, c["q"], c["k"], c["v"], c["gate"], do, c["W"], rows, keys)


# ------------------------------------------------------------ router -------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_route_backward_matches_oracle(swa, dtype):
    g = inp._gen(9)
    B, N, Hq, Hkv, d, W = 1, 300, 4, 2, 128, 64
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, d, dtype, g)
    logits = inp.logits_with_margin((B, N), g)
    nll = torch.rand(B, N, generator=g) * 3
    r = inp.router_inputs(B * N, 256, dtype, 10)
    do = inp.output_grad((B, N, Hq, d), dtype, 11)
    d_reg = torch.randn(B * N, generator=g)
    outs = swa.dual_branch(q.cuda(), k.cuda(), v.cuda(), logits.cuda(), nll.cuda(), W)
    got = swa.route_backward(logits.cuda().reshape(-1), outs["o_full"], outs["o_swa"], do.cuda(),
                             outs["gamma"].reshape(-1), d_reg.cuda(), r["h"].cuda(), r["w"].cuda())
    assert swa.get_device_error() == 0
    od = oracle.dual(f64(q), f64(k), f64(v), f64(logits), f64(nll), W, 1.0 / math.sqrt(d))
    ref = oracle.route_backward(f64(logits).ravel(), od["o_full"].reshape(B * N, -1),
                                od["o_swa"].reshape(B * N, -1), f64(do).reshape(B * N, -1),
                                od["gamma"].ravel(), f64(d_reg), f64(r["h"]), f64(r["w"]))
    if dtype == torch.float32:
        for name in ("d_logits", "dh", "dw"):
            assert_f32_close(got[name], ref[name], name)
        assert abs(got["db"].item() - ref["db"]) <= F32_TOL * max(1.0, abs(ref["db"]))
    else:
        for name in ("d_logits", "dh", "dw"):
            assert_rel_close(got[name], ref[name], name, ROUTE_REL_MEAN)
        assert abs(got["db"].item() - ref["db"]) <= REL_MAX * max(1.0, abs(ref["db"]))


def test_route_backward_optional_outputs(swa):
    """No regulariser term and no linear-map gradients: d_logits alone, equal
    to a quarter of <dO, o_FULL - o_SWA> at logit 0 (sigmoid'(0) = 1/4)."""
    g = inp._gen(12)
    of, os_, do = (inp.randn((64, 256), torch.float32, g) for _ in range(3))
    logits = torch.zeros(64)
    got = swa.route_backward(logits.cuda(), of.cuda(), os_.cuda(), do.cuda())
    assert set(got) == {"d_logits"}
    ref = oracle.route_backward(np.zeros(64), f64(of), f64(os_), f64(do), np.ones(64))
    assert_f32_close(got["d_logits"], ref["d_logits"], "d_logits")
    np.testing.assert_allclose(ref["d_logits"], 0.25 * (f64(do) * (f64(of) - f64(os_))).sum(1),
                               rtol=1e-12)


# -------------------------------------------------------- training step ----
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_training_step_through_the_library(swa, dtype):
    """One training step of a SwiAttn layer through the C ABI: router ->
    dual-branch forward (gated output and its lse) -> routed attention
    backward from o_gated / lse_gated, and router backward through the
    straight-through gate and the regulariser; every gradient against the
    oracle's."""
    g = inp._gen(90)
    B, N, Hq, Hkv, d, W, D = 1, 600, 4, 2, 128, 128, 256
    r = inp.router_inputs(B * N, D, dtype, 91, frac=0.3)
    h, w, bias = r["h"], r["w"], r["bias"]
    for _ in range(10):   # keep every logit at least 1e-3 from the threshold
        lg0, _ = oracle.route(f64(h), f64(w), bias)
        bad = np.nonzero(np.abs(lg0) < 1e-3)[0]
        if bad.size == 0:
            break
        inp.redraw_rows(h, bad, r["gen"])
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, d, dtype, g)
    nll = torch.rand(B, N, generator=g) * 3
    do = inp.output_grad((B, N, Hq, d), dtype, 92)
    d_reg = torch.ones(B * N)
    logits, gate = swa.route(h.cuda(), w.cuda(), bias)
    gate2 = gate.view(B, N)
    out = swa.dual_branch(q.cuda(), k.cuda(), v.cuda(), logits.view(B, N), nll.cuda(), W,
                          want_lse=True)
    dq, dk, dv = swa.prefill_backward(q.cuda(), k.cuda(), v.cuda(), gate2, out["o_gated"],
                                      out["lse_gated"], do.cuda(), W)
    rb = swa.route_backward(logits, out["o_full"], out["o_swa"], do.cuda(),
                            out["gamma"].view(-1), d_reg.cuda(), h.cuda(), w.cuda())
    assert swa.get_device_error() == 0
    # oracle: its own router logits and gates, its own branch outputs
    ref_logits, ref_gate = oracle.route(f64(h), f64(w), bias)
    assert np.abs(ref_logits).min() >= 1e-3
    np.testing.assert_array_equal(gate.cpu().numpy(), ref_gate)
    scale = 1.0 / math.sqrt(d)
    od = oracle.dual(f64(q), f64(k), f64(v), ref_logits.reshape(B, N), f64(nll), W, scale)
    rq, rk, rv = oracle.prefill_backward(f64(q), f64(k), f64(v), ref_gate.reshape(B, N), f64(do),
                                         W, scale)
    rr = oracle.route_backward(ref_logits, od["o_full"].reshape(B * N, -1),
                               od["o_swa"].reshape(B * N, -1), f64(do).reshape(B * N, -1),
                               od["gamma"].ravel(), f64(d_reg), f64(h), f64(w))
    if dtype == torch.float32:
        for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv"),
                               (rb["d_logits"], rr["d_logits"], "d_logits"),
                               (rb["dh"], rr["dh"], "dh"), (rb["dw"], rr["dw"], "dw")):
            assert_f32_close(got, ref, name)
    else:
        for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
            assert_rel_close(got, ref, name)
        for got, ref, name in ((rb["d_logits"], rr["d_logits"], "d_logits"),
                               (rb["dh"], rr["dh"], "dh"), (rb["dw"], rr["dw"], "dw")):
            assert_rel_close(got, ref, name, ROUTE_REL_MEAN)
    # lse_gated is the gated branch's log-sum-exp
    ref_o, ref_lse = oracle.prefill(f64(q), f64(k), f64(v), ref_gate.reshape(B, N), W, scale,
                                    want_lse=True)
    assert np.abs(f64(out["lse_gated"]) - ref_lse).max() <= 1e-3

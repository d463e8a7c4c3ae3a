"""GPU parity over seeded random shapes: many small configurations of the
routed prefill (with and without global anchors), the decode, the dual
branch and the training backward, drawn from one fixed generator, each compared element by element with
the fp64 oracle.  The fixed cases of the other test files pick the edges by
hand; these cover the space between them (batch counts, GQA ratios, window
sizes, sequence lengths that are not multiples of the tile sizes, gate run
lengths and fractions).

A test repeats a call made of tiny band and far items many times, each call
checked for an expired device-side wait; others cover a work list where most
far pairs are split into one-tile items, and far-row counts at the edges of
the far tiling (prefill and backward).

Tolerances as elsewhere: bf16 attention outputs max-abs 2e-2 and mean-abs
2e-3; fp32 outputs 1e-4; the visited-key count of every (row, head) exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swiattn_inputs as inp

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, F32_TOL = 2e-2, 2e-3, 1e-4
N_CASES = 12


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


def draw(rng, choices):
    return choices[int(rng.integers(len(choices)))]


def prefill_cases():
    rng = np.random.default_rng(20261203)
    cases = []
    for c in range(N_CASES):
        B = draw(rng, [1, 2, 3])
        Hkv = draw(rng, [1, 2, 4])
        G = draw(rng, [1, 2, 4])
        N = int(rng.integers(1, 1800))
        W = int(rng.integers(1, 700))
        frac = float(draw(rng, [0.0, 0.05, 0.3, 0.7, 1.0]))
        run = float(draw(rng, [1.0, 8.0, 64.0, 300.0]))
        S = draw(rng, [0, 0, 1, 64, 256])
        cases.append((c, B, N, Hkv * G, Hkv, W, frac, run, S))
    return cases


@pytest.mark.parametrize("case", prefill_cases(), ids=lambda c: f"p{c[0]}")
def test_prefill_random_shapes(swa, case):
    c, B, N, Hq, Hkv, W, frac, run, S = case
    g = inp._gen(5000 + c)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    gate = torch.stack([inp.run_gates(N, frac, g, mean_run=run) if 0 < frac < 1 else
                        torch.full((N,), int(frac), dtype=torch.uint8) for _ in range(B)])
    scale = 1 / math.sqrt(128)
    o, lse = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W, scale, n_anchor=S,
                         want_lse=True)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    if S:
        ref = oracle.prefill_anchored(f64(q), f64(k), f64(v), gate.numpy(), W, S, scale)
    else:
        ref = oracle.prefill(f64(q), f64(k), f64(v), gate.numpy(), W, scale)
    err = np.abs(f64(o) - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (case, err.max(), err.mean())
    # With q = 0 every visited key weighs the same, so exp(lse) counts them.
    o0, lse0 = swa.prefill(torch.zeros_like(q).cuda(), k.cuda(), v.cuda(), gate.cuda(), W, scale,
                           n_anchor=S, want_lse=True)
    torch.cuda.synchronize()
    i = np.arange(N)[None, :]
    routed = gate.numpy() != 0
    lo = np.where(routed, 0, np.maximum(0, i - W + 1))
    count = i - lo + 1 + np.where(routed, 0, np.clip(np.minimum(S, i - W + 1), 0, None))
    got = np.rint(np.exp(f64(lse0))).astype(np.int64)
    np.testing.assert_array_equal(got, np.repeat(count[..., None], Hq, -1))


def decode_cases():
    rng = np.random.default_rng(20261204)
    cases = []
    for c in range(N_CASES):
        B = draw(rng, [1, 3, 7, 33])
        Hkv = draw(rng, [1, 2, 4, 8])
        G = draw(rng, [1, 2, 4, 8])
        d = draw(rng, [64, 128])
        dtype = draw(rng, ["bf16", "bf16", "f32"])
        Lmax = int(rng.integers(1, 3000))
        W = int(rng.integers(1, 1200))
        S = draw(rng, [0, 0, 16, 256])
        cases.append((c, B, Lmax, Hkv * G, Hkv, d, W, dtype, S))
    return cases


@pytest.mark.parametrize("case", decode_cases(), ids=lambda c: f"d{c[0]}")
def test_decode_random_shapes(swa, case):
    c, B, Lmax, Hq, Hkv, d, W, dtype, S = case
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = inp._gen(6000 + c)
    kc = inp.randn((B, Lmax, Hkv, d), tdt, g)
    vc = inp.randn((B, Lmax, Hkv, d), tdt, g)
    q = inp.randn((B, Hq, d), tdt, g)
    sl = torch.randint(1, Lmax + 1, (B,), generator=g, dtype=torch.int32)
    gate = inp.bernoulli_gates((B,), 0.3, g)
    scale = 1 / math.sqrt(d)
    args = [t.cuda() for t in (q, kc, vc, sl, gate)]
    try:
        if S:
            o = swa.decode_anchored(*args, W, S, scale)
        else:
            o = swa.decode(*args, W, scale)
    except swa.SwiAttnError as e:
        # a token row too wide for the split kernel's block is refused
        assert e.status == 2, (case, str(e))
        return
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    if S:
        ref = oracle.decode_anchored(f64(q), f64(kc), f64(vc), sl.numpy(), gate.numpy(), W, S, scale)
    else:
        ref = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), gate.numpy(), W, scale)
    err = np.abs(f64(o) - ref)
    if dtype == "f32":
        assert err.max() <= F32_TOL, (case, err.max())
    else:
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (case, err.max(), err.mean())


def dual_cases():
    rng = np.random.default_rng(20261205)
    cases = []
    for c in range(6):
        B = draw(rng, [1, 2])
        Hkv = draw(rng, [1, 2, 4])
        G = draw(rng, [1, 2, 4])
        N = int(rng.integers(1, 1500))
        W = int(rng.integers(1, 600))
        cases.append((c, B, N, Hkv * G, Hkv, W))
    return cases


@pytest.mark.parametrize("case", dual_cases(), ids=lambda c: f"u{c[0]}")
def test_dual_random_shapes(swa, case):
    c, B, N, Hq, Hkv, W = case
    g = inp._gen(7000 + c)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    logits = inp.logits_with_margin((B, N), g)
    nll = torch.rand(B, N, generator=g) * 3
    scale = 1 / math.sqrt(128)
    out = swa.dual_branch(q.cuda(), k.cuda(), v.cuda(), logits.cuda(), nll.cuda(), W, scale)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ref = oracle.dual(f64(q), f64(k), f64(v), f64(logits), f64(nll), W, scale)
    for name in ("o_full", "o_swa"):
        err = np.abs(f64(out[name]) - ref[name])
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (case, name, err.max(), err.mean())


def backward_cases():
    rng = np.random.default_rng(20261206)
    cases = []
    for c in range(6):
        B = draw(rng, [1, 2])
        Hkv = draw(rng, [1, 2, 4])
        G = draw(rng, [1, 2, 4])
        N = int(rng.integers(2, 900))
        W = int(rng.integers(1, 500))
        frac = float(draw(rng, [0.0, 0.13, 0.5, 1.0]))
        cases.append((c, B, N, Hkv * G, Hkv, W, frac))
    return cases


@pytest.mark.parametrize("case", backward_cases(), ids=lambda c: f"b{c[0]}")
def test_backward_random_shapes(swa, case):
    """dQ, dK, dV of the routed prefill (bf16 tensor-core kernels) against the
    oracle's gradient.  Tolerance as in the backward tests: the gradients are
    stored as bf16 and P, dS are rounded to bf16 before the contractions, so
    max|err| <= 1e-2 max|ref| and mean|err| <= 4e-3 mean|ref|."""
    c, B, N, Hq, Hkv, W, frac = case
    g = inp._gen(8000 + c)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    gate = torch.stack([inp.run_gates(N, frac, g) if 0 < frac < 1 else
                        torch.full((N,), int(frac), dtype=torch.uint8) for _ in range(B)])
    do = inp.output_grad((B, N, Hq, 128), torch.bfloat16, 9000 + c)
    qd, kd, vd, gd, dod = (t.cuda() for t in (q, k, v, gate, do))
    o, lse = swa.prefill(qd, kd, vd, gd, W, want_lse=True)
    grads = swa.prefill_backward(qd, kd, vd, gd, o, lse, dod, W)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    refs = oracle.prefill_backward(f64(q), f64(k), f64(v), gate.numpy(), f64(do), W,
                                   1.0 / math.sqrt(128))
    for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
        r = np.asarray(ref)
        err = np.abs(f64(got).reshape(r.shape) - r)
        assert err.max() <= 1e-2 * np.abs(r).max(), (case, name, err.max(), np.abs(r).max())
        assert err.mean() <= 4e-3 * np.abs(r).mean(), (case, name, err.mean(), np.abs(r).mean())


def test_prefill_tiny_items_repeated(swa):
    """Many calls whose work items are one or two key blocks long, band and far
    items mixed on every CTA (routed rows past the window in short runs, N a few
    hundred rows per head).  Every call must finish without a device-side wait
    expiring; the last call's outputs match the oracle."""
    B, N, Hq, Hkv, W = 4, 700, 8, 2, 100
    g = inp._gen(7777)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    gate = torch.stack([inp.run_gates(N, 0.3, g, mean_run=4.0) for _ in range(B)])
    scale = 1 / math.sqrt(128)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), gate.cuda()
    for _ in range(60):
        o = swa.prefill(qd, kd, vd, gd, W, scale)
        assert swa.get_device_error() == 0
    ref = oracle.prefill(f64(q), f64(k), f64(v), gate.numpy(), W, scale)
    err = np.abs(f64(o) - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())


@pytest.mark.parametrize("N,W", [(4096, 256), (8192, 1024)])
def test_prefill_most_far_pairs_split(swa, N, W):
    """One query head, every row routed except the first row of each 128-row
    tile: every 256-row pair is both a far pair and a band pair, and the far
    pairs past about a quarter of the sequence each cost more than 1.25 x a
    CTA's share, so they are listed as two one-tile items.  The work list then
    holds about 2.8 items per 256 rows (46 for N = 4096, W = 256), more than
    one far and one band item per pair; the output must still match the
    oracle."""
    B, Hq, Hkv = 1, 1, 1
    g = inp._gen(31337)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    gate = torch.ones(B, N, dtype=torch.uint8)
    gate[:, ::128] = 0
    scale = 1 / math.sqrt(128)
    o = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W, scale)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ref = oracle.prefill(f64(q), f64(k), f64(v), gate.numpy(), W, scale)
    err = np.abs(f64(o) - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())


@pytest.mark.parametrize("R", [1, 128, 129, 200])
def test_far_row_counts_at_tile_edges(swa, R):
    """Far-row counts at the edges of the far tiling (the first far tile holds
    the remainder of the count: 127 empty slots for R = 1 and 129, none for
    R = 128): prefill outputs and the backward's dQ, dK, dV against the
    oracle, with the routed rows spread over [W, N)."""
    B, N, Hq, Hkv, W = 1, 1024, 2, 1, 64
    g = inp._gen(4242 + R)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    rows = torch.randperm(N - W, generator=g)[:R] + W
    gate = torch.zeros(B, N, dtype=torch.uint8)
    gate[0, rows] = 1
    scale = 1 / math.sqrt(128)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), gate.cuda()
    o, lse = swa.prefill(qd, kd, vd, gd, W, scale, want_lse=True)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ref = oracle.prefill(f64(q), f64(k), f64(v), gate.numpy(), W, scale)
    err = np.abs(f64(o) - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())
    do = inp.output_grad((B, N, Hq, 128), torch.bfloat16, 77 + R)
    grads = swa.prefill_backward(qd, kd, vd, gd, o, lse, do.cuda(), W)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    refs = oracle.prefill_backward(f64(q), f64(k), f64(v), gate.numpy(), f64(do), W, scale)
    for name, got, r in zip(("dq", "dk", "dv"), grads, refs):
        r = np.asarray(r)
        e = np.abs(f64(got).reshape(r.shape) - r)
        assert e.max() <= 1e-2 * np.abs(r).max(), (name, e.max(), np.abs(r).max())
        assert e.mean() <= 4e-3 * np.abs(r).mean(), (name, e.mean(), np.abs(r).mean())

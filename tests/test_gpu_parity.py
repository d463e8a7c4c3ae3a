"""GPU parity: every call of libswiattn against the fp64 oracle on the same
seeded inputs, through the C ABI (via the thin binding).

Tolerances (stated by the workload definition): bf16 attention outputs
max-abs 2e-2 and mean-abs 2e-3; fp32 outputs 1e-4; gate decisions and visited
key ranges bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swiattn_inputs as inp

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, F32_TOL = 2e-2, 2e-3, 1e-4


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


def assert_bf16_close(got, ref, what=""):
    err = np.abs(f64(got) - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (what, err.max(), err.mean())


def assert_f32_close(got, ref, what=""):
    err = np.abs(f64(got) - ref)
    assert err.max() <= F32_TOL, (what, err.max())


def cuda(*ts):
    return [t.cuda() for t in ts]


# ------------------------------------------------------------------ route --
def test_route_gates_bit_exact(swa):
    d = inp.prefill_4k(seed=0)
    h, w, bias, g = d["h"], d["w"], d["bias"], d["gen"]
    # keep every logit at least 1e-3 away from the threshold (redraw rows)
    for _ in range(10):
        lg, _ = oracle.route(f64(h), f64(w), bias)
        bad = np.nonzero(np.abs(lg) < 1e-3)[0]
        if bad.size == 0:
            break
        inp.redraw_rows(h, bad, g)
    ref_logits, ref_gate = oracle.route(f64(h), f64(w), bias)
    assert np.abs(ref_logits).min() >= 1e-3
    logits, gate = swa.route(h.cuda(), w.cuda(), bias)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gate.cpu().numpy(), ref_gate)
    np.testing.assert_allclose(f64(logits), ref_logits, rtol=0, atol=1e-4)
    frac = ref_gate.mean()
    assert 0.10 < frac < 0.16, frac   # ~13 % routed, as the recipe intends


def test_route_fp32_and_ragged(swa):
    g = inp._gen(5)
    h = inp.randn((77, 36), torch.float32, g)
    w = inp.randn((36,), torch.float32, g)
    ref_logits, ref_gate = oracle.route(f64(h), f64(w), 0.25)
    keep = np.abs(ref_logits) > 1e-4
    logits, gate = swa.route(h.cuda(), w.cuda(), 0.25)
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(logits), ref_logits, atol=1e-5)
    np.testing.assert_array_equal(gate.cpu().numpy()[keep], ref_gate[keep])


# ------------------------------------------------------ tiny fp32 config --
def test_tiny_fp32_prefill(swa):
    d = inp.tiny_fp32(seed=0)
    q, k, v, gate = cuda(d["q"], d["k"], d["v"], d["gate"])
    scale = 1 / math.sqrt(d["d"])
    o, lse = swa.prefill(q, k, v, gate, d["W"], scale, want_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.prefill(f64(d["q"]), f64(d["k"]), f64(d["v"]), d["gate"].numpy(), d["W"],
                                  scale, want_lse=True)
    assert_f32_close(o, ref, "o")
    assert_f32_close(lse, ref_lse, "lse")


def test_tiny_fp32_dual_and_decode(swa):
    d = inp.tiny_fp32(seed=1)
    g = inp._gen(11)
    logits = inp.logits_with_margin((1, d["N"]), g)
    nll = torch.rand(1, d["N"], generator=g) * 4
    scale = 1 / math.sqrt(d["d"])
    out = swa.dual_branch(*cuda(d["q"], d["k"], d["v"], logits, nll), d["W"], scale)
    torch.cuda.synchronize()
    ref = oracle.dual(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(logits), f64(nll), d["W"], scale)
    assert_f32_close(out["o_full"], ref["o_full"])
    assert_f32_close(out["o_swa"], ref["o_swa"])
    np.testing.assert_allclose(f64(out["mse"]), ref["mse"], rtol=1e-4, atol=1e-6)
    np.testing.assert_allclose(f64(out["gamma"]), ref["gamma"], rtol=1e-4)
    np.testing.assert_allclose(f64(out["reg_loss"]), ref["reg"], rtol=1e-4)
    sel = (logits > 0)[..., None, None].numpy()
    assert_f32_close(out["o_gated"], np.where(sel, ref["o_full"], ref["o_swa"]))
    assert np.all(f64(out["mse"])[:, :d["W"]] == 0.0)
    # decode: each sequence is the tiny prefix of length L with its own gate
    B = 4
    kc = d["k"].expand(B, -1, -1, -1).contiguous()
    vc = d["v"].expand(B, -1, -1, -1).contiguous()
    sl = torch.tensor([256, 31, 32, 200], dtype=torch.int32)
    gd = torch.tensor([0, 1, 0, 1], dtype=torch.uint8)
    qd = d["q"][0, sl.long() - 1]
    od = swa.decode(*cuda(qd, kc, vc, sl, gd), d["W"], scale)
    torch.cuda.synchronize()
    refd = oracle.decode(f64(qd), f64(kc), f64(vc), sl.numpy(), gd.numpy(), d["W"], scale)
    assert_f32_close(od, refd)


# ------------------------------------------------- single-layer prefill 4K --
def test_prefill_4k_bf16_routed(swa):
    d = inp.prefill_4k(seed=0)
    logits, gate = swa.route(d["h"].cuda(), d["w"].cuda(), d["bias"])
    q, k, v = cuda(d["q"], d["k"], d["v"])
    scale = 1 / math.sqrt(d["d"])
    o = swa.prefill(q, k, v, gate, d["W"], scale)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    g = gate.cpu().numpy().reshape(1, -1)
    ref = oracle.prefill(f64(d["q"]), f64(d["k"]), f64(d["v"]), g, d["W"], scale)
    assert_bf16_close(o, ref, "prefill 4k")


# ------------------------------------------------------ long prefill 32K --
# lse = m + log(sum p) in fp32: the sum of up to 32768 terms carries a
# relative error of at most n * 2^-24 (2e-3 at n = 32768), which is the
# absolute error of lse; the exponentials' own error (ex2.approx, a few ulp)
# is far below it.
LSE_TOL = 3e-3


@pytest.mark.parametrize("frac", [0.13, 0.05])
def test_prefill_32k_bf16_full(swa, frac):
    """Every (row, head) output and lse of the long-context workload against the
    oracle: max-abs 2e-2 and mean-abs 2e-3 over all 67M output elements."""
    d = inp.prefill_32k(frac=frac, seed=0)
    W = d["W"]
    q, k, v, gate = cuda(d["q"], d["k"], d["v"], d["gate"])
    scale = 1 / math.sqrt(d["d"])
    o, lse = swa.prefill(q, k, v, gate, W, scale, want_lse=True)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    assert torch.isfinite(o.float()).all()
    got, got_lse = f64(o), f64(lse)
    del o, lse, q, k, v
    ref, ref_lse = oracle.prefill(f64(d["q"]), f64(d["k"]), f64(d["v"]), d["gate"].numpy(), W,
                                  scale, want_lse=True)
    err = np.abs(got - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (frac, err.max(), err.mean())
    assert np.abs(got_lse - ref_lse).max() <= LSE_TOL


# ------------------------------------------------------ decode 16 x 32K --
def test_decode_16x32k_bf16(swa):
    """Every head of every sequence (routed ones read 32768 entries, window
    ones the last 1024) against the oracle, max-abs and mean-abs."""
    d = inp.decode_16x32k(seed=0)
    scale = 1 / math.sqrt(d["d"])
    q, kc, vc, sl, gate = cuda(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], d["gate"])
    o, lse = swa.decode(q, kc, vc, sl, gate, d["W"], scale, want_lse=True)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    got, got_lse = f64(o), f64(lse)
    ref = np.empty_like(got)
    ref_lse = np.empty_like(got_lse)
    for b in range(d["B"]):   # one sequence at a time keeps the fp64 caches at 1 GiB
        r, rl = oracle.decode(f64(d["q"][b:b + 1]), f64(d["k_cache"][b:b + 1]),
                              f64(d["v_cache"][b:b + 1]), d["seq_lens"][b:b + 1].numpy(),
                              d["gate"][b:b + 1].numpy(), d["W"], scale, want_lse=True)
        ref[b], ref_lse[b] = r[0], rl[0]
    err = np.abs(got - ref)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())
    assert np.abs(got_lse - ref_lse).max() <= LSE_TOL
    assert int(d["gate"].sum()) >= 1 and int(d["gate"].sum()) < d["B"]   # both kinds present


# ------------------------------------------------- dual branch 8K, GQA --
def test_dual_8k_gqa_bf16_full(swa):
    """Every token of the dual-branch workload: both branch outputs, the
    divergence, gamma and the regulariser against the oracle."""
    d = inp.dual_8k(seed=0)
    B, N, Hq, W = d["B"], d["N"], d["Hq"], d["W"]
    scale = 1 / math.sqrt(d["d"])
    out = swa.dual_branch(*cuda(d["q"], d["k"], d["v"], d["logits"], d["nll"]), W, scale,
                          d["gamma_base"], d["eps"], d["alpha"])
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    mse = f64(out["mse"])
    # identical key sets inside the window: exactly zero divergence
    assert np.all(mse[:, :W] == 0.0)
    assert np.all(mse[:, W:] > 0.0)
    torch.testing.assert_close(out["o_full"][:, :W], out["o_swa"][:, :W], rtol=0, atol=0)
    sel_full = (d["logits"] > 0)[..., None, None].cuda()
    assert torch.equal(out["o_gated"], torch.where(sel_full, out["o_full"], out["o_swa"]))
    got_full, got_swa = f64(out["o_full"]), f64(out["o_swa"])
    gamma, reg = f64(out["gamma"]), f64(out["reg_loss"])
    del out
    ref = oracle.dual(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(d["logits"]), f64(d["nll"]),
                      W, scale, d["gamma_base"], d["eps"], d["alpha"])
    for name, got in (("o_full", got_full), ("o_swa", got_swa)):
        err = np.abs(got - ref[name])
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (name, err.max(), err.mean())
    # mse sums 2048 squared differences of outputs that each carry a relative
    # error of order 2^-8 (bf16 probabilities): a few per cent of mse.
    np.testing.assert_allclose(mse, ref["mse"], rtol=3e-2, atol=1e-3)
    np.testing.assert_allclose(gamma, ref["gamma"], rtol=3e-2)
    np.testing.assert_allclose(reg, ref["reg"], rtol=3e-2)


# ------------------------------------------------------------ edge cases --
EDGE = [
    # B, N, Hq, Hkv, W, gate pattern
    (1, 1, 2, 2, 4, "ones"),
    (1, 5, 2, 2, 3, "alt"),
    (1, 127, 2, 2, 16, "rand"),
    (1, 300, 2, 2, 37, "rand"),
    (2, 300, 4, 2, 128, "runs"),
    (1, 300, 2, 2, 1, "rand"),
    (1, 300, 2, 2, 300, "rand"),
    (1, 300, 2, 2, 1000, "rand"),
    (1, 700, 2, 2, 129, "zeros"),
    (1, 700, 2, 2, 129, "ones"),
    (1, 700, 2, 2, 64, "single"),
    (3, 520, 8, 2, 200, "runs"),
    # 64-key block edges of the tensor-core kernel
    (1, 64, 2, 2, 64, "rand"),
    (1, 65, 2, 2, 63, "rand"),
    (1, 191, 2, 2, 65, "runs"),
    (1, 192, 2, 2, 64, "ones"),
    (1, 193, 2, 2, 127, "alt"),
    (2, 257, 2, 2, 65, "rand"),
]


def _gate(pattern, B, N, g):
    if pattern == "ones":
        return torch.ones(B, N, dtype=torch.uint8)
    if pattern == "zeros":
        return torch.zeros(B, N, dtype=torch.uint8)
    if pattern == "alt":
        return (torch.arange(N) % 2).to(torch.uint8).expand(B, N).contiguous()
    if pattern == "single":
        x = torch.zeros(B, N, dtype=torch.uint8)
        x[:, N - 3] = 1
        return x
    if pattern == "runs":
        return torch.stack([inp.run_gates(N, 0.2, g, mean_run=20.0) for _ in range(B)])
    return inp.bernoulli_gates((B, N), 0.3, g)


@pytest.mark.parametrize("B,N,Hq,Hkv,W,pattern", EDGE)
def test_prefill_edges_bf16(swa, B, N, Hq, Hkv, W, pattern):
    g = inp._gen(100 + N + W)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    gate = _gate(pattern, B, N, g)
    scale = 1 / math.sqrt(128)
    o = swa.prefill(*cuda(q, k, v, gate), W, scale)
    torch.cuda.synchronize()
    ref = oracle.prefill(f64(q), f64(k), f64(v), gate.numpy(), W, scale)
    assert_bf16_close(o, ref, (B, N, W, pattern))
    assert swa.get_device_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N,W,pattern", [(300, 37, "rand"), (700, 129, "runs"), (1000, 1, "rand"),
                                         (260, 500, "alt"), (4100, 1024, "runs")])
def test_visited_key_count_exact(swa, dtype, N, W, pattern):
    """q = 0: every visited key scores 0, so exp(lse) is the exact number of
    visited keys of each row; it must equal hi - lo + 1 of the definition."""
    g = inp._gen(7 + N)
    B, H = 1, 2
    _, k, v = inp.attention_qkv(B, N, H, H, 128, dtype, g)
    q = torch.zeros(B, N, H, 128, dtype=dtype)
    gate = _gate(pattern, B, N, g)
    o, lse = swa.prefill(*cuda(q, k, v, gate), W, 0.1, want_lse=True)
    torch.cuda.synchronize()
    lo, hi = oracle.row_ranges(gate.numpy(), W)
    n_ref = (hi - lo + 1)[..., None].repeat(H, -1)
    n_gpu = np.rint(np.exp(f64(lse))).astype(np.int64)
    np.testing.assert_array_equal(n_gpu, n_ref)


def test_decode_edges(swa):
    g = inp._gen(77)
    for dtype, d, Hq, Hkv in [(torch.bfloat16, 128, 8, 2), (torch.bfloat16, 64, 4, 4),
                              (torch.float32, 128, 4, 1), (torch.float32, 64, 16, 2)]:
        B, Lmax, W = 5, 333, 50
        kc = inp.randn((B, Lmax, Hkv, d), dtype, g)
        vc = inp.randn((B, Lmax, Hkv, d), dtype, g)
        q = inp.randn((B, Hq, d), dtype, g)
        sl = torch.tensor([1, 49, 50, 51, 333], dtype=torch.int32)
        gate = torch.tensor([1, 0, 1, 0, 0], dtype=torch.uint8)
        scale = 1 / math.sqrt(d)
        o = swa.decode(*cuda(q, kc, vc, sl, gate), W, scale)
        torch.cuda.synchronize()
        ref = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), gate.numpy(), W, scale)
        if dtype == torch.float32:
            assert_f32_close(o, ref, (d, Hq, Hkv))
        else:
            assert np.abs(f64(o) - ref).max() <= BF16_MAX


def test_decode_batches_above_32_and_batch_invariance(swa):
    """Batches of up to 32 sequences run on persistent CTAs that claim chunks
    longest first; larger ones get one CTA per (chunk, sequence) slot.  Both
    match the oracle, and every sequence's output is bit for bit the same in a
    batch of 40, in a batch of 32 and alone (its chunks, and each chunk's
    arithmetic, depend on the sequence alone)."""
    g = inp._gen(79)
    B, Lmax, Hq, Hkv, d, W = 40, 600, 8, 2, 128, 100
    kc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g)
    vc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g)
    q = inp.randn((B, Hq, d), torch.bfloat16, g)
    sl = torch.randint(1, Lmax + 1, (B,), generator=g, dtype=torch.int32)
    sl[:4] = torch.tensor([1, Lmax, W, W + 1], dtype=torch.int32)
    gate = inp.bernoulli_gates((B,), 0.3, g)
    scale = 1 / math.sqrt(d)
    qd, kd, vd, sld, gd = cuda(q, kc, vc, sl, gate)
    o40, lse40 = swa.decode(qd, kd, vd, sld, gd, W, scale, want_lse=True)
    o32, lse32 = swa.decode(qd[:32], kd[:32], vd[:32], sld[:32], gd[:32], W, scale, want_lse=True)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ref = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), gate.numpy(), W, scale)
    assert_bf16_close(o40, ref, "B=40")
    assert torch.equal(o40[:32], o32) and torch.equal(lse40[:32], lse32)
    for b in (0, 1, 3, 17, 31, 32, 39):
        o1, lse1 = swa.decode(qd[b:b + 1], kd[b:b + 1], vd[b:b + 1], sld[b:b + 1], gd[b:b + 1], W,
                              scale, want_lse=True)
        torch.cuda.synchronize()
        assert torch.equal(o1[0], o40[b]) and torch.equal(lse1[0], lse40[b]), b


def test_decode_wide_token_rows(swa):
    """One block reads a token row of every KV head (one thread per 16 bytes).
    Rows within the split kernel's block limit are computed; a wider valid row
    is refused with SWIATTN_EUNSUPPORTED before any launch, never with a CUDA
    error.  512 threads (32 heads, Hq = Hkv) and 256 threads (16 heads,
    Hq = 8 Hkv) are within every limit the kernel's register use allows."""
    g = inp._gen(78)
    computed = []
    for Hkv, G in ((32, 1), (56, 1), (64, 1), (16, 8), (32, 8)):
        Hq, d, B, Lmax, W = Hkv * G, 128, 2, 150, 40
        kc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g)
        vc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g)
        q = inp.randn((B, Hq, d), torch.bfloat16, g)
        sl = torch.tensor([150, 77], dtype=torch.int32)
        gate = torch.tensor([1, 0], dtype=torch.uint8)
        scale = 1 / math.sqrt(d)
        try:
            o = swa.decode(*cuda(q, kc, vc, sl, gate), W, scale)
        except swa.SwiAttnError as e:
            assert e.status == 2, (Hkv, G, str(e))   # SWIATTN_EUNSUPPORTED
            continue
        torch.cuda.synchronize()
        ref = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), gate.numpy(), W, scale)
        assert np.abs(f64(o) - ref).max() <= BF16_MAX, (Hkv, G)
        computed.append((Hkv, G))
    assert (32, 1) in computed and (16, 8) in computed
    assert swa.get_device_error() == 0


# -------------------------------------------------------- cross-API invariants --
def test_cross_api_invariants(swa):
    g = inp._gen(31)
    B, N, Hq, Hkv, W = 2, 600, 4, 2, 100
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    scale = 1 / math.sqrt(128)
    qd, kd, vd = cuda(q, k, v)
    ones = torch.ones(B, N, dtype=torch.uint8, device="cuda")
    zeros = torch.zeros_like(ones)
    o1 = swa.prefill(qd, kd, vd, ones, W, scale)
    o0 = swa.prefill(qd, kd, vd, zeros, W, scale)
    logits = inp.logits_with_margin((B, N), g).cuda()
    nll = torch.ones(B, N, device="cuda")
    out = swa.dual_branch(qd, kd, vd, logits, nll, W, scale)
    torch.cuda.synchronize()
    for a, b_ in ((out["o_full"], o1), (out["o_swa"], o0)):
        err = (a.float() - b_.float()).abs()
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN
    # decode of the last token equals the last prefill row
    sl = torch.full((B,), N, dtype=torch.int32, device="cuda")
    for gval, ref in ((1, o1), (0, o0)):
        gd = torch.full((B,), gval, dtype=torch.uint8, device="cuda")
        od = swa.decode(qd[:, -1].contiguous(), kd, vd, sl, gd, W, scale)
        torch.cuda.synchronize()
        assert (od.float() - ref[:, -1].float()).abs().max() <= BF16_MAX


def test_prefill_deterministic(swa):
    d = inp.prefill_32k(frac=0.13, seed=3, N=8192)
    q, k, v, gate = cuda(d["q"], d["k"], d["v"], d["gate"])
    a = swa.prefill(q, k, v, gate, d["W"])
    b = swa.prefill(q, k, v, gate, d["W"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert swa.get_device_error() == 0

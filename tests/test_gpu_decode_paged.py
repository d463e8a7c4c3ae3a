"""GPU parity of decode over a paged KV cache (swiattn_decode_paged).

The paged call reads each token's K/V row through a block table; with the
same cache contents it must give exactly what swiattn_decode gives on the
contiguous cache (the arithmetic is the same, only the addresses differ), and
it is compared with the fp64 oracle on the contiguous copy.  Tolerances as
for decode: bf16 max-abs 2e-2 / mean-abs 2e-3, fp32 1e-4.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swiattn_inputs as inp

pytestmark = pytest.mark.gpu


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


def paged_copy(kc, vc, page_size, seed, spare_pages=3):
    """Scatter contiguous caches [B, Lmax, Hkv, d] into a shuffled page pool;
    returns k_pages, v_pages, block_table (int32 [B, max_pages])."""
    B, Lmax, Hkv, d = kc.shape
    max_pages = -(-Lmax // page_size)
    num_pages = B * max_pages + spare_pages
    perm = torch.randperm(num_pages, generator=inp._gen(seed))[: B * max_pages]
    kp = torch.zeros((num_pages, page_size, Hkv, d), dtype=kc.dtype)
    vp = torch.zeros_like(kp)
    pad = max_pages * page_size - Lmax
    kpad = torch.nn.functional.pad(kc, (0, 0, 0, 0, 0, pad))
    vpad = torch.nn.functional.pad(vc, (0, 0, 0, 0, 0, pad))
    kp[perm] = kpad.reshape(B * max_pages, page_size, Hkv, d)
    vp[perm] = vpad.reshape(B * max_pages, page_size, Hkv, d)
    table = perm.reshape(B, max_pages).to(torch.int32)
    return kp, vp, table


def case(B, Lmax, Hq, Hkv, d, dtype, seed, lens):
    g = inp._gen(seed)
    kc = inp.randn((B, Lmax, Hkv, d), dtype, g)
    vc = inp.randn((B, Lmax, Hkv, d), dtype, g)
    q = inp.randn((B, Hq, d), dtype, g)
    gate = inp.bernoulli_gates((B,), 0.5, g)
    sl = torch.tensor(lens, dtype=torch.int32)
    return q, kc, vc, gate, sl


@pytest.mark.parametrize("page_size", [1, 16, 64, 256, 1024])
def test_paged_equals_contiguous_bitwise(swa, page_size):
    B, Lmax, H, d, W = 4, 1500, 4, 128, 300
    q, kc, vc, gate, sl = case(B, Lmax, H, H, d, torch.bfloat16, page_size, [1500, 1, 299, 777])
    gate[:] = torch.tensor([1, 0, 1, 0], dtype=torch.uint8)
    kp, vp, table = paged_copy(kc, vc, page_size, seed=page_size + 1)
    dev = lambda t: t.cuda()
    ref = swa.decode(dev(q), dev(kc), dev(vc), dev(sl), dev(gate), W)
    got = swa.decode_paged(dev(q), dev(kp), dev(vp), dev(table), dev(sl), dev(gate), W)
    assert swa.get_device_error() == 0
    assert torch.equal(got, ref)


@pytest.mark.parametrize("dtype,d,Hq,Hkv", [(torch.bfloat16, 128, 8, 2), (torch.float32, 64, 4, 4),
                                            (torch.bfloat16, 64, 4, 1)])
def test_paged_matches_oracle(swa, dtype, d, Hq, Hkv):
    B, Lmax, W = 5, 2100, 512
    q, kc, vc, gate, sl = case(B, Lmax, Hq, Hkv, d, dtype, 7, [2100, 513, 512, 64, 1999])
    kp, vp, table = paged_copy(kc, vc, 32, seed=8)
    o, lse = swa.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(), gate.cuda(),
                              W, want_lse=True)
    assert swa.get_device_error() == 0
    ref_o, ref_lse = oracle.decode(f64(q), f64(kc), f64(vc), sl.numpy(), gate.numpy(), W,
                                   1.0 / math.sqrt(d), want_lse=True)
    err = np.abs(f64(o) - ref_o)
    if dtype == torch.float32:
        assert err.max() <= 1e-4
    else:
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(f64(lse) - ref_lse).max() <= 1e-3


def test_multi_layer_step_flattened(swa):
    """Three layers of one decode step in one call: (layer, sequence) pairs
    flattened into B, per-layer pools laid end to end with offset tables,
    per-layer gates.  Equal to one call per layer."""
    layers, B, Lmax, H, d, W = 3, 2, 700, 4, 128, 256
    qs, kps, vps, tables, gates, outs = [], [], [], [], [], []
    offset = 0
    sl = torch.tensor([700, 300], dtype=torch.int32)
    for layer in range(layers):
        q, kc, vc, gate, _ = case(B, Lmax, H, H, d, torch.bfloat16, 20 + layer, [700, 300])
        kp, vp, table = paged_copy(kc, vc, 64, seed=30 + layer)
        outs.append(swa.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(),
                                     gate.cuda(), W))
        qs.append(q)
        kps.append(kp)
        vps.append(vp)
        tables.append(table + offset)
        gates.append(gate)
        offset += kp.shape[0]
    got = swa.decode_paged(torch.cat(qs).cuda(), torch.cat(kps).cuda(), torch.cat(vps).cuda(),
                           torch.cat(tables).cuda(), sl.repeat(layers).cuda(),
                           torch.cat(gates).cuda(), W)
    assert swa.get_device_error() == 0
    assert torch.equal(got, torch.cat(outs))


def test_bad_block_table_entry_is_reported(swa):
    """An entry past the pool, on a page the call reads, is read as page 0 (no
    out-of-range access) and the device error word reports SWIATTN_EINVAL; the
    next query is clean."""
    q, kc, vc, gate, sl = case(2, 300, 2, 2, 128, torch.bfloat16, 40, [300, 200])
    gate[:] = 1   # routed: every page of the sequence is read
    kp, vp, table = paged_copy(kc, vc, 16, seed=41)
    bad = table.clone()
    bad[0, 3] = kp.shape[0] + 5
    swa.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), bad.cuda(), sl.cuda(), gate.cuda(), 64)
    assert swa.get_device_error() == 1
    assert swa.get_device_error() == 0


def test_length_past_cache_is_clamped_and_reported(swa):
    """seq_lens beyond Lmax (device data) is clamped to Lmax, gives exactly the
    Lmax result, and is reported as SWIATTN_EINVAL; nothing is read past the
    cache or the workspace."""
    q, kc, vc, gate, sl = case(2, 400, 2, 2, 128, torch.bfloat16, 50, [400, 123])
    ref = swa.decode(q.cuda(), kc.cuda(), vc.cuda(), sl.cuda(), gate.cuda(), 100)
    assert swa.get_device_error() == 0
    long_sl = torch.tensor([400 + 77, 123], dtype=torch.int32)
    got = swa.decode(q.cuda(), kc.cuda(), vc.cuda(), long_sl.cuda(), gate.cuda(), 100)
    assert swa.get_device_error() == 1
    assert torch.equal(got, ref)


@pytest.mark.parametrize("S", [1, 256, 300, 5000])
def test_anchored_decode_matches_oracle(swa, S):
    """Global anchors: a window query also reads the first S cache entries."""
    B, Lmax, Hq, Hkv, d, W = 6, 3000, 4, 2, 128, 512
    q, kc, vc, gate, sl = case(B, Lmax, Hq, Hkv, d, torch.bfloat16, 60 + S,
                               [3000, 1, 100, 513, 2000, 777])
    gate[:] = torch.tensor([0, 0, 0, 0, 1, 0], dtype=torch.uint8)
    o, lse = swa.decode_anchored(q.cuda(), kc.cuda(), vc.cuda(), sl.cuda(), gate.cuda(), W, S,
                                 want_lse=True)
    assert swa.get_device_error() == 0
    ref_o, ref_lse = oracle.decode_anchored(f64(q), f64(kc), f64(vc), sl.numpy(), gate.numpy(), W,
                                            S, 1.0 / math.sqrt(d), want_lse=True)
    err = np.abs(f64(o) - ref_o)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(f64(lse) - ref_lse).max() <= 1e-3
    # exact visited counts: q = 0 gives lse = ln(number of entries read)
    o0, lse0 = swa.decode_anchored(torch.zeros_like(q).cuda(), kc.cuda(), vc.cuda(), sl.cuda(),
                                   gate.cuda(), W, S, want_lse=True)
    L = sl.numpy().astype(np.int64)
    lo = np.where(gate.numpy() != 0, 0, np.maximum(0, L - W))
    n = (L - lo) + np.minimum(S, lo)
    np.testing.assert_array_equal(np.rint(np.exp(f64(lse0))).astype(np.int64), n[:, None].repeat(Hq, 1))


def test_anchored_decode_zero_is_plain_and_paged_matches(swa):
    B, Lmax, H, d, W, S = 4, 1500, 4, 128, 300, 256
    q, kc, vc, gate, sl = case(B, Lmax, H, H, d, torch.bfloat16, 70, [1500, 1, 299, 777])
    gate[:] = torch.tensor([0, 0, 0, 0], dtype=torch.uint8)
    dev = lambda t: t.cuda()
    plain = swa.decode(dev(q), dev(kc), dev(vc), dev(sl), dev(gate), W)
    zero = swa.decode_anchored(dev(q), dev(kc), dev(vc), dev(sl), dev(gate), W, 0)
    assert torch.equal(plain, zero)
    anch = swa.decode_anchored(dev(q), dev(kc), dev(vc), dev(sl), dev(gate), W, S)
    kp, vp, table = paged_copy(kc, vc, 64, seed=71)
    paged = swa.decode_paged(dev(q), dev(kp), dev(vp), dev(table), dev(sl), dev(gate), W,
                             n_anchor=S)
    assert swa.get_device_error() == 0
    assert torch.equal(paged, anch)

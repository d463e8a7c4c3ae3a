"""swiattn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a host runtime that owns every allocation, or code
that must not allocate while it runs).  It keeps its split-KV partials in a
fixed array inside the library instead of a caller workspace, so it must give
the same results as swiattn_decode.  Collected last on purpose: a run that
stops at the first failure has run every other test by then.
"""
import ctypes
import math

import pytest
import torch

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


def _call_noalloc(lib, q, kc, vc, sl, gate, o, lse, W, scale, dtype):
    B, Hq, d = q.shape
    Lmax, Hkv = kc.shape[1], kc.shape[2]
    vp = ctypes.c_void_p
    return lib.swiattn_decode_noalloc(
        vp(q.data_ptr()), vp(kc.data_ptr()), vp(vc.data_ptr()), vp(sl.data_ptr()),
        vp(gate.data_ptr()), vp(o.data_ptr()), vp(lse.data_ptr() if lse is not None else None),
        B, Lmax, Hq, Hkv, d, W, float(scale), dtype,
        vp(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_decode_matches_workspace_decode_twice(swa, dtype):
    lib = swa._load()
    g = inp._gen(2024)
    B, Lmax, Hq, Hkv, d, W = 6, 3000, 8, 4, 128, 500
    scale = 1 / math.sqrt(d)
    code = swa._DT[dtype]
    for call in range(2):   # two calls in a row share the library's scratch array
        kc = inp.randn((B, Lmax, Hkv, d), dtype, g).cuda()
        vc = inp.randn((B, Lmax, Hkv, d), dtype, g).cuda()
        q = inp.randn((B, Hq, d), dtype, g).cuda()
        sl = torch.tensor([1, 499, 500, 501, 2999, 3000], dtype=torch.int32).roll(call).cuda()
        gate = torch.tensor([0, 1, 0, 1, 0, 1], dtype=torch.uint8).roll(call).cuda()
        ref, ref_lse = swa.decode(q, kc, vc, sl, gate, W, scale, want_lse=True)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        assert _call_noalloc(lib, q, kc, vc, sl, gate, o, lse, W, scale, code) == 0
        torch.cuda.synchronize()
        tol = 1e-4 if dtype == torch.float32 else 2e-2
        assert (o.float() - ref.float()).abs().max().item() <= tol
        assert (lse - ref_lse).abs().max().item() <= 1e-4
    assert swa.get_device_error() == 0


def test_noalloc_decode_rejects_partials_beyond_scratch(swa):
    lib = swa._load()
    B, Hq, Hkv, d, W = 16, 16, 16, 128, 1024
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    sl = torch.full((B,), 8, dtype=torch.int32, device="cuda")
    gate = torch.zeros(B, dtype=torch.uint8, device="cuda")
    small = torch.zeros(B, 8, Hkv, d, dtype=torch.bfloat16, device="cuda")
    # Lmax = 32 512 needs 128 chunks of partials: 17.0 MB > 16 MiB.  The caches
    # are never read because validation rejects the call first.
    rc = _call_noalloc(lib, q, small, small, sl, gate, o, lse, W, 0.1, swa.BF16)
    assert rc == 0
    vp = ctypes.c_void_p
    # At B = Hq = 16, d = 128 the partials fit 16 MiB up to Lmax = 32 000
    # (126 chunks: 16 773 376 bytes with the counter) and not from 32 001
    # (127 chunks: 16 906 496 bytes).
    for Lmax in (32001, 32512):
        rc = lib.swiattn_decode_noalloc(vp(q.data_ptr()), vp(small.data_ptr()),
                                        vp(small.data_ptr()), vp(sl.data_ptr()),
                                        vp(gate.data_ptr()), vp(o.data_ptr()), vp(lse.data_ptr()),
                                        B, Lmax, Hq, Hkv, d, W, 0.1, swa.BF16,
                                        vp(torch.cuda.current_stream().cuda_stream))
        assert rc == 1, Lmax   # SWIATTN_EINVAL, nothing launched
    torch.cuda.synchronize()
    # The largest accepted Lmax runs (full-size caches; 8 tokens of each read).
    big = torch.zeros(B, 32000, Hkv, d, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(lib, q, big, big, sl, gate, o, lse, W, 0.1, swa.BF16) == 0
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    assert torch.equal(o, torch.zeros_like(o))   # zero values: a zero output


def test_noalloc_decode_without_lse(swa):
    """lse is optional, as for swiattn_decode."""
    lib = swa._load()
    g = inp._gen(2025)
    B, Lmax, Hq, Hkv, d, W = 3, 700, 4, 4, 64, 100
    kc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g).cuda()
    vc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g).cuda()
    q = inp.randn((B, Hq, d), torch.bfloat16, g).cuda()
    sl = torch.tensor([700, 99, 350], dtype=torch.int32).cuda()
    gate = torch.tensor([1, 0, 0], dtype=torch.uint8).cuda()
    ref = swa.decode(q, kc, vc, sl, gate, W, 0.125)
    o = torch.empty_like(q)
    assert _call_noalloc(lib, q, kc, vc, sl, gate, o, None, W, 0.125, swa.BF16) == 0
    torch.cuda.synchronize()
    assert (o.float() - ref.float()).abs().max().item() <= 2e-2
    assert swa.get_device_error() == 0


def test_noalloc_decode_reports_out_of_range_lengths(swa):
    """A device-resident length outside [1, Lmax] is clamped into it and
    reported through swiattn_get_device_error, as swiattn_decode does; the
    clamped results equal swiattn_decode's."""
    lib = swa._load()
    g = inp._gen(2026)
    B, Lmax, Hq, Hkv, d, W = 4, 300, 4, 2, 128, 64
    kc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g).cuda()
    vc = inp.randn((B, Lmax, Hkv, d), torch.bfloat16, g).cuda()
    q = inp.randn((B, Hq, d), torch.bfloat16, g).cuda()
    sl = torch.tensor([0, Lmax + 1, 150, -7], dtype=torch.int32).cuda()
    gate = torch.tensor([1, 0, 1, 0], dtype=torch.uint8).cuda()
    assert swa.get_device_error() == 0
    ref = swa.decode(q, kc, vc, sl, gate, W, 0.1)
    assert swa.get_device_error() == 1   # SWIATTN_EINVAL from swiattn_decode
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, q, kc, vc, sl, gate, o, lse, W, 0.1, swa.BF16) == 0
    assert swa.get_device_error() == 1   # the same report from the no-allocation call
    assert torch.equal(o, ref)
    assert swa.get_device_error() == 0   # reading the report cleared it


def test_noalloc_decode_scratch_boundary(swa):
    """The header's example bound: B=16, Hq=16, d=128 fits Lmax = 32000 and
    not 32001 (max(17, ceil(Lmax/256) + 1) chunks of (d+2) floats per
    sequence and head, and 256 bytes for the chunk counter).  The rejected call launches nothing, so its caches,
    smaller than Lmax, are never read."""
    lib = swa._load()
    B, Hq, Hkv, d, W = 16, 16, 16, 128, 1024
    assert swa.decode_workspace(B, 32000, Hq, Hkv, d, W, swa.BF16) <= 16 << 20
    assert swa.decode_workspace(B, 32001, Hq, Hkv, d, W, swa.BF16) > 16 << 20
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    sl = torch.full((B,), 8, dtype=torch.int32, device="cuda")
    gate = torch.zeros(B, dtype=torch.uint8, device="cuda")
    small = torch.zeros(B, 8, Hkv, d, dtype=torch.bfloat16, device="cuda")
    vp = ctypes.c_void_p
    rc = lib.swiattn_decode_noalloc(vp(q.data_ptr()), vp(small.data_ptr()), vp(small.data_ptr()),
                                    vp(sl.data_ptr()), vp(gate.data_ptr()), vp(o.data_ptr()),
                                    vp(None), B, 32001, Hq, Hkv, d, W, 0.1, swa.BF16,
                                    vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 1   # SWIATTN_EINVAL, nothing launched
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0

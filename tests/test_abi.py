"""The C-ABI library loads without a GPU and exports every declared symbol;
host-side validation rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swiattn.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    from sliding_window_attention_router_gb300 import build
    build.build()
    import sliding_window_attention_router_gb300 as swa
    return swa._load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swiattn_\w+)\s*\(", text)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for call in ("swiattn_route", "swiattn_prefill", "swiattn_decode", "swiattn_dual_branch"):
        assert call in names


def test_library_exports_every_declared_symbol(lib):
    import sliding_window_attention_router_gb300 as swa
    names = declared_functions()
    assert sorted(swa.EXPORTS) == names
    for name in names:
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    import sliding_window_attention_router_gb300 as swa
    assert swa.status_string(0) == "SWIATTN_OK"
    assert swa.status_string(1) == "SWIATTN_EINVAL"
    assert swa.status_string(4) == "SWIATTN_ETIMEOUT"
    assert swa.status_string(99) == "SWIATTN_UNKNOWN"


def test_workspace_sizes(lib):
    import sliding_window_attention_router_gb300 as swa
    bf16, f32 = swa.BF16, swa.F32
    n = swa.prefill_workspace(1, 32768, 16, 16, 128, 1024, bf16)
    # the far-row list (int32 per row) and the work list (16 bytes per item,
    # 16 heads x up to 3 items per 256 rows x 128); far queries are gathered
    # in place, not copied
    assert n >= 32768 * 4 + 16 * 3 * 128 * 16 and n % 256 == 0
    assert n < 32768 * 16 * 128 * 2 // 8
    assert swa.prefill_workspace(1, 0, 16, 16, 128, 1024, bf16) == 0
    assert swa.prefill_workspace(1, 64, 6, 4, 128, 8, bf16) == 0   # Hq % Hkv != 0
    dw = swa.decode_workspace(16, 32768, 16, 16, 128, 1024, bf16)
    assert dw >= 16 * (32768 // 256) * 16 * 130 * 4
    assert swa.dual_branch_workspace(2, 8192, 16, 4, 128, 1024, bf16) >= 2 * 8192 * 16 * 4
    # fp32: both branches' lse (used only when lse_gated is requested)
    assert swa.dual_branch_workspace(1, 256, 2, 2, 64, 32, f32) == 2 * 256 * 2 * 4


def test_invalid_arguments_rejected_before_launch(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)          # never dereferenced: validation fails first
    odd = vp((1 << 20) + 8)     # not 16-byte aligned
    # route: bad dtype, misaligned h, d_model not a multiple of 8
    assert lib.swiattn_route(fake, fake, 0.0, 4, 64, 7, fake, fake, None) == 1
    assert lib.swiattn_route(odd, fake, 0.0, 4, 64, 1, fake, fake, None) == 1
    assert lib.swiattn_route(fake, fake, 0.0, 4, 60, 1, fake, fake, None) == 1
    assert lib.swiattn_route(None, None, 0.0, 0, 64, 1, None, None, None) == 0   # no-op
    args = [fake, fake, fake, fake, fake, None]
    # prefill: W < 1, Hq % Hkv, d = 96, misaligned q, workspace too small, bad scale
    assert lib.swiattn_prefill(*args, 1, 64, 4, 4, 128, 0, 0.1, 1, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill(*args, 1, 64, 6, 4, 128, 8, 0.1, 1, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill(*args, 1, 64, 4, 4, 96, 8, 0.1, 1, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill(odd, *args[1:], 1, 64, 4, 4, 128, 8, 0.1, 1, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill(*args, 1, 64, 4, 4, 128, 8, 0.1, 1, fake, 16, None) == 1
    assert lib.swiattn_prefill(*args, 1, 64, 4, 4, 128, 8, 0.0, 1, fake, 1 << 30, None) == 1
    # bf16 head dim 64 is valid but not implemented on the tensor-core path
    assert lib.swiattn_prefill(*args, 1, 64, 4, 4, 64, 8, 0.1, 1, fake, 1 << 30, None) == 2
    # decode: Hq/Hkv = 3 unsupported; workspace too small
    dargs = [fake] * 7
    assert lib.swiattn_decode(*dargs, 2, 64, 6, 2, 128, 8, 0.1, 1, fake, 1 << 30, None) == 2
    assert lib.swiattn_decode(*dargs, 2, 64, 4, 4, 128, 8, 0.1, 1, fake, 8, None) == 1
    # decode: caches longer than 2^30 entries are refused by every decode call
    assert lib.swiattn_decode(*dargs, 1, (1 << 30) + 1, 4, 4, 128, 8, 0.1, 1, fake, 1 << 40,
                              None) == 2
    assert lib.swiattn_decode_noalloc(*dargs, 1, (1 << 30) + 1, 4, 4, 128, 8, 0.1, 1, None) == 2
    # the no-allocation decode validates like swiattn_decode: Hq/Hkv = 3, bad scale, misaligned q
    assert lib.swiattn_decode_noalloc(*dargs, 2, 64, 6, 2, 128, 8, 0.1, 1, None) == 2
    assert lib.swiattn_decode_noalloc(*dargs, 2, 64, 4, 4, 128, 8, 0.0, 1, None) == 1
    assert lib.swiattn_decode_noalloc(odd, *dargs[1:], 2, 64, 4, 4, 128, 8, 0.1, 1, None) == 1
    # dual: missing output
    xargs = [fake] * 5 + [None] + [fake] * 6
    assert lib.swiattn_dual_branch(*xargs, 1, 64, 4, 4, 128, 8, 0.1, 1e-3, 0.1, 100.0, 1, fake,
                                   1 << 30, None) == 1


def test_route_prefill_workspace_and_validation(lib):
    import sliding_window_attention_router_gb300 as swa
    bf16 = swa.BF16
    base = swa.prefill_workspace(2, 4096, 16, 4, 128, 1024, bf16)
    # the prefill's workspace plus the counter that elects the planning CTA
    assert swa.route_prefill_workspace(2, 4096, 16, 4, 128, 1024, bf16) == base + 256
    assert swa.route_prefill_workspace(1, 0, 16, 16, 128, 1024, bf16) == 0
    vp = ctypes.c_void_p
    fake = vp(1 << 20)          # never dereferenced: validation fails first
    odd = vp((1 << 20) + 8)
    ws = 1 << 30

    def call(h=fake, w=fake, d_model=1024, logits=fake, gate=fake, W=64, S=0, d=128, scale=0.1,
             dt=1, nbytes=ws, Hq=4):
        return lib.swiattn_route_prefill(h, w, 0.0, d_model, fake, fake, fake, fake, None, logits,
                                         gate, 1, 256, Hq, 4, d, W, S, scale, dt, fake, nbytes,
                                         None)
    assert call(d_model=1020) == 1          # not a multiple of 8 (bf16)
    assert call(h=odd) == 1                 # misaligned hidden states
    assert call(logits=None) == 1           # router outputs are required
    assert call(gate=None) == 1
    assert call(W=0) == 1
    assert call(S=-1) == 1
    assert call(scale=0.0) == 1
    assert call(Hq=6) == 1                  # Hq % Hkv != 0
    assert call(dt=7) == 1
    assert call(nbytes=16) == 1             # workspace too small
    assert call(d=64) == 2                  # bf16 head dim 64: not on the tensor-core path


def test_prefill_host_workspace_and_validation(lib):
    import sliding_window_attention_router_gb300 as swa
    bf16 = swa.BF16
    base = swa.prefill_workspace(1, 4096, 16, 16, 128, 1024, bf16)
    n = swa.prefill_host_workspace(1, 4096, 16, 16, 128, 1024, bf16)
    # staging for q, k, v (8 MiB each), gate, o, lse on top of the prefill's workspace
    assert n >= base + 4 * 4096 * 16 * 128 * 2 + 4096 + 4096 * 16 * 4 and n % 256 == 0
    assert swa.prefill_host_workspace(1, 0, 16, 16, 128, 1024, bf16) == 0
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    args = [fake] * 5 + [None]
    assert lib.swiattn_prefill_host(None, *args[1:], 1, 64, 4, 4, 128, 8, 0, 0.1, 1, fake, 1 << 30,
                                    None) == 1                                  # missing q
    assert lib.swiattn_prefill_host(*args, 1, 64, 4, 4, 128, 8, 0, 0.1, 1, fake, 16, None) == 1
    assert lib.swiattn_prefill_host(*args, 1, 64, 4, 4, 128, 8, 0, 0.1, 7, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill_host(*args, 1, 64, 4, 4, 128, 8, -1, 0.1, 1, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill_host(*args, 1, 64, 4, 4, 128, 8, 0, 0.0, 1, fake, 1 << 30, None) == 1


def test_backward_workspace_and_validation(lib):
    import sliding_window_attention_router_gb300 as swa
    n = swa.prefill_backward_workspace(1, 32768, 16, 16, 128, 1024, swa.BF16)
    # compacted q and dO of far rows alone are twice the size of q
    assert n >= 2 * 32768 * 16 * 128 * 2 and n % 256 == 0
    assert swa.prefill_backward_workspace(1, 100, 6, 4, 128, 8, swa.BF16) == 0   # Hq % Hkv
    assert swa.prefill_backward_workspace(1, 256, 2, 2, 64, 32, swa.F32) == 256 * 2 * 4
    assert swa.route_backward_workspace(1000, 256, swa.BF16) >= 16 * 256 * 4
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    odd = vp((1 << 20) + 8)
    a10 = [fake] * 10
    # W < 1; Hq % Hkv; misaligned dq; bf16 d = 64 unsupported; workspace too small; null lse
    assert lib.swiattn_prefill_backward(*a10, 1, 64, 4, 4, 128, 0, 0.1, 1, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill_backward(*a10, 1, 64, 6, 4, 128, 8, 0.1, 1, fake, 1 << 30, None) == 1
    bad = a10[:7] + [odd] + a10[8:]
    assert lib.swiattn_prefill_backward(*bad, 1, 64, 4, 4, 128, 8, 0.1, 1, fake, 1 << 30, None) == 1
    assert lib.swiattn_prefill_backward(*a10, 1, 64, 4, 4, 64, 8, 0.1, 1, fake, 1 << 30, None) == 2
    assert lib.swiattn_prefill_backward(*a10, 1, 64, 4, 4, 128, 8, 0.1, 1, fake, 16, None) == 1
    nolse = a10[:5] + [None] + a10[6:]
    assert lib.swiattn_prefill_backward(*nolse, 1, 64, 4, 4, 128, 8, 0.1, 1, fake, 1 << 30, None) == 1
    r8 = [fake] * 8
    # hd not a multiple of 8; d_reg without gamma; dw without workspace; tokens 0 no-op
    assert lib.swiattn_route_backward(*r8, 10, 12, 16, 1, fake, None, None, None, None, 0, None) == 1
    nog = r8[:6] + [None, fake]
    assert lib.swiattn_route_backward(*nog, 10, 16, 16, 1, fake, None, None, None, None, 0, None) == 1
    assert lib.swiattn_route_backward(*r8, 10, 16, 16, 1, fake, None, fake, None, None, 0, None) == 1
    assert lib.swiattn_route_backward(*[None] * 8, 0, 16, 16, 1, None, None, None, None, None, 0,
                                      None) == 0


def test_decode_paged_validation(lib):
    import sliding_window_attention_router_gb300 as swa
    assert swa.decode_paged_workspace(16, 512, 64, 16, 16, 128, 1024, swa.BF16) == \
        swa.decode_workspace(16, 512 * 64, 16, 16, 128, 1024, swa.BF16)
    # anchors add whole 256-entry chunks of partials per sequence
    assert swa.decode_anchored_workspace(16, 32768, 16, 16, 128, 1024, 256, swa.BF16) == \
        swa.decode_workspace(16, 32768 + 256, 16, 16, 128, 1024, swa.BF16)
    assert swa.decode_paged_workspace(2, 8, 48, 4, 4, 128, 64, swa.BF16) == 0   # not a power of 2
    fake = ctypes.c_void_p(1 << 20)
    a8 = [fake] * 8
    # page size not a power of two; no pool pages; unsupported group size
    P = lib.swiattn_decode_paged
    assert P(*a8, 2, 8, 48, 16, 4, 4, 128, 64, 0, 0.1, 1, fake, 1 << 30, None) == 1
    assert P(*a8, 2, 8, 64, 0, 4, 4, 128, 64, 0, 0.1, 1, fake, 1 << 30, None) == 1
    assert P(*a8, 2, 8, 64, 16, 6, 2, 128, 64, 0, 0.1, 1, fake, 1 << 30, None) == 2
    # workspace too small; null block table; negative anchor count
    assert P(*a8, 2, 8, 64, 16, 4, 4, 128, 64, 0, 0.1, 1, fake, 8, None) == 1
    nt = a8[:3] + [None] + a8[4:]
    assert P(*nt, 2, 8, 64, 16, 4, 4, 128, 64, 0, 0.1, 1, fake, 1 << 30, None) == 1
    assert P(*a8, 2, 8, 64, 16, 4, 4, 128, 64, -1, 0.1, 1, fake, 1 << 30, None) == 1
    A = lib.swiattn_decode_anchored
    a7 = [fake] * 7
    assert A(*a7, 2, 64, 4, 4, 128, 8, -3, 0.1, 1, fake, 1 << 30, None) == 1


def test_no_gpu_reports_cuda_error_or_runs(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    assert lib.swiattn_num_sms() == -1


def _decode_chunk_len(m):
    """Chunk length of a decode visit of m = na + n cache entries (na anchors,
    then the window or history n): the smallest power of two from 64 up to 256
    tokens with chunk * 8 >= m.  The two segments never share a chunk."""
    c = 64
    while c < 256 and c * 8 < m:
        c *= 2
    return c


def test_decode_workspace_holds_every_chunk_partial(lib):
    """The split kernel writes one partial per (sequence, chunk, query head) and
    the combine reads them back; the workspace must hold the most chunks any
    visit of up to Lmax entries (plus up to S anchors) can have.  The partials
    come first; the last 256 bytes hold the split kernel's chunk counter."""
    import sliding_window_attention_router_gb300 as swa
    Hq, d = 256, 64                  # a chunk's partials: 256 * 66 floats = 67 584 bytes
    per_chunk = Hq * (d + 2) * 4
    for Lmax in (1, 7, 63, 64, 65, 200, 511, 512, 513, 1024, 1025, 2047, 2048, 2049, 4096, 5000):
        for S in (0, 1, 63, 64, 300, 4096):
            size = swa.decode_anchored_workspace(1, Lmax, Hq, Hq, d, 16, S, swa.BF16) - 256
            assert size % per_chunk == 0
            max_chunks = size // per_chunk
            for lo_span in range(1, Lmax + 1):
                n = lo_span                                  # visited window / history
                na = min(S, Lmax - n)                        # anchors below it
                m = na + n
                c = _decode_chunk_len(m)
                need = -(-na // c) + -(-n // c)
                assert need <= max_chunks, (Lmax, S, n, na, need, max_chunks)

"""GPU parity of the global-anchor variant of the routed prefill
(swiattn_prefill_anchored): window rows also attend the first S keys.

Against the fp64 oracle on the same seeded inputs (bf16 max-abs 2e-2 /
mean-abs 2e-3, fp32 1e-4) and with exact visited counts: with q = 0 every
visited key has the same score, so exp(lse) is the number of keys a row read,
compared as an integer with min(i+1, W) + min(S, i-W+1) (window rows) or i+1
(routed rows).
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


def expected_counts(gate, W, S):
    B, N = gate.shape
    i = np.arange(N)[None, :]
    window = np.minimum(i + 1, W) + np.clip(np.minimum(S, i - W + 1), 0, None)
    return np.where(gate != 0, i + 1, window)


CASES = [  # B, N, Hq, Hkv, W, S, frac
    (1, 2000, 4, 2, 256, 256, 0.13),
    (2, 777, 2, 2, 100, 300, 0.3),
    (1, 1500, 2, 1, 1024, 256, 0.0),
    (1, 300, 2, 2, 64, 1, 0.5),
    (1, 100, 2, 2, 1000, 256, 0.2),
    (1, 1000, 2, 2, 128, 5000, 0.1),
    (1, 700, 4, 4, 129, 129, 1.0),
    (1, 400, 2, 2, 64, 63, 0.2),     # 64-key block edges of the tensor-core kernel
    (1, 400, 2, 2, 65, 65, 0.2),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,W,S,frac", CASES)
def test_anchored_prefill_bf16(swa, B, N, Hq, Hkv, W, S, frac):
    g = inp._gen(N + S)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    gate = (torch.stack([inp.run_gates(N, frac, g) for _ in range(B)]) if 0 < frac < 1
            else torch.full((B, N), int(frac), dtype=torch.uint8))
    o = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W, n_anchor=S)
    assert swa.get_device_error() == 0
    ref = oracle.prefill_anchored(f64(q), f64(k), f64(v), gate.numpy(), W, S, 1 / math.sqrt(128))
    err = np.abs(f64(o) - ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    # exact visited counts
    _, lse = swa.prefill(torch.zeros_like(q).cuda(), k.cuda(), v.cuda(), gate.cuda(), W,
                         want_lse=True, n_anchor=S)
    got = np.rint(np.exp(f64(lse))).astype(np.int64)
    np.testing.assert_array_equal(got, expected_counts(gate.numpy(), W, S)[:, :, None].repeat(Hq, 2))


@pytest.mark.parametrize("d,W,S", [(64, 32, 16), (128, 50, 70)])
def test_anchored_prefill_fp32(swa, d, W, S):
    g = inp._gen(d + W)
    B, N, Hq, Hkv = 1, 300, 2, 1
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, d, torch.float32, g)
    gate = inp.bernoulli_gates((B, N), 0.13, g)
    o = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W, n_anchor=S)
    ref = oracle.prefill_anchored(f64(q), f64(k), f64(v), gate.numpy(), W, S, 1 / math.sqrt(d))
    assert np.abs(f64(o) - ref).max() <= 1e-4


def test_anchored_decode_equals_last_prefill_row(swa):
    """Decode with anchors reads what the last prefill row reads."""
    g = inp._gen(77)
    B, N, H, d, W, S = 1, 2300, 2, 128, 512, 256
    q, k, v = inp.attention_qkv(B, N, H, H, d, torch.bfloat16, g)
    gate = torch.zeros((B, N), dtype=torch.uint8)
    o = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W, n_anchor=S)
    od = swa.decode_anchored(q[:, -1].contiguous().cuda(), k.cuda(), v.cuda(),
                             torch.tensor([N], dtype=torch.int32).cuda(),
                             torch.zeros(1, dtype=torch.uint8).cuda(), W, S)
    assert swa.get_device_error() == 0
    assert (od.float() - o[:, -1].float()).abs().max().item() <= 2e-2

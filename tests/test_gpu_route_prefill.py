"""GPU parity of the fused router + routed prefill (swiattn_route_prefill):
one call computes the layer's router logits and hard gates and the routed
prefill those gates select.

The fused call must equal swiattn_route followed by swiattn_prefill_anchored
bit for bit (same logits, gates and outputs), across batches, ragged lengths,
GQA and anchors, and on a reused workspace (the counter that elects the
planning CTA resets every call).  Against the fp64 oracle: gates are
bit-exact wherever the oracle's logit is at least 1e-3 from 0, and the output
meets the bf16 tolerance (max-abs 2e-2, mean-abs 2e-3) with the oracle run on
the GPU's own gates.
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


def layer_inputs(B, N, Hq, Hkv, d_model, frac, seed, dtype=torch.bfloat16):
    r = inp.router_inputs(B * N, d_model, dtype, seed, frac=frac)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128 if dtype == torch.bfloat16 else 64, dtype,
                                r["gen"])
    return r["h"], r["w"], r["bias"], q, k, v


CASES = [  # B, N, Hq, Hkv, d_model, W, S, frac
    (1, 4096, 16, 16, 2048, 1024, 0, 0.13),
    (2, 3000, 16, 4, 1024, 512, 0, 0.3),
    (3, 777, 4, 2, 512, 100, 64, 0.2),
    (1, 129, 2, 2, 256, 1024, 0, 0.5),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,D,W,S,frac", CASES)
def test_fused_equals_route_then_prefill(swa, B, N, Hq, Hkv, D, W, S, frac):
    h, w, bias, q, k, v = (t.cuda() if isinstance(t, torch.Tensor) else t
                           for t in layer_inputs(B, N, Hq, Hkv, D, frac, seed=B * N + D))
    o, logits, gate = swa.route_prefill(h, w, bias, q, k, v, W, n_anchor=S)
    ref_logits, ref_gate = swa.route(h, w, bias)
    ref_o = swa.prefill(q, k, v, ref_gate.view(B, N), W, n_anchor=S)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    assert torch.equal(logits.view(-1), ref_logits)
    assert torch.equal(gate.view(-1), ref_gate)
    assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
    assert 0 < int(gate.sum()) < B * N


def test_workspace_reuse(swa):
    B, N, Hq, D, W = 2, 2048, 8, 1024, 256
    h, w, bias, q, k, v = (t.cuda() if isinstance(t, torch.Tensor) else t
                           for t in layer_inputs(B, N, Hq, Hq, D, 0.13, seed=5))
    ws = torch.empty(swa.route_prefill_workspace(B, N, Hq, Hq, 128, W, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    first = swa.route_prefill(h, w, bias, q, k, v, W, workspace=ws)[0].clone()
    for _ in range(3):
        again = swa.route_prefill(h, w, bias, q, k, v, W, workspace=ws)[0]
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    assert swa.get_device_error() == 0


def test_fused_against_oracle(swa):
    B, N, Hq, Hkv, D, W = 1, 1500, 4, 2, 512, 200
    h, w, bias, q, k, v = layer_inputs(B, N, Hq, Hkv, D, 0.2, seed=17)
    o, logits, gate = swa.route_prefill(h.cuda(), w.cuda(), bias, q.cuda(), k.cuda(), v.cuda(), W)
    torch.cuda.synchronize()
    ref_logits, _ = oracle.route(h.to(torch.float64), w.to(torch.float64), bias)
    ref_logits = np.asarray(ref_logits).reshape(-1)
    g = gate.view(-1).cpu().numpy()
    sure = np.abs(ref_logits) >= 1e-3
    assert sure.mean() > 0.99
    assert np.array_equal(g[sure], (ref_logits[sure] > 0).astype(np.uint8))
    assert np.array_equal(g, (logits.view(-1).cpu().numpy() > 0).astype(np.uint8))
    ref_o = oracle.prefill(q.to(torch.float64), k.to(torch.float64), v.to(torch.float64),
                           gate.view(B, N).cpu(), W, 1.0 / math.sqrt(128))
    err = np.abs(o.float().cpu().numpy().astype(np.float64) - ref_o)
    assert err.max() < 2e-2 and err.mean() < 2e-3


def test_fused_fp32(swa):
    B, N, Hq, D, W = 1, 256, 2, 64, 32
    h, w, bias, q, k, v = (t.cuda() if isinstance(t, torch.Tensor) else t
                           for t in layer_inputs(B, N, Hq, Hq, D, 0.13, seed=3,
                                                 dtype=torch.float32))
    o, logits, gate = swa.route_prefill(h, w, bias, q, k, v, W)
    ref_logits, ref_gate = swa.route(h, w, bias)
    ref_o = swa.prefill(q, k, v, ref_gate.view(B, N), W)
    torch.cuda.synchronize()
    assert torch.equal(logits.view(-1), ref_logits)
    assert torch.equal(gate.view(-1), ref_gate)
    assert torch.equal(o, ref_o)

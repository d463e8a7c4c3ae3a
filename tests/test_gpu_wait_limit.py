"""Failure detection on the GPU without a fault: a device wait that runs out.

Every wait of the tensor-core kernels on a shared-memory barrier is bounded.
When one runs out, the waiter raises its CTA's abort flag and records a
timeout in the device error word; every role of the CTA then leaves its loop,
waits (with a separate fixed bound) for its own copies and tensor-core
operations still in flight, and the CTA frees its tensor memory and exits.

These tests lower the limit to 1 ns through the library's test aid
(swiattn_set_wait_limit_ns).  Below 0.1 ms a waiter polls instead of
suspending, at most `limit` times, so the first wait that is not complete at
once gives up; the
long-context shapes have many such waits (a warp waiting for the next item's
query slot waits about one far item).  Each
test then checks that swiattn_get_device_error reports SWIATTN_ETIMEOUT,
restores the default limit and checks that the next call on the same context
matches the oracle.  (A wait first tries the barrier with one potentially
blocking try_wait, which the hardware may hold until the phase completes; the
backward kernels' waits are all short enough to end there, so the limit does
not reach them and they are not tested this way.)
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swiattn_inputs as inp

pytestmark = pytest.mark.gpu

SWIATTN_ETIMEOUT = 4


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


def status_under_tiny_limit(swa, call):
    """Run `call` with a 1 ns wait limit; return the device error it left."""
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    swa.set_wait_limit_ns(1)
    try:
        call()
        torch.cuda.synchronize()
        return swa.get_device_error()
    finally:
        swa.set_wait_limit_ns(0)


def small_prefill_matches_oracle(swa):
    g = inp._gen(901)
    B, N, H, W = 1, 1500, 2, 256
    q, k, v = inp.attention_qkv(B, N, H, H, 128, torch.bfloat16, g)
    gate = inp.run_gates(N, 0.2, g, mean_run=32.0).reshape(B, N)
    o = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ref = oracle.prefill(f64(q), f64(k), f64(v), gate.numpy(), W, 1 / math.sqrt(128))
    err = np.abs(f64(o) - ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_prefill_wait_expiry_reports_timeout_then_recovers(swa):
    d = inp.prefill_32k(frac=0.13, seed=0)
    q, k, v, gate = (d[n].cuda() for n in ("q", "k", "v", "gate"))
    st = status_under_tiny_limit(swa, lambda: swa.prefill(q, k, v, gate, d["W"]))
    assert st == SWIATTN_ETIMEOUT
    small_prefill_matches_oracle(swa)
    # the full-size call under the default limit is complete and finite again
    o = swa.prefill(q, k, v, gate, d["W"])
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    assert torch.isfinite(o.float()).all()


def test_dual_branch_wait_expiry_reports_timeout_then_recovers(swa):
    d = inp.dual_8k(seed=0, B=1, N=32768)
    args = [d[n].cuda() for n in ("q", "k", "v", "logits", "nll")]
    st = status_under_tiny_limit(swa, lambda: swa.dual_branch(*args, d["W"]))
    assert st == SWIATTN_ETIMEOUT
    g = inp._gen(902)
    B, N, Hq, Hkv, W = 1, 1200, 4, 2, 200
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    logits = inp.logits_with_margin((B, N), g)
    nll = torch.ones(B, N)
    out = swa.dual_branch(q.cuda(), k.cuda(), v.cuda(), logits.cuda(), nll.cuda(), W)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ref = oracle.dual(f64(q), f64(k), f64(v), f64(logits), f64(nll), W, 1 / math.sqrt(128))
    for name in ("o_full", "o_swa"):
        err = np.abs(f64(out[name]) - ref[name])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, name

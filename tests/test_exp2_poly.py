"""Error bound of the FMA-pipe 2^x used for part of the softmax weights.

The kernel evaluates 2^x as 2^round(x) * q(f), f = x - round(x) in [-1/2, 1/2],
with a degree-3 polynomial q whose coefficients are read here from the CUDA
header; the fp32 steps are replayed with numpy float32 arithmetic and compared
with exp2 in float64 over the range the softmax uses (scores minus the running
maximum: at most 8 above it, clamped 125 below).
"""
import os
import re

import numpy as np

PTX = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "sliding_window_attention_router_gb300", "csrc", "ptx.cuh")


def _coeffs():
    text = open(PTX).read()
    return [np.float32(float(re.search(rf"kExp2C{k}\s*=\s*([0-9.eE+-]+)f", text).group(1)))
            for k in range(4)]


def _exp2_fp32(x):
    c0, c1, c2, c3 = _coeffs()
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    shift = np.float32(12582912.0)
    t = (x + shift).astype(np.float32)
    r = (t - shift).astype(np.float32)
    f = (x - r).astype(np.float32)
    q = (c3 * f + c2).astype(np.float32)
    q = (q * f + c1).astype(np.float32)
    q = (q * f + c0).astype(np.float32)
    bits = (q.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_relative_error_below_bf16_rounding():
    x = np.concatenate([np.linspace(-125.0, 9.0, 2_000_001), np.arange(-125, 10) + 0.5,
                        np.arange(-125, 10).astype(np.float64)]).astype(np.float32)
    got = _exp2_fp32(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    # bf16 keeps 8 significant bits (rounding error up to 2^-9 ~ 2e-3); the
    # polynomial must stay far below that.
    assert rel.max() < 1e-4, rel.max()


def test_clamped_tail_is_tiny_and_positive():
    got = _exp2_fp32(np.array([-200.0, -126.0, -125.0], np.float32))
    assert np.all(got > 0) and np.all(got < 3e-38)

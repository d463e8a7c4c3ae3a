"""Pins of the oracle's global-anchor variant (SWA glossary: every query also
attends the first S tokens, which the window never evicts).

The visited set is recovered from attention outputs (q = 0 gives uniform
weights, one-hot values expose which keys were averaged) and compared with
the glossary's W=4 table OR'd with the anchor columns; S = 0 must reproduce
plain sliding-window attention exactly, S >= N causal attention, and routed
rows must be unaffected.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _w4_table():
    rows, W = [], None
    with open(os.path.join(GOLDEN, "swa_w4_n7_mask.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("# W"):
                W = int(line.split()[2])
            elif line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return W, np.array(rows, dtype=np.int64)


def _visited_from_outputs(S, gate, W, N):
    """q = 0: every visited key gets weight 1/n; v_j = e_j recovers the set."""
    q = np.zeros((1, N, 1, N))
    k = np.random.default_rng(0).standard_normal((1, N, 1, N))
    v = np.zeros((1, N, 1, N))
    v[0, np.arange(N), 0, np.arange(N)] = 1.0
    o = oracle.prefill_anchored(q, k, v, gate, W, S, 0.5)
    return (o[0, :, 0, :] > 0).astype(np.int64), o


@pytest.mark.parametrize("S", [1, 2, 3])
def test_anchored_w4_table(S):
    W, table = _w4_table()
    N = table.shape[0]
    vis, o = _visited_from_outputs(S, np.zeros((1, N), np.uint8), W, N)
    expect = table.copy()
    causal = np.tril(np.ones((N, N), np.int64))
    expect[:, :S] = causal[:, :S]
    np.testing.assert_array_equal(vis, expect)
    # uniform weights over the visited keys
    np.testing.assert_allclose(o[0, :, 0, :].sum(axis=1), 1.0, rtol=1e-14)


def test_zero_anchors_is_plain_window():
    rng = np.random.default_rng(3)
    B, N, Hq, Hkv, d, W = 2, 40, 4, 2, 8, 5
    q, k, v = (rng.standard_normal((B, N, h, d)) for h in (Hq, Hkv, Hkv))
    gate = (rng.random((B, N)) < 0.3).astype(np.uint8)
    a, la = oracle.prefill_anchored(q, k, v, gate, W, 0, 0.4, want_lse=True)
    b, lb = oracle.prefill(q, k, v, gate, W, 0.4, want_lse=True)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_anchors_cover_everything_is_causal_and_routed_rows_unchanged():
    rng = np.random.default_rng(4)
    B, N, H, d, W = 1, 30, 2, 8, 4
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    zeros, ones = np.zeros((B, N), np.uint8), np.ones((B, N), np.uint8)
    np.testing.assert_array_equal(oracle.prefill_anchored(q, k, v, zeros, W, N, 0.3),
                                  oracle.prefill(q, k, v, ones, W, 0.3))
    gate = (rng.random((B, N)) < 0.5).astype(np.uint8)
    a = oracle.prefill_anchored(q, k, v, gate, W, 7, 0.3)
    b = oracle.prefill(q, k, v, ones, W, 0.3)
    routed = gate[0] != 0
    np.testing.assert_array_equal(a[0, routed], b[0, routed])


def test_decode_anchored_equals_last_prefill_row():
    rng = np.random.default_rng(5)
    N, Hq, Hkv, d, W, S = 50, 4, 2, 8, 6, 9
    q, k, v = (rng.standard_normal((1, N, h, d)) for h in (Hq, Hkv, Hkv))
    for g in (0, 1):
        gate = np.full((1, N), g, np.uint8)
        full = oracle.prefill_anchored(q, k, v, gate, W, S, 0.3)
        o = oracle.decode_anchored(q[:, -1], k, v, [N], [g], W, S, 0.3)
        np.testing.assert_allclose(o, full[:, -1], rtol=0, atol=1e-15)


def test_lse_counts_anchored_keys():
    """q = 0: lse = ln(number of visited keys) = ln(min(S, i-W+1) + min(i+1, W))."""
    N, W, S = 60, 10, 4
    q = np.zeros((1, N, 1, 4))
    k = np.random.default_rng(6).standard_normal((1, N, 1, 4))
    v = np.ones((1, N, 1, 4))
    _, lse = oracle.prefill_anchored(q, k, v, np.zeros((1, N), np.uint8), W, S, 1.0,
                                     want_lse=True)
    i = np.arange(N)
    n = np.minimum(i + 1, W) + np.clip(np.minimum(S, i - W + 1), 0, None)
    np.testing.assert_allclose(lse[0, :, 0], np.log(n), rtol=0, atol=1e-13)

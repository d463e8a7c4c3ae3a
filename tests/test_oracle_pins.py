"""Pins of the fp64 oracle against what the pages and mathematics fix.

Each test ties the oracle to something other than itself: the glossary's W=4
visibility table, the FAQ's W=N equivalence, the report's gated-sum special
cases and regulariser constants, closed-form softmax examples, and library
routines (scipy softmax / expit, numpy logaddexp) on tiny inputs.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    meta, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line:
                continue
            if line.startswith("#"):
                parts = line[1:].split()
                if len(parts) == 2 and parts[0] in ("W", "N"):
                    meta[parts[0]] = int(parts[1])
                continue
            rows.append([int(x) for x in line.split()])
    return meta, np.array(rows, dtype=np.int64)


def _read_constants(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# Window definition: the glossary's W=4, 7-token table.
# --------------------------------------------------------------------------
def test_w4_table_ranges():
    meta, table = _read_table("swa_w4_n7_mask.txt")
    W, N = meta["W"], meta["N"]
    lo, hi = oracle.row_ranges(np.zeros((1, N), np.uint8), W)
    vis = np.zeros((N, N), np.int64)
    for i in range(N):
        vis[i, lo[0, i]:hi[0, i] + 1] = 1
    np.testing.assert_array_equal(vis, table)


def test_w4_table_from_attention_outputs():
    """q = 0 gives uniform weights over the visited keys; one-hot values
    v_j = e_j make o_i the indicator of the visited set divided by its size."""
    meta, table = _read_table("swa_w4_n7_mask.txt")
    W, N = meta["W"], meta["N"]
    d = 8
    q = np.zeros((1, N, 1, d))
    k = _rand((1, N, 1, d), 1)
    v = np.zeros((1, N, 1, d))
    for j in range(N):
        v[0, j, 0, j] = 1.0
    o = oracle.prefill(q, k, v, np.zeros((1, N), np.uint8), W, scale=0.7)
    got = o[0, :, 0, :N]
    n = table.sum(1, keepdims=True)
    np.testing.assert_array_equal(got > 0, table.astype(bool))
    np.testing.assert_allclose(got, table / n, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# FAQ: W >= N is the causal mask, i.e. full attention.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("W_extra", [0, 5])
def test_window_ge_n_equals_full(W_extra):
    B, N, H, d = 2, 23, 2, 8
    q, k, v = _rand((B, N, H, d), 2), _rand((B, N, H, d), 3), _rand((B, N, H, d), 4)
    W = N + W_extra
    o_swa = oracle.prefill(q, k, v, np.zeros((B, N), np.uint8), W, 0.3)
    o_full = oracle.prefill(q, k, v, np.ones((B, N), np.uint8), W, 0.3)
    np.testing.assert_array_equal(o_swa, o_full)


# --------------------------------------------------------------------------
# Report, gated output O = s*O_FULL + (1-s)*O_SWA with a hard 0/1 gate.
# --------------------------------------------------------------------------
def test_gate_selects_branch():
    B, N, H, d, W = 1, 40, 3, 4, 6
    q, k, v = _rand((B, N, H, d), 5), _rand((B, N, H, d), 6), _rand((B, N, H, d), 7)
    gate = (np.random.default_rng(8).random((B, N)) < 0.4).astype(np.uint8)
    o = oracle.prefill(q, k, v, gate, W, 0.5)
    o_full = oracle.prefill(q, k, v, np.ones_like(gate), W, 0.5)
    o_swa = oracle.prefill(q, k, v, np.zeros_like(gate), W, 0.5)
    g = gate[..., None, None].astype(np.float64)
    np.testing.assert_array_equal(o, g * o_full + (1 - g) * o_swa)
    # and the two branches really differ beyond the window
    assert np.abs(o_full[:, W:] - o_swa[:, W:]).max() > 1e-3


def test_window_one_returns_own_value():
    B, N, H, d = 1, 9, 2, 4
    q, k, v = _rand((B, N, H, d), 9), _rand((B, N, H, d), 10), _rand((B, N, H, d), 11)
    o = oracle.prefill(q, k, v, np.zeros((B, N), np.uint8), 1, 1.0)
    np.testing.assert_array_equal(o, v)


def test_row_zero_is_first_value():
    B, N, H, d = 1, 9, 2, 4
    q, k, v = _rand((B, N, H, d), 12), _rand((B, N, H, d), 13), _rand((B, N, H, d), 14)
    for gate in (np.zeros((B, N), np.uint8), np.ones((B, N), np.uint8)):
        o = oracle.prefill(q, k, v, gate, 3, 1.0)
        np.testing.assert_array_equal(o[:, 0], v[:, 0])


def test_gqa_contiguous_groups():
    """Hq=4 query heads on Hkv=2 KV heads: constant values per KV head give each
    query head its group's constant; heads 0,1 read KV head 0, heads 2,3 head 1."""
    B, N, Hq, Hkv, d = 1, 17, 4, 2, 3
    q, k = _rand((B, N, Hq, d), 15), _rand((B, N, Hkv, d), 16)
    v = np.zeros((B, N, Hkv, d))
    v[:, :, 0, :] = 3.0
    v[:, :, 1, :] = -7.0
    gate = (np.arange(N) % 3 == 0).astype(np.uint8)[None]
    o = oracle.prefill(q, k, v, gate, 4, 0.9)
    np.testing.assert_allclose(o[:, :, :2], 3.0, rtol=1e-14)
    np.testing.assert_allclose(o[:, :, 2:], -7.0, rtol=1e-14)


def _three_token_example():
    """k_j = e_j, q_2 = (0, ln 2, ln 5)/scale: row 2's full-branch weights are
    (1, 2, 5)/8 and its W=2 window weights (2, 5)/7; v_j = 8 e_j."""
    scale = 0.25
    d = 3
    k = np.eye(3).reshape(1, 3, 1, d)
    q = np.zeros((1, 3, 1, d))
    q[0, 0, 0] = [0.4, -0.2, 0.0]
    q[0, 1, 0] = [0.1, 0.3, 0.0]
    q[0, 2, 0] = [0.0, math.log(2.0) / scale, math.log(5.0) / scale]
    v = 8.0 * np.eye(3).reshape(1, 3, 1, d)
    return q, k, v, scale


def test_closed_form_three_tokens():
    q, k, v, scale = _three_token_example()
    o_full = oracle.prefill(q, k, v, np.ones((1, 3), np.uint8), 2, scale)
    o_swa = oracle.prefill(q, k, v, np.zeros((1, 3), np.uint8), 2, scale)
    np.testing.assert_allclose(o_full[0, 2, 0], [1.0, 2.0, 5.0], rtol=1e-13)
    np.testing.assert_allclose(o_swa[0, 2, 0], [0.0, 16.0 / 7.0, 40.0 / 7.0], rtol=1e-13,
                               atol=1e-15)
    # row 1 full branch: weights exp(scale*q1.k0), exp(scale*q1.k1)
    a, b = math.exp(scale * 0.1), math.exp(scale * 0.3)
    np.testing.assert_allclose(o_full[0, 1, 0], [8 * a / (a + b), 8 * b / (a + b), 0.0],
                               rtol=1e-13)


def test_lse_counts_visited_keys():
    """q = 0: every score is 0, so lse = log(number of visited keys)."""
    B, N, H, d, W = 2, 70, 2, 4, 9
    q = np.zeros((B, N, H, d))
    k, v = _rand((B, N, H, d), 17), _rand((B, N, H, d), 18)
    gate = (np.random.default_rng(19).random((B, N)) < 0.3).astype(np.uint8)
    _, lse = oracle.prefill(q, k, v, gate, W, 1.0, want_lse=True)
    i = np.arange(N)[None, :]
    n = np.where(gate == 1, i + 1, np.minimum(i + 1, W))
    np.testing.assert_allclose(lse, np.log(n)[..., None].repeat(H, -1), rtol=0, atol=1e-13)


def test_matches_library_softmax_bruteforce():
    """Explicit mask matrix + scipy.special.softmax on tiny inputs."""
    B, N, Hq, Hkv, d, W, scale = 2, 31, 4, 2, 5, 7, 0.37
    q, k, v = _rand((B, N, Hq, d), 20), _rand((B, N, Hkv, d), 21), _rand((B, N, Hkv, d), 22)
    gate = (np.random.default_rng(23).random((B, N)) < 0.3).astype(np.uint8)
    o, lse = oracle.prefill(q, k, v, gate, W, scale, want_lse=True)
    for b in range(B):
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            s = scale * q[b, :, h] @ k[b, :, kv].T
            ii, jj = np.meshgrid(np.arange(N), np.arange(N), indexing="ij")
            visible = (jj <= ii) & ((gate[b][:, None] == 1) | (jj >= ii - W + 1))
            s = np.where(visible, s, -np.inf)
            np.testing.assert_allclose(o[b, :, h], scipy.special.softmax(s, axis=1) @ v[b, :, kv],
                                       rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[b, :, h], scipy.special.logsumexp(s, axis=1),
                                       rtol=1e-13)


def test_prefill_rows_matches_all_rows():
    B, N, Hq, Hkv, d, W = 2, 50, 4, 2, 6, 8
    q, k, v = _rand((B, N, Hq, d), 24), _rand((B, N, Hkv, d), 25), _rand((B, N, Hkv, d), 26)
    gate = (np.random.default_rng(27).random((B, N)) < 0.3).astype(np.uint8)
    o, lse = oracle.prefill(q, k, v, gate, W, 0.2, want_lse=True)
    sel = np.array([[0, 0, 0], [1, 49, 3], [0, 17, 2], [1, 8, 1]])
    o_s, lse_s = oracle.prefill_rows(q, k, v, gate, W, 0.2, sel, want_lse=True)
    for r, (b, i, h) in enumerate(sel):
        np.testing.assert_array_equal(o_s[r], o[b, i, h])
        assert lse_s[r] == lse[b, i, h]


# --------------------------------------------------------------------------
# Router: gate = 1(sigmoid(R(h)) > 0.5), R linear.
# --------------------------------------------------------------------------
def test_route_closed_form_and_threshold():
    D = 6
    w = np.array([0.5, -0.25, 1.0, 2.0, -1.5, 0.125])
    h = np.ones((3, D))
    h[1] *= -1.0
    h[2] = 0.0
    logits, gate = oracle.route(h, w, bias=-1.875)
    # sum(w) = 1.875: logits exactly 0, -3.75, -1.875
    np.testing.assert_array_equal(logits, [0.0, -3.75, -1.875])
    np.testing.assert_array_equal(gate, [0, 0, 0])  # strict: sigmoid(0) = 0.5 is not > 0.5
    logits, gate = oracle.route(h, w, bias=-1.8)
    np.testing.assert_array_equal(gate, [1, 0, 0])


def test_route_matches_sigmoid_threshold():
    rng = np.random.default_rng(28)
    T, D = 500, 64
    h, w = rng.standard_normal((T, D)), rng.standard_normal(D) / 8
    logits, gate = oracle.route(h, w, 0.3)
    np.testing.assert_allclose(logits, h @ w + 0.3, rtol=1e-12, atol=1e-12)
    keep = np.abs(logits) > 1e-9
    np.testing.assert_array_equal(gate[keep], (scipy.special.expit(logits[keep]) > 0.5)[...])


# --------------------------------------------------------------------------
# Regulariser: constants and closed forms.
# --------------------------------------------------------------------------
def test_regulariser_constants_closed_forms():
    c = _read_constants("regulariser_constants.txt")
    gb, eps, alpha = c["gamma_base"], c["eps"], c["alpha"]
    # NLL = 0, mse = 0, logit = 0: gamma = gb/eps = 1e-2, softplus(0) = ln 2
    g, r = oracle.regulariser([0.0], [0.0], [0.0], gb, eps, alpha)
    assert g[0] == pytest.approx(1e-2, rel=1e-15)
    assert r[0] == pytest.approx(1e-2 * math.log(2.0), rel=1e-15)
    # NLL = 1, mse = 0.01, logit = 2: gamma = 1e-3/2.1, softplus(2) = ln(1+e^2)
    g, r = oracle.regulariser([2.0], [1.0], [0.01], gb, eps, alpha)
    assert g[0] == pytest.approx(1e-3 / 2.1, rel=1e-14)
    assert r[0] == pytest.approx(1.0128228624014155e-3, rel=1e-14)
    # the weight falls as either difficulty signal grows
    g2, _ = oracle.regulariser([0.0, 0.0], [3.0, 0.0], [0.0, 0.03], gb, eps, alpha)
    assert g2[0] < 1e-2 and g2[1] < 1e-2
    assert g2[0] == pytest.approx(1e-3 / 3.1) and g2[1] == pytest.approx(1e-3 / 3.1)


@pytest.mark.parametrize("x", [-745.0, -60.0, -1.0, -1e-8, 0.0, 1e-8, 0.7, 30.0, 60.0, 700.0])
def test_softplus_matches_logaddexp(x):
    assert oracle.softplus(x) == pytest.approx(float(np.logaddexp(0.0, x)), rel=1e-15, abs=0)


# --------------------------------------------------------------------------
# Dual branch.
# --------------------------------------------------------------------------
def test_dual_closed_form_mse():
    q, k, v, scale = _three_token_example()
    logits = np.array([[0.0, 1.0, 2.0]])
    nll = np.array([[0.5, 0.5, 1.0]])
    out = oracle.dual(q, k, v, logits, nll, 2, scale)
    # rows 0, 1 are inside the window: identical branches
    assert out["mse"][0, 0] == 0.0 and out["mse"][0, 1] == 0.0
    # row 2: (1-0)^2 + (2-16/7)^2 + (5-40/7)^2 = 1 + 4/49 + 25/49
    assert out["mse"][0, 2] == pytest.approx(78.0 / 49.0, rel=1e-13)
    g = 1e-3 / (0.1 + 1.0 + 100.0 * 78.0 / 49.0)
    assert out["gamma"][0, 2] == pytest.approx(g, rel=1e-13)
    assert out["reg"][0, 2] == pytest.approx(g * float(np.logaddexp(0, 2.0)), rel=1e-13)


def test_dual_branches_equal_prefill_and_zero_inside_window():
    B, N, Hq, Hkv, d, W = 2, 45, 4, 2, 6, 11
    q, k, v = _rand((B, N, Hq, d), 29), _rand((B, N, Hkv, d), 30), _rand((B, N, Hkv, d), 31)
    logits, nll = _rand((B, N), 32), np.abs(_rand((B, N), 33))
    out = oracle.dual(q, k, v, logits, nll, W, 0.4)
    np.testing.assert_array_equal(out["o_full"], oracle.prefill(q, k, v, np.ones((B, N)), W, 0.4))
    np.testing.assert_array_equal(out["o_swa"], oracle.prefill(q, k, v, np.zeros((B, N)), W, 0.4))
    assert np.all(out["mse"][:, :W] == 0.0)
    assert np.all(out["mse"][:, W:] > 0.0)
    mse = ((out["o_full"] - out["o_swa"]) ** 2).sum(axis=(2, 3))
    np.testing.assert_allclose(out["mse"], mse, rtol=1e-12)
    g, r = oracle.regulariser(logits.ravel(), nll.ravel(), out["mse"].ravel())
    np.testing.assert_array_equal(out["gamma"].ravel(), g)
    np.testing.assert_array_equal(out["reg"].ravel(), r)
    sel = np.array([[1, 44], [0, 3], [1, 11]])
    rows = oracle.dual_rows(q, k, v, logits, nll, W, 0.4, sel)
    for r_, (b, i) in enumerate(sel):
        np.testing.assert_array_equal(rows["o_full"][r_], out["o_full"][b, i])
        np.testing.assert_array_equal(rows["o_swa"][r_], out["o_swa"][b, i])
        assert rows["mse"][r_] == out["mse"][b, i]
        assert rows["reg"][r_] == out["reg"][b, i]


# --------------------------------------------------------------------------
# Decode over a shared cache.
# --------------------------------------------------------------------------
def test_decode_visited_set_one_hot():
    """q = 0 and one-hot values recover the visited cache entries: the last W
    for a window token, all L for a routed one."""
    B, Lmax, H, W = 4, 24, 1, 5
    d = Lmax
    seq_lens = np.array([24, 3, 17, 9], np.int32)
    gate = np.array([0, 0, 1, 1], np.uint8)
    q = np.zeros((B, H, d))
    kc = _rand((B, Lmax, H, d), 34)
    vc = np.zeros((B, Lmax, H, d))
    for j in range(Lmax):
        vc[:, j, 0, j] = 1.0
    o = oracle.decode(q, kc, vc, seq_lens, gate, W, 1.0)
    for b in range(B):
        L = int(seq_lens[b])
        lo = 0 if gate[b] else max(0, L - W)
        want = np.zeros(d)
        want[lo:L] = 1.0 / (L - lo)
        np.testing.assert_allclose(o[b, 0], want, rtol=0, atol=1e-15)


def test_decode_equals_last_prefill_row():
    B, N, Hq, Hkv, d, W = 3, 33, 4, 2, 8, 6
    q, k, v = _rand((B, N, Hq, d), 35), _rand((B, N, Hkv, d), 36), _rand((B, N, Hkv, d), 37)
    gate = np.array([[0] * N, [1] * N, [0] * N], np.uint8)
    gate[2, -1] = 1
    o = oracle.prefill(q, k, v, gate, W, 0.3)
    od = oracle.decode(q[:, -1], k, v, np.full(B, N, np.int32), gate[:, -1], W, 0.3)
    np.testing.assert_array_equal(od, o[:, -1])


def test_invalid_arguments_rejected():
    q = np.zeros((1, 4, 3, 2))
    k = np.zeros((1, 4, 2, 2))
    with pytest.raises(ValueError):
        oracle.prefill(q, k, k, np.zeros((1, 4)), 2, 1.0)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.decode(np.zeros((1, 1, 2)), np.zeros((1, 4, 1, 2)), np.zeros((1, 4, 1, 2)),
                      [5], [0], 2, 1.0)  # seq_len > Lmax

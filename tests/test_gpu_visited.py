"""GPU: each row's visited key set, exactly.

The routed method fixes, per query row i, the set of keys its softmax covers:
[max(0, i-W+1), i] for a window row and [0, i] for a routed row (SwiAttn
report, section 2; the window is the SWA glossary's definition and its W=4
table), optionally with the first S keys added to window rows (the glossary's
global anchors).  An output that is close to the oracle's does not prove that
the kernel visited exactly that set: a window shifted by one key at a block
edge changes a row's output by less than the bf16 tolerance.  So the set is
read back from the production kernels with position probes:

- count probe: q = 0 gives every visited key the same score, so exp(lse) is
  the number of keys the row's softmax summed (an integer);
- max probe: key j carries its position in two bf16-exact digits and the
  query weighs them so that the score is 16 j; every other visited key then
  has weight at most e^-16 of the largest, so the output is the value row of
  the largest visited key, whose columns hold the bits of its position;
- min probe: the same with the sign flipped (score -16 j).

A set of distinct integers whose smallest element is lo, whose largest is hi
and whose size is hi - lo + 1 is exactly [lo, hi].  A key counted twice shows
up in the count.  For anchored rows, whose set is two runs, two more probes
restrict the maximum to keys below S and the minimum to keys from S on (a
large negative score on the other side), which pins each run's inner end.

Expected values come from the oracle: its row ranges for the plain sets, and
for anchored sets the oracle's own attention on the same probe inputs
(decoded the same way).  Everything is compared as integers.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swiattn_inputs as inp

pytestmark = pytest.mark.gpu

NBITS = 16          # positions below 65536
STEP = 16.0         # score gap between consecutive keys in the min/max probes
BIG = float(1 << 20)


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


def probe_kv(B, N, Hkv, d, dtype, S=None, device="cuda"):
    """Keys: [j >> 8, j & 255, (j >= S)] in the first columns; values: the
    bits of j.  All values are exact in bf16."""
    j = torch.arange(N, device=device)
    k = torch.zeros(B, N, Hkv, d, dtype=dtype, device=device)
    k[..., 0] = (j >> 8).to(dtype)[None, :, None]
    k[..., 1] = (j & 255).to(dtype)[None, :, None]
    if S is not None:
        k[..., 2] = (j >= S).to(dtype)[None, :, None]
    v = torch.zeros(B, N, Hkv, d, dtype=dtype, device=device)
    for c in range(NBITS):
        v[..., c] = ((j >> c) & 1).to(dtype)[None, :, None]
    return k, v


def probe_q(shape, d, dtype, sign, restrict=0.0):
    """Queries scoring key j as sign * 16 j (+ restrict * (j >= S))."""
    q = torch.zeros(*shape, d, dtype=torch.float32)
    q[..., 0] = sign * STEP * 256
    q[..., 1] = sign * STEP
    q[..., 2] = restrict
    return q.to(dtype)


def decode_position(o):
    """Position held in the bits of each output row (rounded per column)."""
    bits = np.rint(f64(o)[..., :NBITS]).astype(np.int64)
    assert np.all((bits == 0) | (bits == 1))
    return (bits << np.arange(NBITS)).sum(-1)


def count_of(lse):
    return np.rint(np.exp(f64(lse))).astype(np.int64)


def prefill_probes(swa, gate, Hq, Hkv, W, dtype, S=0):
    """(count, min, max) of every row and head, plus for anchors the maximum
    below S and the minimum from S on; each [B, N, Hq]."""
    B, N = gate.shape
    d = 128 if dtype == torch.bfloat16 else 64
    k, v = probe_kv(B, N, Hkv, d, dtype, S if S else None)
    g = gate.cuda()
    res = {}
    _, lse = swa.prefill(torch.zeros(B, N, Hq, d, dtype=dtype).cuda(), k, v, g, W, 1.0,
                         want_lse=True, n_anchor=S)
    res["count"] = count_of(lse)
    for name, sign, restrict in (("min", -1.0, 0.0), ("max", 1.0, 0.0),
                                 ("max_below_S", 1.0, -BIG), ("min_from_S", -1.0, BIG)):
        if restrict and not S:
            continue
        # min_from_S: keys below S get +BIG * 0, keys from S on -16 j + BIG
        q = probe_q((B, N, Hq), d, dtype, sign, restrict)
        o = swa.prefill(q.cuda(), k, v, g, W, 1.0, n_anchor=S)
        res[name] = decode_position(o)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    return res


def expected_plain(gate, W, Hq):
    lo, hi = oracle.row_ranges(gate.numpy(), W)
    rep = lambda a: np.repeat(a[..., None], Hq, -1)
    return {"count": rep(hi - lo + 1), "min": rep(lo), "max": rep(hi)}


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


EDGE = [
    # B, N, Hq, Hkv, W, gate pattern (tile, block and window edges of the kernels)
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
    (1, 64, 2, 2, 64, "rand"),
    (1, 65, 2, 2, 63, "rand"),
    (1, 191, 2, 2, 65, "runs"),
    (1, 193, 2, 2, 127, "alt"),
    (2, 257, 2, 2, 65, "rand"),
    (1, 4100, 2, 2, 1024, "runs"),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,N,Hq,Hkv,W,pattern", EDGE)
def test_prefill_visited_sets_exact(swa, dtype, B, N, Hq, Hkv, W, pattern):
    if dtype == torch.float32 and N > 1000:
        pytest.skip("the fp32 path is checked on the short shapes")
    gate = _gate(pattern, B, N, inp._gen(300 + N + W))
    got = prefill_probes(swa, gate, Hq, Hkv, W, dtype)
    want = expected_plain(gate, W, Hq)
    for key in ("count", "min", "max"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


@pytest.mark.parametrize("frac", [0.13, 0.05])
def test_prefill_32k_visited_sets_exact(swa, frac):
    """The long-context workload's gates: every row and head of the 32K
    sequence, through the same kernel and launch as the benchmark."""
    d = inp.prefill_32k(frac=frac, seed=0)
    got = prefill_probes(swa, d["gate"], d["Hq"], d["Hkv"], d["W"], torch.bfloat16)
    want = expected_plain(d["gate"], d["W"], d["Hq"])
    for key in ("count", "min", "max"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


ANCHORED = [  # B, N, Hq, Hkv, W, S, routed fraction
    (1, 2000, 4, 2, 256, 256, 0.13),
    (2, 777, 2, 2, 100, 300, 0.3),
    (1, 1500, 2, 1, 1024, 256, 0.0),
    (1, 300, 2, 2, 64, 1, 0.5),
    (1, 1000, 2, 2, 128, 5000, 0.1),
    (1, 400, 2, 2, 64, 63, 0.2),
    (1, 400, 2, 2, 65, 65, 0.2),
]


def oracle_anchored_probes(gate, Hq, Hkv, W, S, dtype):
    B, N = gate.shape
    d = 128 if dtype == torch.bfloat16 else 64
    k, v = probe_kv(B, N, Hkv, d, dtype, S, device="cpu")
    k64, v64 = f64(k), f64(v)
    res = {}
    _, lse = oracle.prefill_anchored(np.zeros((B, N, Hq, d)), k64, v64, gate.numpy(), W, S, 1.0,
                                     want_lse=True)
    res["count"] = np.rint(np.exp(lse)).astype(np.int64)
    for name, sign, restrict in (("min", -1.0, 0.0), ("max", 1.0, 0.0),
                                 ("max_below_S", 1.0, -BIG), ("min_from_S", -1.0, BIG)):
        q = f64(probe_q((B, N, Hq), d, dtype, sign, restrict))
        o = oracle.prefill_anchored(q, k64, v64, gate.numpy(), W, S, 1.0)
        res[name] = decode_position(torch.from_numpy(o))
    return res


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,N,Hq,Hkv,W,S,frac", ANCHORED)
def test_anchored_prefill_visited_sets_exact(swa, dtype, B, N, Hq, Hkv, W, S, frac):
    g = inp._gen(400 + N + S)
    gate = (torch.stack([inp.run_gates(N, frac, g) for _ in range(B)]) if 0 < frac < 1
            else torch.full((B, N), int(frac), dtype=torch.uint8))
    got = prefill_probes(swa, gate, Hq, Hkv, W, dtype, S=S)
    want = oracle_anchored_probes(gate, Hq, Hkv, W, S, dtype)
    for key in want:
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


def decode_probes(swa, q_shape, Lmax, Hkv, d, dtype, sl, gate, W, n_anchor=0):
    B = q_shape[0]
    k, v = probe_kv(B, Lmax, Hkv, d, dtype)
    sl, gate = sl.cuda(), gate.cuda()
    call = (lambda q, **kw: swa.decode_anchored(q, k, v, sl, gate, W, n_anchor, 1.0, **kw)) \
        if n_anchor else (lambda q, **kw: swa.decode(q, k, v, sl, gate, W, 1.0, **kw))
    res = {}
    _, lse = call(torch.zeros(*q_shape, d, dtype=dtype).cuda(), want_lse=True)
    res["count"] = count_of(lse)
    res["min"] = decode_position(call(probe_q(q_shape, d, dtype, -1.0).cuda()))
    res["max"] = decode_position(call(probe_q(q_shape, d, dtype, 1.0).cuda()))
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    return res


def expected_decode(sl, gate, W, Hq):
    """The decode query of sequence b is row L_b - 1 of a prefill with that
    sequence's gate: its range comes from the oracle's row ranges."""
    out = {"count": [], "min": [], "max": []}
    for L, gt in zip(sl.tolist(), gate.tolist()):
        lo, hi = oracle.row_ranges(np.full((1, L), gt, np.uint8), W)
        out["count"].append(hi[0, -1] - lo[0, -1] + 1)
        out["min"].append(lo[0, -1])
        out["max"].append(hi[0, -1])
    return {key: np.repeat(np.array(val)[:, None], Hq, 1) for key, val in out.items()}


@pytest.mark.parametrize("dtype,d,Hq,Hkv", [(torch.bfloat16, 128, 8, 2), (torch.bfloat16, 64, 4, 4),
                                            (torch.float32, 128, 4, 1)])
def test_decode_visited_sets_exact(swa, dtype, d, Hq, Hkv):
    B, Lmax, W = 8, 700, 50
    sl = torch.tensor([1, 49, 50, 51, 64, 257, 513, 700], dtype=torch.int32)
    gate = torch.tensor([1, 0, 1, 0, 0, 1, 0, 1], dtype=torch.uint8)
    got = decode_probes(swa, (B, Hq), Lmax, Hkv, d, dtype, sl, gate, W)
    want = expected_decode(sl, gate, W, Hq)
    for key in ("count", "min", "max"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


def test_decode_16x32k_visited_sets_exact(swa):
    """The decode workload's shape and gates (16 sequences of 32768 cached
    tokens, W = 1024), every sequence and head."""
    d = inp.decode_16x32k(seed=0)
    got = decode_probes(swa, (d["B"], d["Hq"]), d["Lmax"], d["Hkv"], d["d"], torch.bfloat16,
                        d["seq_lens"], d["gate"], d["W"])
    want = expected_decode(d["seq_lens"], d["gate"], d["W"], d["Hq"])
    for key in ("count", "min", "max"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


def test_anchored_decode_visited_sets_exact(swa):
    B, Lmax, Hq, Hkv, d, W, S = 6, 900, 4, 2, 128, 100, 256
    sl = torch.tensor([1, 100, 257, 357, 700, 900], dtype=torch.int32)
    gate = torch.tensor([0, 0, 0, 0, 0, 1], dtype=torch.uint8)
    got = decode_probes(swa, (B, Hq), Lmax, Hkv, d, torch.bfloat16, sl, gate, W, n_anchor=S)
    k, v = probe_kv(B, Lmax, Hkv, d, torch.bfloat16, device="cpu")
    _, lse = oracle.decode_anchored(np.zeros((B, Hq, d)), f64(k), f64(v), sl.numpy(),
                                    gate.numpy(), W, S, 1.0, want_lse=True)
    np.testing.assert_array_equal(got["count"], np.rint(np.exp(lse)).astype(np.int64))
    for name, sign in (("min", -1.0), ("max", 1.0)):
        q = f64(probe_q((B, Hq), d, torch.bfloat16, sign))
        o = oracle.decode_anchored(q, f64(k), f64(v), sl.numpy(), gate.numpy(), W, S, 1.0)
        np.testing.assert_array_equal(got[name], decode_position(torch.from_numpy(o)), err_msg=name)


@pytest.mark.parametrize("B,N,Hq,Hkv,W", [(1, 300, 2, 2, 37), (2, 700, 4, 2, 129),
                                         (2, 8192, 16, 4, 1024)])
def test_dual_branch_visited_sets_exact(swa, B, N, Hq, Hkv, W):
    """Both branches of every row: O_FULL over [0, i], O_SWA over the window.
    The count comes from the gated output's lse with all logits positive
    (full) or negative (window)."""
    k, v = probe_kv(B, N, Hkv, 128, torch.bfloat16)
    nll = torch.ones(B, N, device="cuda")
    pos = torch.ones(B, N, device="cuda")
    got = {}
    for name, sign in (("min", -1.0), ("max", 1.0)):
        q = probe_q((B, N, Hq), 128, torch.bfloat16, sign).cuda()
        out = swa.dual_branch(q, k, v, pos, nll, W, 1.0)
        got["full_" + name] = decode_position(out["o_full"])
        got["swa_" + name] = decode_position(out["o_swa"])
    zq = torch.zeros(B, N, Hq, 128, dtype=torch.bfloat16, device="cuda")
    for name, lg in (("full_count", pos), ("swa_count", -pos)):
        out = swa.dual_branch(zq, k, v, lg, nll, W, 1.0, want_lse=True)
        got[name] = count_of(out["lse_gated"])
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ones = torch.ones(B, N, dtype=torch.uint8)
    for branch, gate in (("full", ones), ("swa", torch.zeros_like(ones))):
        want = expected_plain(gate, W, Hq)
        for key in ("count", "min", "max"):
            np.testing.assert_array_equal(got[f"{branch}_{key}"], want[key],
                                          err_msg=f"{branch} {key}")

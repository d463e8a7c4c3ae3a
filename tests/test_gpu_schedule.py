"""The work lists of the routed prefill and of its backward, read back from the workspace after a call
and checked as index work (bit-exact): every far tile with rows is covered
exactly once (by its pair, or by a one-tile item of the pair), every band
pair with a row to write appears once per head, far items come first and
nothing else is listed.  Several gate patterns, including the shapes where
far pairs are split.

The workspace offsets follow the library's layout of the prefill workspace
(far-row list, count, tile prefixes, far tiles' last rows, the list's length
and counter, then 16-byte items {kind, batch, head, pair}); the far tiling is
re-derived here from the gates: far rows are rows i >= W with gate 1, in
ascending order, and the first 128-row far tile holds the remainder of their
count.
"""
import math

import numpy as np
import pytest
import torch

import swiattn_inputs as inp

BAND, FAR, FAR_A, FAR_B = 0, 1, 2, 3


@pytest.fixture(scope="module")
def swa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_router_gb300 as m
    return m


def up(x):
    return (x + 255) & ~255


def read_list(swa, q, k, v, gate, W):
    B, N = gate.shape
    ws = torch.zeros(swa.prefill_workspace(B, N, q.shape[2], k.shape[2], 128, W, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    swa.prefill(q, k, v, gate, W, 1 / math.sqrt(128), workspace=ws)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    NT = (N + 127) // 128
    off = up(B * N * 4)
    off = up(off + B * 4)
    off = up(off + B * (NT + 1) * 4)
    off = up(off + B * NT * 4)
    n = int(ws[off:off + 4].view(torch.int32).item())
    items_off = up(off + 16)
    items = ws[items_off:items_off + 16 * n].view(torch.int32).view(n, 4).cpu().numpy()
    return items.astype(np.int64)


def expected(gate, W, Hq):
    B, N = gate.shape
    NP = (N + 255) // 256
    far_tiles, band = set(), set()
    for b in range(B):
        g = gate[b]
        far = np.nonzero((g != 0) & (np.arange(N) >= W))[0]
        R = len(far)
        front = (128 - R % 128) % 128
        for t in range((R + front + 127) // 128):
            if min(R, 128 * (t + 1) - front) > max(0, 128 * t - front):
                for h in range(Hq):
                    far_tiles.add((b, h, t))
        isfar = (g != 0) & (np.arange(N) >= W)
        for p in range(NP):
            rows = np.arange(256 * p, min(N, 256 * p + 256))
            if len(rows) and not isfar[rows].all():
                for h in range(Hq):
                    band.add((b, h, p))
    return far_tiles, band


def check(items, gate, W, Hq):
    far_tiles, band = expected(gate, W, Hq)
    kinds = items[:, 0]
    assert set(np.unique(kinds)) <= {BAND, FAR, FAR_A, FAR_B}
    nfar = int((kinds != BAND).sum())
    assert (kinds[:nfar] != BAND).all() and (kinds[nfar:] == BAND).all()   # far items first
    got_far = []
    for kind, b, h, p in items[:nfar]:
        if kind == FAR:
            # a whole pair: its first tile has rows; its second may be empty
            # (the last pair of an odd number of far tiles)
            got_far.append((b, h, 2 * p))
            if (b, h, 2 * p + 1) in far_tiles:
                got_far.append((b, h, 2 * p + 1))
        else:
            got_far.append((b, h, 2 * p + (kind == FAR_B)))
    assert len(got_far) == len(set(got_far)) and set(got_far) == far_tiles
    got_band = [(b, h, p) for _, b, h, p in items[nfar:]]
    assert len(got_band) == len(set(got_band)) and set(got_band) == band
    return nfar, int(((kinds == FAR_A) | (kinds == FAR_B)).sum())


def cases():
    out = []
    for c, (B, N, Hq, W, kind) in enumerate([(1, 4096, 4, 1024, "router"), (2, 3000, 2, 300, "runs"),
                                             (1, 4096, 1, 256, "split"), (3, 1500, 2, 100, "random"),
                                             (1, 2048, 2, 64, "all"), (1, 700, 1, 1000, "runs")]):
        out.append((c, B, N, Hq, W, kind))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("case", cases(), ids=lambda c: f"{c[5]}{c[0]}")
def test_work_list_covers_every_tile_once(swa, case):
    c, B, N, Hq, W, kind = case
    g = inp._gen(2024 + c)
    q, k, v = inp.attention_qkv(B, N, Hq, Hq, 128, torch.bfloat16, g)
    if kind == "router":
        gate = torch.stack([inp.bernoulli_gates((N,), 0.125, g) for _ in range(B)])
    elif kind == "runs":
        gate = torch.stack([inp.run_gates(N, 0.3, g, mean_run=16.0) for _ in range(B)])
    elif kind == "split":
        gate = torch.ones(B, N, dtype=torch.uint8)
        gate[:, ::128] = 0
    elif kind == "all":
        gate = torch.ones(B, N, dtype=torch.uint8)
    else:
        gate = torch.stack([inp.bernoulli_gates((N,), 0.5, g) for _ in range(B)])
    items = read_list(swa, q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W)
    nfar, nsplit = check(items, gate.numpy(), W, Hq)
    if kind == "split":
        assert nsplit > 0


def test_checker_accepts_valid_lists_and_catches_planted_mistakes():
    rng = np.random.default_rng(0)
    for _ in range(200):
        B, Hq = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        N, W = int(rng.integers(1, 1200)), int(rng.integers(1, 400))
        gate = (rng.random((B, N)) < rng.random()).astype(np.uint8)
        far, band = expected(gate, W, Hq)
        items = []
        for b, h, p in sorted({(b, h, t // 2) for b, h, t in far}):
            if rng.random() < 0.5 and (b, h, 2 * p + 1) in far:
                items += [[FAR_A, b, h, p], [FAR_B, b, h, p]]
            else:
                items.append([FAR, b, h, p])
        items += [[BAND, b, h, p] for b, h, p in sorted(band)]
        items = np.array(items, dtype=np.int64).reshape(-1, 4)
        check(items, gate, W, Hq)
        if len(items) > 1:
            with pytest.raises(AssertionError):
                check(np.concatenate([items, items[-1:]]), gate, W, Hq)   # duplicated
            with pytest.raises(AssertionError):
                check(items[:-1], gate, W, Hq)                            # dropped
        nfar = int((items[:, 0] != BAND).sum())
        if 0 < nfar < len(items):
            with pytest.raises(AssertionError):
                check(items[::-1].copy(), gate, W, Hq)                    # band before far


# ---------------------------------------------------------------------------
# The training backward's work lists.  Its workspace holds the far-row list,
# count and tile prefixes, the compacted far rows' indices, four per-row
# statistics arrays, the compacted q and dO, four counters {n_kv, next_kv, n_q,
# next_q}, then 32-byte items {kind, b, h, t, a0, a1, a2, cost}: the dK/dV list
# (one item per batch, KV head and 128-key block) and the dQ list (band and far
# query tiles, each listed once per query head with the heads adjacent), both
# sorted by descending cost (costs above 4095 share the top bucket).

KV, Q_BAND, Q_FAR = 0, 1, 2
NO_ROW = -(1 << 30)


def bwd_offsets(B, N, Hq, Hkv):
    NT = (N + 127) // 128
    Npad = NT * 128
    rows = B * Hq * Npad
    off = up(B * N * 4)
    off = up(off + B * 4)
    off = up(off + B * (NT + 1) * 4)
    rowidx = off
    off = up(off + B * Npad * 4)
    for _ in range(4):
        off = up(off + 4 * rows)
    off = up(off + 2 * rows * 128)
    off = up(off + 2 * rows * 128)
    counters = off
    items_kv = up(off + 16)
    items_q = up(items_kv + 32 * B * Hkv * NT)
    return rowidx, counters, items_kv, items_q


def far_rows(gate_b, W):
    return np.nonzero((gate_b != 0) & (np.arange(len(gate_b)) >= W))[0]


def expected_bwd(gate, W, Hq, Hkv):
    """Items from the pairs each one must cover: key block t (keys
    [128 t, 128 t + 128)) is seen through the window by rows [128 t,
    128 t + 127 + W) and through the far path by far rows i >= 128 t + W;
    a query tile walks the keys its rows see."""
    B, N = gate.shape
    NT = (N + 127) // 128
    kv, q, rowidx = [], [], []
    for b in range(B):
        far = far_rows(gate[b], W)
        R = len(far)
        front = (128 - R % 128) % 128
        rowidx.append(np.concatenate([np.full(front, NO_ROW), far]).astype(np.int64))
        for h in range(Hkv):
            for t in range(NT):
                k0 = 128 * t
                band_hi = min(N, k0 + 127 + W)             # rows [k0, band_hi)
                a0 = -(-(band_hi - k0) // 128)
                pos = np.nonzero(far >= k0 + W)[0] + front
                a1, a2 = (int(pos.min()) // 128, int(pos.max()) // 128 + 1) if len(pos) else (0, 0)
                kv.append((KV, b, h, t, a0, a1, a2, (Hq // Hkv) * (a0 + a2 - a1)))
        isfar = np.zeros(N, bool)
        isfar[far] = True
        for t in range(NT):
            q0, q1 = 128 * t, min(N, 128 * t + 128)
            if not isfar[q0:q1].all():
                lo = max(0, q0 - W + 1)
                cost = (q1 - 1 - lo) // 128 + 1
                q.extend((Q_BAND, b, h, t, lo, cost, 0, cost) for h in range(Hq))
        for t in range((R + front) // 128):
            last = int(far[min(R, 128 * (t + 1) - front) - 1])
            q.extend((Q_FAR, b, h, t, 0, last // 128 + 1, 0, last // 128 + 1) for h in range(Hq))
    return kv, q, rowidx


def check_bwd(kv_items, q_items, rowidx, gate, W, Hq, Hkv):
    kv, q, rows = expected_bwd(gate, W, Hq, Hkv)
    got_kv = [tuple(int(x) for x in r) for r in kv_items]
    got_q = [tuple(int(x) for x in r) for r in q_items]
    assert sorted(got_kv) == sorted(kv)
    assert sorted(got_q) == sorted(q)
    for got in (got_kv, got_q):
        c = [min(r[7], 4095) for r in got]
        assert all(x >= y for x, y in zip(c, c[1:]))          # descending cost
    assert len(got_q) % Hq == 0
    for i in range(0, len(got_q), Hq):                        # heads adjacent
        grp = got_q[i:i + Hq]
        assert [r[2] for r in grp] == list(range(Hq))
        assert len({r[:2] + r[3:] for r in grp}) == 1
    for b, want in enumerate(rows):
        assert np.array_equal(rowidx[b][:len(want)], want)


def bwd_cases():
    return [(0, 1, 1024, 2, 1, 64, "edges"), (1, 2, 3000, 8, 2, 300, "runs"),
            (2, 1, 2048, 4, 4, 128, "random"), (3, 1, 700, 2, 1, 1000, "none"),
            (4, 1, 1536, 2, 2, 64, "all"), (5, 2, 1000, 4, 1, 129, "random")]


@pytest.mark.gpu
@pytest.mark.parametrize("case", bwd_cases(), ids=lambda c: f"{c[6]}{c[0]}")
def test_backward_work_lists_cover_every_block_and_tile(swa, case):
    c, B, N, Hq, Hkv, W, kind = case
    g = inp._gen(5150 + c)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    if kind == "edges":
        gate = torch.zeros(B, N, dtype=torch.uint8)
        gate[0, torch.randperm(N - W, generator=g)[:129] + W] = 1
    elif kind == "runs":
        gate = torch.stack([inp.run_gates(N, 0.3, g, mean_run=16.0) for _ in range(B)])
    elif kind == "all":
        gate = torch.ones(B, N, dtype=torch.uint8)
    else:
        gate = torch.stack([inp.bernoulli_gates((N,), 0.4, g) for _ in range(B)])
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), gate.cuda()
    o, lse = swa.prefill(qd, kd, vd, gd, W, want_lse=True)
    do = inp.output_grad((B, N, Hq, 128), torch.bfloat16, 91 + c).cuda()
    ws = torch.zeros(swa.prefill_backward_workspace(B, N, Hq, Hkv, 128, W, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    swa.prefill_backward(qd, kd, vd, gd, o, lse, do, W, workspace=ws)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    ro, co, ko, qo = bwd_offsets(B, N, Hq, Hkv)
    NT = (N + 127) // 128
    cnt = ws[co:co + 16].view(torch.int32).cpu().numpy()
    kv_items = ws[ko:ko + 32 * int(cnt[0])].view(torch.int32).view(-1, 8).cpu().numpy()
    q_items = ws[qo:qo + 32 * int(cnt[2])].view(torch.int32).view(-1, 8).cpu().numpy()
    rowidx = ws[ro:ro + 4 * B * NT * 128].view(torch.int32).view(B, -1).cpu().numpy()
    check_bwd(kv_items, q_items, rowidx, gate.numpy(), W, Hq, Hkv)


def test_backward_checker_catches_planted_mistakes():
    rng = np.random.default_rng(1)
    for _ in range(60):
        B, Hkv = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        Hq = Hkv * int(rng.integers(1, 3))
        N, W = int(rng.integers(1, 900)), int(rng.integers(1, 300))
        gate = (rng.random((B, N)) < rng.random()).astype(np.uint8)
        kv, q, rows = expected_bwd(gate, W, Hq, Hkv)
        kv = sorted(kv, key=lambda r: -min(r[7], 4095))
        grp = sorted(range(0, len(q), Hq), key=lambda i: -min(q[i][7], 4095))
        q = [q[i + h] for i in grp for h in range(Hq)]
        kv_a, q_a = np.array(kv).reshape(-1, 8), np.array(q).reshape(-1, 8)
        pad = [np.concatenate([r, rng.integers(-5, 5, 8)]) for r in rows]
        check_bwd(kv_a, q_a, pad, gate, W, Hq, Hkv)
        bad = kv_a.copy()
        bad[0, 5] += 1                                           # far tile range off by one
        with pytest.raises(AssertionError):
            check_bwd(bad, q_a, pad, gate, W, Hq, Hkv)
        if len(q_a):
            with pytest.raises(AssertionError):
                check_bwd(kv_a, q_a[:-1], pad, gate, W, Hq, Hkv)   # a head's item dropped
        if len(kv_a) > 1 and min(kv_a[0, 7], 4095) != min(kv_a[-1, 7], 4095):
            with pytest.raises(AssertionError):
                check_bwd(kv_a[::-1].copy(), q_a, pad, gate, W, Hq, Hkv)   # ascending order
        long_rows = [r for r in rows if len(r)]
        if long_rows and any((r != NO_ROW).any() for r in rows):
            b = next(i for i, r in enumerate(rows) if (r != NO_ROW).any())
            moved = [p.copy() for p in pad]
            j = int(np.nonzero(rows[b] != NO_ROW)[0][0])
            moved[b][j] += 1                                     # a far row index changed
            with pytest.raises(AssertionError):
                check_bwd(kv_a, q_a, moved, gate, W, Hq, Hkv)

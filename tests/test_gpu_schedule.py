"""The routed prefill's work list, read back from the workspace after a call
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

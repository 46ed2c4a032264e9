"""The persistent schedule, checked on the CPU (no GPU needed).

The debug library runs the kernel's own unit iterator on the host
(gemm_ws_debug_schedule) for a given device shape. These tests check, for
many problem shapes, device shapes and stream-K settings, that

- every ring stage of every output tile (each 64-column quarter) is computed
  by exactly one unit: nothing is skipped, nothing is done twice;
- the pieces of a stream-K tile are numbered 0..n-1 by consecutive clusters,
  in K order, and all agree on n and on the first cluster;
- every workspace slot stays inside the buffer the handle allocates (one
  partial part per SM), slots are never shared, and unit ids are unique and
  below the reported bound;
- every cluster runs at most one piece, as its last unit, all pieces are
  equal within one stage, and piece s of every tile starts at the same k;
- stream-out and GEMM_WS_STREAM_K=0 plans never use stream-K.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

from async_pipelines_gb300 import build as _build
from async_pipelines_gb300 import gemm_ws

BM, BN, BK = 128, 256, 64

# (cta_group, SMs, clusters that fit): CTA pairs and single CTAs on 152 and
# 148 SMs, and CTA pairs on a GPU shared with other work (36 pairs fit).
DEVICES = [(2, 152, 76), (1, 152, 152), (2, 152, 36), (2, 148, 74)]
DEVICE_IDS = ["pair152", "single152", "pair152_36", "pair148"]

SHAPES = [
    (256, 256, 8192, 1), (8192, 8192, 8192, 1), (4096, 4096, 4096, 1),
    (5000, 3000, 4000, 4), (2048, 2048, 16384, 1), (1024, 1024, 32768, 1),
    (128, 8, 2048, 1), (1000, 776, 20000, 1), (200, 296, 4096, 3), (8192, 8192, 64, 1),
    (256, 256, 256, 1), (640, 1024, 384, 2), (4000, 4104, 96, 2), (1, 8, 8, 1),
    (300, 520, 200, 2), (256, 256, 0, 1), (2048, 2048, 2048, 1), (4096, 2560, 1024, 1),
    (320, 264, 8192, 2), (6144, 6144, 2048, 1),
]


@pytest.fixture(scope="module")
def lib():
    if _build.stale(_build.DEBUG_LIB):
        _build.build()
    return gemm_ws.load_debug_library()


def schedule(lib, dev, stream_k, M, N, K, L, streamout=False):
    cg, sms, maxc = dev
    plan = (ctypes.c_int * 9)()
    n = ctypes.c_int64()
    rc = lib.gemm_ws_debug_schedule(cg, sms, maxc, stream_k, M, N, K, L, int(streamout),
                                    None, 0, ctypes.byref(n), plan)
    assert rc == gemm_ws.OK
    rows = np.zeros((max(n.value, 1), 15), dtype=np.int32)
    rc = lib.gemm_ws_debug_schedule(cg, sms, maxc, stream_k, M, N, K, L, int(streamout),
                                    rows.ctypes.data, n.value, ctypes.byref(n), plan)
    assert rc == gemm_ws.OK
    return list(plan), rows[:n.value]


def check(plan, rows, dev, M, N, K, L):
    cg, sms, maxc = dev
    cs, clusters, id_bound, T, ns, sk_first, sk_clusters, tm, tn = plan
    ksub = 1 if cg == 1 else 2
    assert cs == cg
    assert tm == -(-M // (BM * cs)) and tn == -(-N // BN) and T == L * tm * tn
    assert ns == -(-(-(-K // BK)) // ksub)
    assert 1 <= clusters <= maxc
    cols = ("c", "i", "id", "tile", "mb", "n0", "width", "l", "kb0", "kb1", "piece", "pieces",
            "sk_tile", "first", "slot")
    R = {k: rows[:, j] for j, k in enumerate(cols)}

    # each tile has one (m block, n block, batch), and together they are all of them
    where = {}
    for t, mb, n0, l in zip(R["tile"], R["mb"], R["n0"], R["l"]):
        key = (int(mb), int(n0) // BN, int(l))
        assert where.setdefault(int(t), key) == key
        assert 0 <= key[0] < tm and 0 <= key[1] < tn and 0 <= key[2] < L
    assert sorted(where) == list(range(T)) and len(set(where.values())) == T

    # every stage of every 64-column quarter of every tile exactly once
    cover = np.zeros((T, 4, max(ns, 1)), dtype=np.int32)
    seen_empty = np.zeros((T, 4), dtype=np.int32)
    for t, n0, width, kb0, kb1 in zip(R["tile"], R["n0"], R["width"], R["kb0"], R["kb1"]):
        assert width in (BN, BN // 2, BN // 4)
        assert int(n0) % width == 0
        first = (int(n0) % BN) // (BN // 4)
        quarters = range(first, first + int(width) // (BN // 4))
        assert 0 <= kb0 <= kb1 <= ns
        for h in quarters:
            if ns == 0:
                seen_empty[t, h] += 1
            cover[t, h, kb0:kb1] += 1
    if ns == 0:
        assert np.all(seen_empty == 1)
    else:
        assert np.all(cover == 1)

    # walk order, ids
    for c in range(clusters):
        mine = R["i"][R["c"] == c]
        assert list(mine) == list(range(len(mine)))
    assert len(set(R["id"].tolist())) == len(rows)
    assert R["id"].min() >= 0 and R["id"].max() < id_bound

    # stream-K pieces
    split = R["pieces"] > 1
    assert np.all(R["slot"][~split] == -1)
    if sk_first == T:
        assert not split.any()
        return
    assert sk_first % clusters == 0
    assert np.all(R["tile"][split] >= sk_first)
    assert np.all(R["sk_tile"][split] == R["tile"][split] - sk_first)
    slots = R["slot"][split]
    assert len(set(slots.tolist())) == len(slots)
    assert slots.min() >= 0 and (slots.max() + 1) * cs <= sms               # partial parts
    for t in np.unique(R["tile"][split]):
        sel = R["tile"] == t
        n_p = R["pieces"][sel]
        assert np.all(n_p == n_p[0]) and np.all(R["first"][sel] == R["first"][sel][0])
        order = np.argsort(R["piece"][sel])
        assert list(R["piece"][sel][order]) == list(range(n_p[0]))
        assert list(R["c"][sel][order]) == list(range(R["first"][sel][0],
                                                      R["first"][sel][0] + n_p[0]))
        kb0, kb1 = R["kb0"][sel][order], R["kb1"][sel][order]
        assert kb0[0] == 0 and kb1[-1] == ns and np.all(kb1[:-1] == kb0[1:])
    # one piece per cluster, as its last unit; all tiles of the region split
    # the same number of ways into pieces equal within one stage, with piece
    # s of every tile starting at the same k
    in_sk = R["tile"] >= sk_first
    assert np.all(split == in_sk)
    for c in np.unique(R["c"][in_sk]):
        mine = R["c"] == c
        assert (mine & in_sk).sum() == 1
        assert R["i"][mine & in_sk][0] == R["i"][mine].max()
    assert len(set(R["pieces"][in_sk].tolist())) == 1
    S = int(R["pieces"][in_sk][0])
    assert 2 <= S <= 32 and sk_clusters == (T - sk_first) * S
    length = R["kb1"][in_sk] - R["kb0"][in_sk]
    assert length.max() - length.min() <= 1
    starts = {}
    for piece, kb0 in zip(R["piece"][in_sk], R["kb0"][in_sk]):
        assert starts.setdefault(int(piece), int(kb0)) == kb0


@pytest.mark.parametrize("dev", DEVICES, ids=DEVICE_IDS)
@pytest.mark.parametrize("stream_k", [0, 1, 2], ids=["sk_off", "sk_auto", "sk_always"])
def test_schedule_covers_every_stage_once(lib, dev, stream_k):
    for (M, N, K, L) in SHAPES:
        plan, rows = schedule(lib, dev, stream_k, M, N, K, L)
        check(plan, rows, dev, M, N, K, L)
        if stream_k == 0:
            assert plan[5] == plan[3], (M, N, K, L)


@pytest.mark.parametrize("dev", DEVICES, ids=DEVICE_IDS)
def test_streamout_never_uses_stream_k(lib, dev):
    for (M, N, K, L) in SHAPES:
        plan, rows = schedule(lib, dev, 2, M, N, K, L, streamout=True)
        check(plan, rows, dev, M, N, K, L)
        assert plan[5] == plan[3]


def test_stream_k_where_expected(lib):
    dev = DEVICES[0]
    sk = lambda *s: (lambda p: p[3] - p[5])(schedule(lib, dev, 1, *s)[0])
    assert sk(1024, 1024, 32768, 1) == 16      # few tiles, long K: every tile
    assert sk(256, 256, 8192, 1) == 1
    assert sk(2048, 2048, 16384, 1) == 0       # one partial wave, over half full: whole tiles
    assert sk(4096, 4096, 4096, 1) == 0        # 256 = 3 * 76 + 28: half-width tail is cheaper
    # 1024 = 13 * 76 + 36 and 36 tiles: the last partial wave split in two
    # pieces per tile (measured ~0.6 us faster than half-width tiles in both)
    assert sk(8192, 8192, 8192, 1) == 36
    assert sk(1536, 1536, 8192, 1) == 36
    assert sk(8192, 8192, 4096, 1) == 0        # 32-stage tiles: half-width tail is cheaper
    assert sk(1024, 1024, 1024, 1) == 0        # short K: pieces would be too small
    assert sk(256, 256, 0, 1) == 0
    # 152 tiles = exactly two waves of 76 clusters: nothing to balance
    plan, _ = schedule(lib, dev, 2, 76 * 256 * 2, 256, 4096, 1)
    assert plan[3] == 152 and plan[5] == 152


@pytest.mark.parametrize("M,N,K,L,cs", [
    (8192, 8192, 64, 1, 1), (256, 256, 256, 1, 1), (8192, 8192, 512, 1, 1),
    (2048, 2048, 1024, 1, 1), (3072, 3072, 1024, 1, 1),   # <= 2 waves (144 pair tiles)
    (3328, 3328, 1024, 1, 2), (8192, 8192, 1024, 1, 2),   # more (169): CTA pairs
    (512, 512, 2048, 1, 2), (4096, 4096, 4096, 1, 2), (8192, 8192, 8192, 1, 2),
])
def test_tile_configuration_rule(lib, M, N, K, L, cs):
    """Default handles: single-CTA tiles for K <= 512, or K <= 1024 with at
    most two waves (2 x 76) of 256 x 256 pair tiles; CTA pairs otherwise. The
    chosen plan still covers every stage exactly once."""
    dev = (0, 152, 76)
    plan, rows = schedule(lib, dev, 1, M, N, K, L)
    assert plan[0] == cs
    check(plan, rows, (cs, 152, 76 if cs == 2 else 152), M, N, K, L)


@pytest.mark.parametrize("stream_k", [1, 2], ids=["sk_auto", "sk_always"])
def test_schedule_random_shapes(lib, stream_k):
    """Seeded random shapes (ragged M, N multiples of 8, K multiples of 8 up
    to 40k, L up to 4) on every device shape, including the default tile
    rule: every plan still covers every stage exactly once and keeps its
    pieces and workspace indices in bounds."""
    rng = np.random.default_rng(20261202 + stream_k)
    devices = DEVICES + [(0, 152, 76)]
    for _ in range(60):
        M = int(rng.integers(1, 12000))
        N = 8 * int(rng.integers(1, 1500))
        K = 8 * int(rng.integers(0, 5000))
        L = int(rng.integers(1, 5))
        for dev in devices:
            plan, rows = schedule(lib, dev, stream_k, M, N, K, L)
            cs = plan[0]
            # the default rule picks per problem; check against the config it chose
            eff = dev if dev[0] else (cs, 152, 76 if cs == 2 else 152)
            check(plan, rows, eff, M, N, K, L)


def _model_best_halves(T, P, half_cost=0.8):
    """The tail rule stated for the schedule, by exhaustive search: split the
    last s tiles (s <= min(P, T)) into two half units each, so as to minimise
    the slowest cluster's work (whole unit 1, half unit half_cost); ties keep
    fewer halves."""
    best = None
    for s in range(0, min(P, T) + 1):
        F, U = T - s, T + s
        n_full, n_units = -(-F // P), -(-U // P)
        worst = n_full + half_cost * (n_units - n_full)
        if best is None or worst < best[0] - 1e-9:
            best = (worst, s)
    return best[1]


@pytest.mark.parametrize("dev", DEVICES[:2] + DEVICES[3:], ids=["pair152", "single152", "pair148"])
def test_half_units_are_the_last_tiles(lib, dev):
    """Half-width units come only from the last tiles in raster order, their
    number matches the stated cost model, and a tile count that is a
    multiple of the clusters gets none; problems with at most a quarter as
    many tiles as clusters run every tile as four quarter units instead."""
    for (M, N, K, L) in SHAPES + [(8192, 8192, 8192, 1), (76 * 512, 256, 4096, 1)]:
        plan, rows = schedule(lib, dev, 0, M, N, K, L)
        T, P = plan[3], dev[2]
        if 4 * T <= P:
            # so few tiles that four units per tile fit at once: every tile
            # runs as four 64-column quarters, one per cluster
            assert np.all(rows[:, 6] == BN // 4) and len(rows) == 4 * T, (M, N, K, L)
            assert plan[1] == 4 * T
            continue
        assert not np.any(rows[:, 6] == BN // 4)
        halves = sorted({int(t) for t, wd in zip(rows[:, 3], rows[:, 6]) if wd == BN // 2})
        assert halves == list(range(T - len(halves), T)), (M, N, K, L)
        assert len(halves) == _model_best_halves(T, P), (M, N, K, L)
        if T % P == 0:
            assert not halves
        if dev == DEVICES[0] and (M, N, K) == (8192, 8192, 8192):
            assert (T, len(halves)) == (1024, 36)   # 988 whole tiles + 72 half units

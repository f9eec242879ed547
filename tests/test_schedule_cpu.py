"""The persistent tile schedule (data-parallel units, split-K, Stream-K) as
tcg_gemm would run it, checked on the host without a GPU.

"CUTLASS" (stanleyjacob.dev), Part IV Stage 2 (a persistent grid walks the
output tiles) and Stage 6 (split-K / Stream-K partition the K loop and
reduce the partial tiles).  Invariants checked for every plan:
  * every (tile, k-block) iteration of the problem is computed exactly once;
  * the pieces of a tile are numbered 0..nsplit-1, cover its K range in that
    order, and agree on nsplit;
  * unsplit tiles write no partial; the partial slots of split pieces are
    distinct, so no two pieces overwrite each other;
  * the work is balanced: with Stream-K no worker has more than one
    k-block iteration above the average.
"""
from collections import defaultdict

import pytest

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import _build


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return tcg.lib()


SHAPES = [(8192, 8192, 8192), (4096, 4096, 4096), (4095, 3001, 1537), (16, 8192, 8192),
          (8192, 128, 8192), (512, 512, 512), (300, 200, 129), (1, 1, 1), (2048, 2560, 256),
          (1000, 9000, 3000)]


def check(M, N, K, ab, sms, mode):
    rows = tcg.debug_schedule(M, N, K, ab, num_sms=sms, sk_mode=mode)
    assert rows, "empty schedule"
    plan_tiles = {}
    pieces = defaultdict(list)
    for wid, tile, m, n, kb0, kb1, split, nsplit, slot, half in rows:
        assert 0 <= kb0 < kb1, (tile, kb0, kb1)
        key = (m, n)
        assert plan_tiles.setdefault(tile, key) == key, "a tile index maps to two output tiles"
        pieces[(tile, half)].append((split, kb0, kb1, nsplit, slot, wid))
    # a tile runs whole, or as its two column halves (the last wave's tail), never both
    halves = defaultdict(set)
    for tile, half in pieces:
        halves[tile].add(half)
    assert all(h == {0} or h == {1, 2} for h in halves.values()), halves
    half_tiles = sorted(t for t, h in halves.items() if h == {1, 2})
    assert half_tiles == list(range(len(halves) - len(half_tiles), len(halves))), "halves are the last tiles"
    # the tile index -> (m, n) map is one to one and covers the whole output grid
    assert len(set(plan_tiles.values())) == len(plan_tiles)
    num_m = max(m for m, _ in plan_tiles.values()) + 1
    num_n = max(n for _, n in plan_tiles.values()) + 1
    assert set(plan_tiles.values()) == {(m, n) for m in range(num_m) for n in range(num_n)}
    assert sorted(plan_tiles) == list(range(num_m * num_n))
    # and that grid spans the problem (no tile is taller or wider than 256)
    assert num_m * 256 >= M and num_n * 256 >= N, (num_m, num_n)
    slots = []
    num_kb = None
    per_worker = defaultdict(int)
    for (tile, half), ps in pieces.items():
        ps.sort()
        nsplit = ps[0][3]
        assert all(p[3] == nsplit for p in ps)
        assert [p[0] for p in ps] == list(range(nsplit)), (tile, ps)
        assert ps[0][1] == 0
        for a, b in zip(ps, ps[1:]):
            assert a[2] == b[1], "pieces of a tile must be contiguous in K"
        if num_kb is None:
            num_kb = ps[-1][2]
        assert ps[-1][2] == num_kb, "every tile covers the same K range"
        if nsplit == 1:
            assert ps[0][4] == -1
        else:
            slots += [p[4] for p in ps]
        for p in ps:
            per_worker[p[5]] += p[2] - p[1]
    assert len(slots) == len(set(slots)), "two pieces share a partial slot"
    assert all(s >= 0 for s in slots)
    total = sum(per_worker.values())
    return rows, per_worker, total


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_schedule_covers_every_iteration_once(shape, mode):
    M, N, K = shape
    for sms in (152, 148, 7):
        check(M, N, K, "bf16", sms, mode)


@pytest.mark.parametrize("shape", [(4095, 3001, 1537), (4096, 4096, 4096), (8192, 128, 8192), (16, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_all_tile_stream_k_is_balanced(shape):
    M, N, K = shape
    rows, per_worker, total = check(M, N, K, "bf16", 152, 3)
    workers = len(per_worker)
    assert max(per_worker.values()) <= -(-total // workers), (max(per_worker.values()), total / workers)
    assert min(per_worker.values()) >= total // workers


def test_partial_wave_is_evened_out():
    """4096^3 with 256 x 256 pair tiles: 256 tiles on 76 pairs leave a last
    wave of 28.  Both remedies even it out: the default schedule runs those
    28 tiles as 56 half-width units (three full waves, then one of half
    tiles on 56 of the 76 pairs), and the partial-wave Stream-K schedule
    (mode 2) spreads the k-blocks of the last tiles over every pair."""
    rows0, w0, t0 = check(4096, 4096, 4096, "bf16", 152, 0)
    assert max(r[3] for r in rows0) + 1 == 16 and len(rows0) == 228 + 56
    assert sum(1 for r in rows0 if r[9]) == 56 and all(r[1] >= 228 for r in rows0 if r[9])
    assert max(w0.values()) == 4 * 32 and min(w0.values()) == 3 * 32   # the busiest pairs end with a half tile
    rows2, w2, t2 = check(4096, 4096, 4096, "bf16", 152, 2)
    assert max(r[3] for r in rows2) + 1 == 16 and t2 == 256 * 32
    assert max(w2.values()) < 4 * 32
    assert max(w2.values()) - min(w2.values()) <= 1 + max(r[5] - r[4] for r in rows2)


def test_wave_fitting_width_choices():
    """The last-wave remedies the planner's wave model picks for the workloads
    (on 152 SMs = 76 pairs): a half-width tail where the last wave of
    256-wide tiles would use at most half of the pairs, a narrower tile
    (K-major B only) where it would not."""
    def plan(M, N, K, ab="bf16"):
        rows = tcg.debug_schedule(M, N, K, ab, num_sms=152, sk_mode=0)
        ntiles = max(r[3] for r in rows) + 1
        fits = [bn for bn in (256, 224, 192, 160) if -(-N // bn) == ntiles]
        assert len(fits) == 1, fits
        return fits[0], len({r[1] for r in rows if r[9]})
    assert plan(8192, 8192, 8192) == (256, 36)     # 13 full waves, then 36 tiles as 72 half units
    assert plan(8192, 8192, 8192, "e4m3") == (256, 36)
    assert plan(4096, 4096, 4096) == (256, 28)     # 3 full waves + 56 half units
    assert plan(4095, 3001, 1537) == (224, 0)      # 40 leftover tiles: 80 halves would not fit one wave


def test_fp8_schedule():
    check(8192, 8192, 8192, "e4m3", 152, 1)
    check(4095, 3001, 1537, "e4m3", 152, 3)


@pytest.mark.parametrize("ab, width", [("mxe4m3", 256), ("mxfp4", 256), ("nvfp4", 256)])
def test_block_scaled_pair_tile_grid(ab, width):
    # block-scaled pairs: 256 x 256 tiles by default (256 x 192 on request)
    M = N = K = 8192
    rows, per_worker, total = check(M, N, K, ab, 152, 0)
    assert max(r[2] for r in rows) + 1 == M // 256
    assert max(r[3] for r in rows) + 1 == -(-N // width)
    assert tcg.debug_schedule(M, N, K, ab, num_sms=152, sk_mode=0)[0][7] == 1   # K is not split


@pytest.mark.parametrize("shape", [(49152, 49152, 64), (200, 300, 1 << 20), ((1 << 20) - 3, 72, 40)],
                         ids=["36864_pair_tiles", "k_2pow20", "m_2pow20"])
@pytest.mark.parametrize("mode", [0, 3])
def test_schedule_at_extreme_sizes(shape, mode):
    """The extreme sizes the GPU tests run (36,864 pair tiles; K = 2^20 with
    split K; about a million rows): every iteration once, slots distinct."""
    M, N, K = shape
    rows, per_worker, total = check(M, N, K, "bf16", 152, mode)
    num_kb = max(r[5] for r in rows)
    units = len({(r[1], r[9]) for r in rows})   # whole tiles, or the two halves of a tail tile
    assert total == units * num_kb

"""The persistent GEMM schedule (csrc/schedule.h), checked on the CPU.

The header is compiled as plain C++ by g++ (tests/sched_dump.cpp prints the
plan and every unit of every cluster), and the properties the kernel relies
on are checked here for a grid of tile counts, K block counts and resident
cluster counts:

* every K block of every tile is computed exactly once;
* the tail takes only the last, partial round of tiles, on at most the
  resident clusters: either each tile in equal parts inside it (a multiple
  of the tile count) or stream-K ranges of two K blocks or more on average;
  a few deep tiles (weight-gradient shapes, K blocks in the thousands) are
  spread over more than 8 clusters each;
* a cluster leaves sums in at most one slot (its own), that unit is the first
  of its tail range, and it waits on nothing before it;
* the owner of a split tile is the last unit of its range, and the parts it
  adds are exactly the published units of clusters c+1 .. c+others, which
  continue its K range in order and end at the tile's last K block;
* every published part is added by exactly one owner;
* the longest cluster does no more K blocks than with whole tiles only, and
  at least one fewer whenever a tail is planned.
"""
import os
import subprocess
from collections import defaultdict

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "fp32_emulated_gemm_split_gb300", "csrc")

TILES = [1, 2, 3, 5, 16, 28, 36, 47, 48, 75, 76, 77, 96, 100, 151, 152, 153, 192, 256, 1024,
         4320]
KBS = [1, 2, 3, 4, 5, 8, 16, 17, 63, 64, 128, 256]
RESIDENT = [1, 2, 37, 64, 74, 76]
FIX2 = [0, 3, 8, 15]          # hand-over cost in half K blocks
# few tiles with many K blocks: 256 x 256 weight gradients over 65K-1.1M rows
DEEP_TILES = [1, 2, 3, 5, 9, 77]
DEEP_KBS = [1024, 4096, 17280]


@pytest.fixture(scope="module")
def dump(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("sched") / "sched_dump")
    subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(HERE, "sched_dump.cpp"), "-o", exe],
                   check=True, capture_output=True, text=True)
    cases = [(t, k, r, f) for t in TILES for k in KBS for r in RESIDENT for f in FIX2]
    cases += [(t, k, r, f) for t in DEEP_TILES for k in DEEP_KBS for r in (2, 74, 76)
              for f in FIX2]
    out = subprocess.run([exe], input="".join(f"{t} {k} {r} {f}\n" for t, k, r, f in cases),
                         check=True, capture_output=True, text=True, timeout=300).stdout
    plans = {}
    cur = None
    for line in out.splitlines():
        f = line.split()
        if f[0] == "case":
            t, k, r, fx, tt, tc, g = map(int, f[1:])
            cur = {"tail_tiles": tt, "tail_clusters": tc, "grid": g, "units": defaultdict(list)}
            plans[(t, k, r, fx)] = cur
        else:
            c, i, tile, kb0, kb1, pub, oth = map(int, f[1:])
            cur["units"][c].append((i, tile, kb0, kb1, pub, oth))
    assert len(plans) == len(cases)
    return plans


def test_plan_takes_only_the_last_round(dump):
    for (tiles, kb, res, fx), p in dump.items():
        tt, tc, g = p["tail_tiles"], p["tail_clusters"], p["grid"]
        assert 1 <= g <= res
        if tt == 0:
            assert tc == 0 and g == min(tiles, res)
            continue
        assert tt == tiles % res
        assert 2 <= tc <= res
        assert tc % tt == 0 or tc <= tt * kb // 2
        assert g == (res if tiles > tt else tc)


def test_aligned_parts_stay_inside_a_tile(dump):
    """With Ct a multiple of the tail's tile count every cluster has exactly
    one unit in the tail: each part lies inside one tile."""
    for (tiles, kb, res, fx), p in dump.items():
        tt, tc = p["tail_tiles"], p["tail_clusters"]
        if tt == 0 or tc % tt:
            continue
        first = tiles - tt
        for c, us in p["units"].items():
            tail = [u for u in us if u[1] >= first]
            assert len(tail) == (1 if c < tc else 0), (tiles, kb, res, fx, c)


def test_every_k_block_once(dump):
    for (tiles, kb, res, fx), p in dump.items():
        seen = defaultdict(int)
        for c, us in p["units"].items():
            assert 0 <= c < p["grid"]
            assert [u[0] for u in us] == list(range(len(us)))
            for _, tile, kb0, kb1, _, _ in us:
                assert 0 <= tile < tiles and 0 <= kb0 < kb1 <= kb
                for k in range(kb0, kb1):
                    seen[(tile, k)] += 1
        assert len(seen) == tiles * kb and set(seen.values()) == {1}, (tiles, kb, res)


def test_parts_and_owners(dump):
    for key, p in dump.items():
        units = p["units"]
        published = {}                      # cluster -> (tile, kb0, kb1)
        for c, us in units.items():
            pubs = [u for u in us if u[4] >= 0]
            assert len(pubs) <= 1, key
            for i, tile, kb0, kb1, pub, oth in us:
                if pub >= 0:
                    assert pub == c and kb0 > 0 and oth == 0
                    # nothing before it waits: earlier units are whole tiles
                    assert all(u[5] == 0 and u[4] < 0 for u in us[:i])
                    published[c] = (tile, kb0, kb1)
                elif oth == 0:
                    assert kb0 == 0 and kb1 == key[1]          # a whole tile
        consumed = set()
        for c, us in units.items():
            for i, tile, kb0, kb1, pub, oth in us:
                if pub >= 0 or oth == 0:
                    continue
                assert kb0 == 0 and i == len(us) - 1, key       # owner waits last
                end = kb1
                for o in range(1, oth + 1):
                    ptile, pk0, pk1 = published[c + o]
                    assert ptile == tile and pk0 == end
                    end = pk1
                    assert (c + o) not in consumed
                    consumed.add(c + o)
                assert end == key[1], key
        assert consumed == set(published), key


def test_tail_shortens_the_longest_cluster(dump):
    for (tiles, kb, res, fx), p in dump.items():
        work = [sum(u[3] - u[2] for u in us) for us in p["units"].values()]
        whole = -(-tiles // res) * kb
        assert max(work) <= whole
        if p["tail_tiles"]:
            # the planner's cost counts at least twice the longest range
            assert max(work) <= whole - 1 - fx // 2, (tiles, kb, res, fx)


def test_known_plans(dump):
    """Plans worked by hand for BF16x9 (a hand-over costs 3 half blocks) on
    76 clusters: 8192^3 (1024 tiles of 128 K blocks, 36 left over: in two
    aligned parts 2*64 + 3 = 131, stream-K over all 76 2*61 + 6 = 128: the
    stream-K tail); 4096^3 (256 tiles of 64, 28 left over: 67 against 2*24 +
    6 = 54: stream-K); 12288 x 256 x 1024 (48 tiles of 16: no aligned split
    fits, stream-K 2*11 + 6 = 28 <= 30: split); 131072 x 256 x 1024 (512 of
    16, 56 left over: 2*12 + 6 = 30: split, the break-even); the fused 128-wide
    12288 x 256 x 1024 (96 tiles of 16, 20 left over: 3 aligned parts 2*6 + 3
    = 15 against 2*5 + 6 = 16: aligned, 60 clusters); and 1105920 x 256 x 256
    (4320 tiles of 4: 64 left over, 2*4 + 6 > 6: no tail)."""
    def plan(t, k):
        p = dump[(t, k, 76, 3)]
        return p["tail_tiles"], p["tail_clusters"]
    assert plan(1024, 128) == (36, 76)
    assert plan(256, 64) == (28, 76)
    assert plan(48, 16) == (48, 76)
    assert plan(4320, 4) == (0, 0)
    assert dump[(96, 16, 76, 3)]["tail_clusters"] == 60
    assert dump[(96, 16, 76, 3)]["grid"] == 76


def test_deep_tiles_spread_over_every_cluster(dump):
    """A 256 x 256 weight gradient over 1.1M rows is one tile of 17280 K
    blocks: it takes every resident cluster (cost 2*228 + 3 + 68 = 527 half
    blocks against 2*2160 + 3 = 4323 for 8 parts), 227-228 blocks each; a
    tile of 128 blocks takes 16 (2*8 + 3 + 8 = 27 against 35 for 8)."""
    p = dump[(1, 17280, 76, 3)]
    assert (p["tail_tiles"], p["tail_clusters"], p["grid"]) == (1, 76, 76)
    work = [sum(u[3] - u[2] for u in us) for us in p["units"].values()]
    assert max(work) - min(work) <= 1 and max(work) == 228
    assert dump[(1, 128, 76, 3)]["tail_clusters"] == 16
    for t in DEEP_TILES[:-1]:
        assert dump[(t, 17280, 76, 3)]["tail_clusters"] >= 75

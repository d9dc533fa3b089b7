"""The decode schedule, simulated on the host (no GPU).

The paged-decode kernels split the work by a plan the device writes: per
batch row the slots of its units (a few empty slots standing for a piece
start, then the unit's 128-key tiles), laid end to end; CTAs walk equal
ranges of that sequence, and a unit cut by range boundaries leaves one
split-KV partial per piece, which the combine kernel finds again from the
same plan.  With grouped-query heads and a grid of whole head groups the KV
head rides on the CTA index instead of being part of the unit.

This file restates that arithmetic in Python (the plan kernel's prefix, the
walk of each CTA, the combine kernel's piece count) and checks, for ragged
batches, windows, several CTA counts and both unit layouts, that every tile
of every (batch row, KV head, row group) unit is walked exactly once, that
each unit's pieces carry the indices 0 .. npieces - 1 once each, that the
combine kernel counts the same pieces, and that npieces stays within the
planner's max_pieces.  The planner fields come from the library's host
planner; nothing here runs on a GPU.
"""
import random

import pytest

KV_TILE = 128


@pytest.fixture(scope="module")
def fw():
    from ragged_softmax_attention_gb300 import build
    import ragged_softmax_attention_gb300 as fw
    fw.load_library(build.build())
    return fw


def window_first_key(n, q_len, window):
    return 0 if window < 0 else max(0, n - q_len - window)


def row_tiles(n, q_len, window):
    return -(-n // KV_TILE) - window_first_key(n, q_len, window) // KV_TILE


def simulate(lens, q_len, hq, hkv, window, piece_cost, grid, plan):
    """Walks of every CTA and the combine's piece counts for one launch."""
    G = hq // hkv
    row_groups = plan["row_groups"]
    ride = hkv > 1 and grid % hkv == 0
    units_per_row = row_groups if ride else hkv * row_groups
    range_groups = hkv if ride else 1
    # Plan kernel: slot prefix per batch row, total, span.
    PB = [0]
    for n in lens:
        rt = row_tiles(n, q_len, window)
        PB.append(PB[-1] + ((piece_cost + rt) * units_per_row if rt > 0 else 0))
    T = PB[-1]
    span = max(plan["min_span_tiles"], -(-T // max(1, grid // range_groups)))
    # Walk of each CTA.
    walked = {}                                      # (b, g, rg) -> list of (tiles, k, npieces)
    for cta in range(grid):
        if ride:
            rng, step, g_ride = cta // hkv, grid // hkv, cta % hkv
        else:
            rng, step, g_ride = cta, grid, None
        while rng * span < T:
            pos, end = rng * span, min(T, (rng + 1) * span)
            while pos < end:
                b = max(i for i in range(len(lens)) if PB[i] <= pos)
                vb = (PB[b + 1] - PB[b]) // units_per_row
                off = pos - PB[b]
                u, vl = divmod(off, vb)
                if vl < piece_cost:
                    pos += piece_cost - vl
                    continue
                tb, tl = vb - piece_cost, vl - piece_cost
                th = min(tb, tl + (end - pos))
                pstart = PB[b] + u * vb + piece_cost
                g, rg = (g_ride, u) if ride else divmod(u, row_groups)
                k = (pstart + tl) // span - pstart // span
                npieces = (pstart + tb - 1) // span - pstart // span + 1
                walked.setdefault((b, g, rg), []).append((list(range(tl, th)), k, npieces))
                pos += th - tl
            rng += step
    # Combine kernel: piece count of every query row's unit.
    head_mode = 1 if G > 32 else 0
    combine = {}
    for b in range(len(lens)):
        vb = (PB[b + 1] - PB[b]) // units_per_row
        if vb == 0:
            continue
        tb = vb - piece_cost
        for t in range(q_len):
            for h in range(hq):
                g = h // G
                if head_mode == 0:
                    rg = t // plan["tokens_per_unit"]
                else:
                    chunks = -(-G // plan["heads_per_unit"])
                    rg = t * chunks + (h - g * G) // plan["rows_per_unit"]
                unit = rg if ride else g * row_groups + rg
                pstart = PB[b] + unit * vb + piece_cost
                combine[(b, g, rg)] = (pstart + tb - 1) // span - pstart // span + 1
    return walked, combine


def check(lens, q_len, hq, hkv, window, piece_cost, grid, fw):
    plan = fw.plan_decode(len(lens), q_len, hq, hkv, 128, max(lens + [1]), num_sms=grid)
    walked, combine = simulate(lens, q_len, hq, hkv, window, piece_cost, grid, plan)
    units = {(b, g, rg) for b, n in enumerate(lens) if row_tiles(n, q_len, window) > 0
             for g in range(hkv) for rg in range(plan["row_groups"])}
    assert set(walked) == units
    for key, pieces in walked.items():
        tiles = sorted(t for ts, _, _ in pieces for t in ts)
        assert tiles == list(range(row_tiles(lens[key[0]], q_len, window))), key
        npieces = {n for _, _, n in pieces}
        assert len(npieces) == 1, key
        (npieces,) = npieces
        assert sorted(k for _, k, _ in pieces) == list(range(npieces)), key
        assert npieces <= plan["max_pieces"], key
        assert combine[key] == npieces, key


@pytest.mark.parametrize("grid", [152, 8, 3, 1])
@pytest.mark.parametrize("hq,hkv,q_len", [(40, 8, 1), (32, 8, 3), (8, 2, 4), (16, 1, 2), (64, 1, 1)])
@pytest.mark.parametrize("piece_cost", [0, 4, 5])
def test_every_tile_walked_once(fw, grid, hq, hkv, q_len, piece_cost):
    rnd = random.Random(grid * 1000 + hq * 10 + piece_cost)
    lens = [rnd.choice([0, 1, 127, 128, 129, 700, 3000, rnd.randint(1, 9000)]) for _ in range(11)]
    check(lens, q_len, hq, hkv, -1, piece_cost, grid, fw)


@pytest.mark.parametrize("window", [0, 100, 4096])
@pytest.mark.parametrize("grid", [152, 16, 5])
def test_windows_walk_only_their_tiles(fw, window, grid):
    rnd = random.Random(window + grid)
    lens = [rnd.randint(0, 20000) for _ in range(9)] + [0, 4097, 128]
    check(lens, 2, 40, 8, window, 4, grid, fw)


def test_partial_head_groups_keep_the_heads_in_the_units(fw):
    """A grid that is not a multiple of Hkv keeps the heads in the unit
    sequence; the walk still covers every tile once."""
    lens = [5000, 0, 333, 12000, 1]
    for grid in (150, 151, 7, 9):
        check(lens, 1, 40, 8, -1, 5, grid, fw)

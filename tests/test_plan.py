"""The work split: the arithmetic of the chunked plan on the host (CPU), and the device
plan kernel against it task for task (GPU).

The plan's job ("[FlyDSL] pa_decode: MXFP4 K/V ...", commit messages: planned tasks,
tasks from a CU budget, direct output with one partition): every tile of every
(sequence, KV head) unit runs exactly once, in order, each CTA gets an equal share of
tiles, no unit has more than max_partitions partitions, and the task and partial-slot
counts stay within the workspace the host sized.
"""
import numpy as np
import pytest
import torch

from tests import plan_model as pm

MIXES = [
    ("long16", [int(x) for x in np.random.default_rng(5).integers(120000, 131073, 16)], 1),
    ("ragged", [0, 1, 255, 256, 257, 4000, 0, 70000, 3, 131072], 2),
    ("uniform4096", [2048] * 4096, 1),
    ("even128", [2048] * 128, 1),  # short, even sequences: laid out whole at budget 152
    ("one", [500000], 1),
    ("empty", [0, 0, 0], 4),
    ("mixed", [int(x) for x in np.random.default_rng(9).integers(1, 9000, 37)], 2),
]
BUDGETS = [1, 7, 152, 304]
MAXP = [1, 2, 3, 128]
# (query length, sliding window): none, and windows that start inside the first tiles,
# at a tile edge, and far into long contexts
WINDOWS = [(1, 0), (4, 3000), (1, 256), (2, 70000)]


@pytest.mark.parametrize("name,lens,hkv", MIXES, ids=[m[0] for m in MIXES])
@pytest.mark.parametrize("budget", BUDGETS)
@pytest.mark.parametrize("maxp", MAXP)
@pytest.mark.parametrize("qlen,window", WINDOWS, ids=[f"q{q}w{w}" for q, w in WINDOWS])
def test_plan_arithmetic(name, lens, hkv, budget, maxp, qlen, window):
    cap = 1 << 20
    m = pm.plan(lens, hkv, budget, maxp, cap, qlen=qlen, window=window)
    tiles = m["tiles"]
    # a unit starts at the tile of the first token that any query position's window holds
    for s, L in enumerate(lens):
        lo = max(0, L - qlen - window + 1) if window > 0 else 0
        assert m["firsts"][s] == lo // pm.TILE
        assert m["firsts"][s] + tiles[s] == (L + pm.TILE - 1) // pm.TILE
    # every tile of every unit exactly once, partitions in order and contiguous
    by_unit = {}
    for (s, hp, b, e) in m["tasks"]:
        by_unit.setdefault((s, hp & 0xFFFF), []).append((hp >> 16, b, e))
    assert len(by_unit) == len(lens) * hkv
    for (s, h), parts in by_unit.items():
        assert [q for q, _, _ in parts] == list(range(len(parts)))
        f = m["firsts"][s]
        assert parts[0][1] == f and parts[-1][2] == f + tiles[s]
        for (_, _, e0), (_, b1, _) in zip(parts, parts[1:]):
            assert e0 == b1
        assert all(e > b for _, b, e in parts) or tiles[s] == 0
        assert len(parts) <= max(1, maxp)
        assert m["nparts"][s * hkv + h] == len(parts)
    # sizes the host reserved
    assert len(m["tasks"]) <= pm.capacity(len(lens), hkv, budget)
    assert maxp < 2 or m["slots"] <= 2 * budget
    # chunks: non-decreasing over the task list, each CTA's range is its chunk
    assert all(a <= b for a, b in zip(m["chunks"], m["chunks"][1:]))
    first = m["chunk_first"]
    assert first[-1] == len(m["tasks"]) and all(a <= b for a, b in zip(first, first[1:]))
    for c in range(budget):
        assert all(m["chunks"][t] == c for t in range(first[c], first[c + 1]))
    # whole units where splitting was allowed but dropped: one task per unit, and no chunk
    # carries more than two unit gaps beyond C positions of tiles and gaps
    if maxp >= 2 and not m["split"]:
        assert all(p == 1 for p in m["nparts"]) and m["slots"] == 0
        assert m["nchunks"] <= budget
        carried = np.zeros(m["nchunks"], dtype=np.int64)
        for (s, hp, b, e), c in zip(m["tasks"], m["chunks"]):
            carried[c] += e - b + pm.UNIT_COST
        assert carried.max(initial=0) <= m["C"] + 2 * pm.UNIT_COST
    # balance: with splitting on, every task's tiles lie inside its chunk's range of the
    # line (each unit is a gap of UNIT_COST followed by its tiles), so no chunk runs more
    # than C tiles, and every chunk but the last covers exactly C positions
    if m["split"]:
        C = m["C"]
        unit_of = {}
        for u, pos in enumerate(m["unit_pos"]):
            unit_of[(u // hkv, u % hkv)] = pos
        for (s, hp, b, e), c in zip(m["tasks"], m["chunks"]):
            if e > b:
                pos = unit_of[(s, hp & 0xFFFF)] - m["firsts"][s]
                assert c * C <= pos + b and pos + e <= (c + 1) * C
        per = pm.chunk_tiles(m)
        assert per.max(initial=0) <= C
        assert m["nchunks"] <= budget
        load = pm.chunk_load(m)
        assert np.all(load[: m["nchunks"] - 1] == C)
        assert m["length"] == (sum(tiles) + pm.UNIT_COST * len(tiles)) * hkv
        if sum(tiles) > 0:
            assert C == max(pm.ceil_div(m["length"], budget), (max(tiles) - 1) // (maxp - 1) + 1)


def test_plan_balance_long_context():
    # 16 long sequences over 152 CTAs: counting each task start at UNIT_COST tiles, the
    # busiest CTA runs at most one tile more than the mean (the proportional split this
    # replaces left ~10% of the GPU idle), and a CTA that finishes one sequence and starts
    # the next runs UNIT_COST tiles fewer than one inside a sequence
    lens = MIXES[0][1]
    m = pm.plan(lens, 1, 152, 128, 1 << 20)
    per = pm.chunk_tiles(m)
    starts = np.zeros_like(per)
    for (s, hp, b, e), c in zip(m["tasks"], m["chunks"]):
        starts[c] += 1
    work = per + pm.UNIT_COST * (starts - 1)
    assert work.max() - work.sum() / 152 <= 1.0
    two = per[starts == 2]
    assert len(two) > 0 and two.max() <= m["C"] - pm.UNIT_COST


def test_plan_keeps_short_even_units_whole():
    # 128 sequences of 8 tiles over 152 chunks: split at chunk edges, every sequence would
    # become two partial tasks; whole, each chunk runs at most one sequence (10 positions
    # against C = 9), within the two-gap allowance, so nothing is split
    m = pm.plan([2048] * 128, 1, 152, 128, 1 << 20)
    assert not m["split"] and len(m["tasks"]) == 128 and m["slots"] == 0
    assert pm.chunk_tiles(m).max() == 8
    # 64 such sequences: C = 5, a chunk would carry two whole sequences (20 positions), so
    # the split stays
    m = pm.plan([2048] * 64, 1, 152, 128, 1 << 20)
    assert m["split"] and pm.chunk_tiles(m).max() <= m["C"]
    # long contexts are always split: a unit is many chunks long
    m = pm.plan(MIXES[0][1], 1, 152, 128, 1 << 20)
    assert m["split"] and max(m["nparts"]) > 1
    # more sequences than one plan round: the check is not made
    m = pm.plan([2048] * 1100, 1, 152, 128, 1 << 20)
    assert m["split"]


@pytest.mark.gpu
@pytest.mark.parametrize("name,lens,hkv", MIXES, ids=[m[0] for m in MIXES])
@pytest.mark.parametrize("budget,maxp", [(152, 128), (7, 3), (304, 1), (1, 2)])
@pytest.mark.parametrize("window", [0, 3000])
def test_device_plan_matches_model(name, lens, hkv, budget, maxp, window):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_attention_decode_02_gb300 import build, ops
    build.build()
    ops.load_library()
    B = len(lens)
    S, W, D = 128, max(1, (max(lens) + 127) // 128), 128
    dev = "cuda"
    qlen = 2 if window else 1
    q = torch.zeros(B, qlen, 8 * hkv, D, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(2, hkv, S, D, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(B, W, dtype=torch.int32, device=dev)
    ctx = torch.tensor(lens, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    args = ops.make_args(q, kc, kc, bt, ctx, out, max_partitions=maxp, task_budget=budget,
                         sliding_window=window)
    ws = ops.alloc_workspace(args)
    ops.pa_decode_plan(args, ws)
    torch.cuda.synchronize()
    got = pm.read_workspace(ws.cpu().numpy(), B, hkv, budget)
    m = pm.plan(lens, hkv, budget, maxp, W * S, qlen=qlen, window=window)
    assert got["ntasks"] == len(m["tasks"])
    assert got["tasks"] == m["tasks"]
    assert got["chunks"] == m["chunks"]
    assert got["chunk_first"] == m["chunk_first"]
    assert got["nparts"] == m["nparts"]
    split = [i for i, p in enumerate(m["nparts"]) if p >= 2]
    assert [got["part_base"][i] for i in split] == [m["part_base"][i] for i in split]

"""The work split that pa_decode_plan builds, restated on the host for tests.

Units are (sequence, KV head) pairs in sequence-major order, each with the tiles
[first, ceil(L/256)), where first is the tile holding the first token any query
position's sliding window reaches (0 without a window).  Task tile ranges carry that
offset.  The units are laid end to end on a line, each as a gap of UNIT_COST positions
(the fixed cost of a task) followed by its tiles, and the line is cut into `budget`
chunks of C positions (C = ceil(length / budget), raised when needed so that no unit
touches more than max_partitions chunks); a unit becomes one partition per chunk its
tiles touch.  With max_partitions 1, or an empty unit, the unit is one task in the
chunk its tiles start in.  Splitting is also dropped when no unit is longer than C plus
its gap and, with every unit laid out whole in the chunk its tiles start in, no chunk
carries more than C + 2 UNIT_COST positions (up to WHOLE_UNIT_CHUNKS chunks, and for at
most PLAN_ROUND sequences).

The workspace layout mirrors the library's (256-byte aligned regions): status word and
task count, then nparts, part_base, counters (int32 per unit), tasks (4 x int32 per
task, `capacity` of them), task_chunk (int32 per task), chunk_first (int32, budget + 1).
"""
import math

import numpy as np

TILE = 256
UNIT_COST = 2  # line positions charged per unit before its tiles
WHOLE_UNIT_CHUNKS = 2048
PLAN_ROUND = 1024  # sequences the plan kernel's block holds at once


def _align(x, a=256):
    return (x + a - 1) // a * a


def unit_tiles(L, qlen=1, window=0):
    """(first tile, tile count) of a unit with context L."""
    lo = max(0, L - qlen - window + 1) if window > 0 else 0
    first = lo // TILE
    return first, (L + TILE - 1) // TILE - first


def plan(context_lens, hkv, budget, max_partitions, cap_tokens, unit_cost=UNIT_COST, qlen=1,
         window=0):
    clamped = [min(max(int(L), 0), cap_tokens) for L in context_lens]
    firsts = [unit_tiles(L, qlen, window)[0] for L in clamped]
    tiles = [unit_tiles(L, qlen, window)[1] for L in clamped]
    total = (sum(tiles) + unit_cost * len(tiles)) * hkv  # length of the line
    maxt = max(tiles, default=0)
    C = max(1, -(-total // budget))
    if max_partitions >= 2 and maxt > 0:
        C = max(C, (maxt - 1) // (max_partitions - 1) + 1)
    nchunks = -(-total // C) if total > 0 else 1
    split = max_partitions >= 2
    if split and 0 < maxt <= C + unit_cost and len(tiles) <= PLAN_ROUND and nchunks <= WHOLE_UNIT_CHUNKS:
        load, U = [0] * nchunks, 0
        for n in tiles:
            for h in range(hkv):
                U += unit_cost
                load[min(U // C, nchunks - 1)] += n + unit_cost
                U += n
        if max(load) <= C + 2 * unit_cost:
            split, max_partitions = False, 1
    tasks, chunks, nparts, part_base, unit_pos = [], [], [], [], []
    U, slot = 0, 0
    for s, n in enumerate(tiles):
        for h in range(hkv):
            U += unit_cost  # the unit's gap; its first tile sits at U
            unit_pos.append(U)
            if n == 0 or max_partitions < 2:
                pieces = [(0, n, min(U // C, nchunks - 1))]
            else:
                pieces = [(max(U, c * C) - U, min(U + n, (c + 1) * C) - U, c)
                          for c in range(U // C, (U + n - 1) // C + 1)]
            nparts.append(len(pieces))
            part_base.append(slot if len(pieces) >= 2 else 0)
            if len(pieces) >= 2:
                slot += len(pieces)
            for q, (b, e, c) in enumerate(pieces):
                tasks.append((s, h | (q << 16), b + firsts[s], e + firsts[s]))
                chunks.append(c)
            U += n
    first = [len(tasks)] * (budget + 1)
    prev = -1
    for t, c in enumerate(chunks):
        for k in range(prev + 1, c + 1):
            first[k] = t
        prev = c
    return {"tiles": tiles, "firsts": firsts, "C": C, "nchunks": nchunks, "tasks": tasks, "chunks": chunks,
            "nparts": nparts, "part_base": part_base, "chunk_first": first, "slots": slot,
            "length": total, "unit_pos": unit_pos, "hkv": hkv, "unit_cost": unit_cost, "split": split}


def capacity(batch, hkv, budget):
    return batch * hkv + budget


def read_workspace(ws: np.ndarray, batch, hkv, budget):
    """Decode the plan regions of a workspace (uint8 array, host copy)."""
    units = batch * hkv
    cap = capacity(batch, hkv, budget)
    i32 = lambda off, n: ws[off:off + 4 * n].view(np.int32).copy()
    off = 256
    nparts = i32(off, units)
    off = _align(off + 4 * units)
    part_base = i32(off, units)
    off = _align(off + 4 * units)
    off = _align(off + 4 * units)  # counters
    ntasks = int(i32(4, 1)[0])
    tasks = i32(off, 4 * cap).reshape(cap, 4)[:ntasks]
    off = _align(off + 16 * cap)
    chunks = i32(off, cap)[:ntasks]
    off = _align(off + 4 * cap)
    first = i32(off, budget + 1)
    return {"ntasks": ntasks, "tasks": [tuple(int(x) for x in t) for t in tasks],
            "chunks": chunks.tolist(), "nparts": nparts.tolist(),
            "part_base": part_base.tolist(), "chunk_first": first.tolist()}


def chunk_tiles(model):
    """Tiles each chunk runs."""
    out = np.zeros(len(model["chunk_first"]) - 1, dtype=np.int64)
    for (s, hp, b, e), c in zip(model["tasks"], model["chunks"]):
        out[c] += e - b
    return out


def chunk_load(model):
    """Line positions (tiles and unit gaps) inside each chunk's range."""
    C, w = model["C"], model["unit_cost"]
    out = np.zeros(len(model["chunk_first"]) - 1, dtype=np.int64)
    for c in range(len(out)):
        lo, hi = c * C, min((c + 1) * C, model["length"])
        if hi > lo:
            out[c] = hi - lo
    return out


def ceil_div(a, b):
    return math.ceil(a / b)

"""The launch-time tile schedule (host logic, no GPU), against its
definition written here independently: tiles longest first (the MaskInfo's
row order, or a stable sort by size for per-head masks), a tile of n blocks
costing 8n + 12; the greedy assignment (each tile to the CTA with the least
work so far, ties to the lower index, written with a binary heap) and
MULTIFIT (first-fit decreasing into the lowest-numbered CTA with room, under
the smallest capacity a bisection between the mean and the greedy's maximum
finds), kept when its maximum is at least 3% below the greedy's.  Every tile appears exactly
once, each CTA's list runs longest first and is closed by an end entry, and
no CTA carries more than under the greedy assignment.
"""
import ctypes as C
import heapq

import numpy as np
import pytest

from helpers import ensure_built


def tiles_of(row_len, row_order, rows, heads, n_b, n_g, group, splits):
    gs = group // splits
    tiles = []
    if heads == 1:
        for i in row_order:
            n = int(row_len[i]) * gs
            for bg in range(n_b * n_g):
                for sp in range(splits):
                    tiles.append((int(i), n, bg, sp))
    else:
        for g in range(n_g):
            for i in range(rows):
                for sp in range(splits):
                    n = sum(int(row_len[(g * group + gh) * rows + i]) for gh in range(sp * gs, (sp + 1) * gs))
                    for b in range(n_b):
                        tiles.append((i, n, b * n_g + g, sp))
        tiles.sort(key=lambda t: -t[1])  # stable
    return tiles


def cost(t):
    return 8 * t[1] + 12


def greedy_owners(tiles, grid):
    heap = [(0, c) for c in range(grid)]
    owners = []
    for t in tiles:
        load, c = heapq.heappop(heap)
        owners.append(c)
        heapq.heappush(heap, (load + cost(t), c))
    return owners


def first_fit(tiles, grid, cap):
    load = np.zeros(grid, dtype=np.int64)
    owners = []
    for t in tiles:
        room = load <= cap - cost(t)
        if not room.any():
            return None, None
        c = int(np.argmax(room))
        load[c] += cost(t)
        owners.append(c)
    return owners, int(load.max())


def loads(tiles, owners, grid):
    load = np.zeros(grid, dtype=np.int64)
    for t, c in zip(tiles, owners):
        load[c] += cost(t)
    return load


def reference_lists(row_len, row_order, rows, heads, n_b, n_g, group, splits, grid):
    tiles = tiles_of(row_len, row_order, rows, heads, n_b, n_g, group, splits)
    owners = greedy_owners(tiles, grid)
    greedy_max = int(loads(tiles, owners, grid).max())
    total = sum(cost(t) for t in tiles)
    lo, hi = max(max(cost(t) for t in tiles), -(-total // grid)), greedy_max - 1
    best, best_max = None, greedy_max
    while lo <= hi:
        cap = lo + (hi - lo) // 2
        ff, mx = first_fit(tiles, grid, cap)
        if ff is not None:
            best, best_max = ff, mx
            hi = min(cap, mx) - 1
        else:
            lo = cap + 1
    if best is not None and 100 * (greedy_max - best_max) >= 3 * greedy_max:
        owners = best
    lists = [[] for _ in range(grid)]
    for t, c in zip(tiles, owners):
        lists[c].append(t)
    return lists, tiles, greedy_max


def library_lists(row_len, row_order, rows, heads, n_b, n_g, group, splits, grid):
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    rl = np.ascontiguousarray(row_len, dtype=np.int32)
    ro = np.ascontiguousarray(row_order, dtype=np.int32)
    ptr = lambda a: a.ctypes.data_as(C.POINTER(C.c_int32))  # noqa: E731
    stride = C.c_int32(0)
    probe = np.zeros(4, dtype=np.int32)
    st = L.bsa_debug_tile_schedule(ptr(rl), ptr(ro), rows, heads, n_b, n_g, group, splits, grid, ptr(probe), 0,
                                   C.byref(stride))
    assert st == _abi.INVALID_ARG and stride.value > 0  # cap 0 is too small, the stride comes back
    cap = stride.value
    out = np.zeros(grid * cap * 4, dtype=np.int32)
    _abi.check(L.bsa_debug_tile_schedule(ptr(rl), ptr(ro), rows, heads, n_b, n_g, group, splits, grid, ptr(out),
                                         cap, C.byref(stride)), "bsa_debug_tile_schedule")
    out = out.reshape(grid, cap, 4)
    lists = []
    for c in range(grid):
        k = 0
        lst = []
        while k < cap and out[c, k, 1] >= 0:
            lst.append(tuple(int(x) for x in out[c, k]))
            k += 1
        assert k < cap, "a list without its end entry"
        assert np.all(out[c, k:, 1] == -1)
        lists.append(lst)
    return lists, cap


def order_of(row_len):
    return np.argsort(-np.asarray(row_len), kind="stable").astype(np.int32)


def cases():
    rng = np.random.default_rng(3)
    causal = np.arange(1, 65, dtype=np.int32)                 # 64 rows, causal at 8192
    local = np.minimum(np.arange(1, 65), 9).astype(np.int32)  # local window (1024, 0)
    equal = np.full(16, 16, dtype=np.int32)                   # dense mask, no empty block
    distinct = rng.permutation(np.arange(1, 201)).astype(np.int32)
    yield "causal fwd GQA 32", causal, 1, dict(n_b=1, n_g=32, group=1, splits=1, grid=152)
    yield "causal dkv GQA 32/8", causal, 1, dict(n_b=1, n_g=8, group=4, splits=1, grid=152)
    yield "causal dkv MQA split", causal[:16], 1, dict(n_b=1, n_g=1, group=16, splits=8, grid=128)
    yield "local fwd MHA 16", local, 1, dict(n_b=1, n_g=16, group=1, splits=1, grid=152)
    yield "equal rows, B 2", equal, 1, dict(n_b=2, n_g=16, group=1, splits=1, grid=152)
    yield "all sizes distinct", distinct, 1, dict(n_b=1, n_g=3, group=1, splits=1, grid=37)
    yield "one CTA", causal[:8], 1, dict(n_b=2, n_g=2, group=1, splits=1, grid=1)
    per_head = rng.integers(0, 20, size=(8, 24)).astype(np.int32)   # 8 mask heads x 24 rows
    yield "per-head fwd", per_head.reshape(-1), 8, dict(n_b=2, n_g=8, group=1, splits=1, grid=152)
    yield "per-head dkv GQA 8/2 split", per_head.reshape(-1), 8, dict(n_b=1, n_g=2, group=4, splits=2, grid=64)


@pytest.mark.parametrize("name,row_len,heads,kw", list(cases()), ids=[c[0] for c in cases()])
def test_schedule_follows_its_definition(name, row_len, heads, kw):
    ensure_built()
    rows = row_len.size // heads
    row_order = order_of(row_len) if heads == 1 else np.arange(rows, dtype=np.int32)
    got, cap = library_lists(row_len, row_order, rows, heads, **kw)
    want, tiles, greedy_max = reference_lists(row_len, row_order, rows, heads, **kw)
    assert got == want
    assert cap == max(len(x) for x in want) + 1
    flat = [t for lst in got for t in lst]
    assert len(flat) == len(tiles) == len(set((t[0], t[2], t[3]) for t in flat))
    for lst in got:
        assert all(a[1] >= b[1] for a, b in zip(lst, lst[1:])), "a CTA's list is not longest first"
    assert max(sum(cost(t) for t in lst) for lst in got) <= greedy_max


def test_causal_dkv_tiles_are_balanced():
    """The dK/dV tiles of GQA 32/8 causal at 8192 (every key block once per
    KV head): the greedy assignment leaves its busiest CTAs 6.7% above the
    mean, the kept assignment under 1%."""
    ensure_built()
    row_len = np.arange(64, 0, -1, dtype=np.int32)
    got, _ = library_lists(row_len, order_of(row_len), 64, 1, n_b=1, n_g=8, group=4, splits=1, grid=152)
    _, tiles, _ = reference_lists(row_len, order_of(row_len), 64, 1, 1, 8, 4, 1, 152)
    per_cta = np.array([sum(cost(t) for t in lst) for lst in got])
    mean = per_cta.sum() / 152
    greedy = loads(tiles, greedy_owners(tiles, 152), 152)
    assert greedy.max() / mean > 1.06
    assert per_cta.max() / mean < 1.01


def test_schedule_rejects_bad_arguments():
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    rl = np.arange(1, 9, dtype=np.int32)
    ro = order_of(rl)
    out = np.zeros(64, dtype=np.int32)
    stride = C.c_int32(0)
    ptr = lambda a: a.ctypes.data_as(C.POINTER(C.c_int32))  # noqa: E731
    # group not a multiple of splits, no CTA
    assert L.bsa_debug_tile_schedule(ptr(rl), ptr(ro), 8, 1, 1, 1, 3, 2, 4, ptr(out), 4, C.byref(stride)) == \
        _abi.INVALID_ARG
    assert L.bsa_debug_tile_schedule(ptr(rl), ptr(ro), 8, 1, 1, 1, 1, 1, 0, ptr(out), 4, C.byref(stride)) == \
        _abi.INVALID_ARG

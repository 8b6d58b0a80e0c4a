"""CPU checks of the backward's work-list packing (host logic, no GPU).
kv-major: the items the library builds for given column lengths cover every
(kv block, kv head) column exactly once, cut columns write distinct
partial-sum slots within the allowed number, the CTA index is consistent,
and the exact-fill packing of the one-pass kernel evens the CTAs out.
q-major: every (q tile, q head) with kv blocks is one item with its list
offset and length, and the CTA records add up."""
import ctypes

import numpy as np
import pytest

import prefix_tree_block_gb300 as pt
from prefix_tree_block_gb300 import build as ptbuild

CTAS = 152


@pytest.fixture(scope="module")
def lib():
    ptbuild.build()
    return pt.load_library()


def pack(lib, cols, g, hkv, max_slots, fill, ctas=CTAS):
    cols = np.ascontiguousarray(cols, np.int32)
    cap = int(sum(max(1, -(-g * int(c) // 4)) for c in cols) * hkv + 4 * ctas + 16)
    items = np.zeros((cap, 5), np.int32)
    cta = np.zeros(ctas + 1, np.int32)
    n_items, n_slots, grid = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = lib.pt_debug_pack_dkdv(cols.ctypes.data, len(cols), g, hkv, max_slots, ctas, int(fill), items.ctypes.data,
                                cap, cta.ctypes.data, ctypes.byref(n_items), ctypes.byref(n_slots), ctypes.byref(grid))
    assert rc == pt.PT_OK, rc
    return items[:n_items.value], cta[:grid.value + 1], n_slots.value, grid.value


def check_lists(cols, g, hkv, max_slots, items, cta, n_slots, grid, ctas=CTAS):
    assert 1 <= grid <= ctas
    assert cta[0] == 0 and cta[-1] == len(items) and np.all(np.diff(cta) >= 0)
    by_col = {}
    for jb, hk, x0, x1, slot in items:
        by_col.setdefault((int(jb), int(hk)), []).append((int(x0), int(x1), int(slot)))
    assert set(by_col) == {(j, h) for j in range(len(cols)) for h in range(hkv)}
    used = []
    for (j, h), chunks in by_col.items():
        chunks.sort()
        n = g * int(cols[j])
        x = 0
        for x0, x1, _ in chunks:
            assert x0 == x and x1 >= x0
            x = x1
        assert x == n
        if len(chunks) == 1:
            assert chunks[0][2] == -1
        else:  # a cut column: every chunk writes a slot of its own
            assert all(c[2] >= 0 for c in chunks)
            used += [c[2] for c in chunks]
    assert sorted(used) == list(range(n_slots))
    if max_slots <= 0:
        assert n_slots == 0
    else:
        assert n_slots <= max_slots


def loads(items, cta, grid):
    steps = items[:, 3] - items[:, 2]
    return np.array([steps[cta[b]:cta[b + 1]].sum() + 2 * (cta[b + 1] - cta[b]) for b in range(grid)])


@pytest.mark.parametrize("fill", [False, True])
@pytest.mark.parametrize("max_slots", [0, 48, 100000])
def test_random_columns_covered_once(lib, fill, max_slots):
    rng = np.random.default_rng(7 + max_slots + fill)
    for _ in range(60):
        nk = int(rng.integers(1, 260))
        g, hkv = int(rng.integers(1, 9)), int(rng.integers(1, 5))
        cols = rng.integers(0, nk + 1, nk)
        cols[rng.random(nk) < 0.2] = 0
        items, cta, n_slots, grid = pack(lib, cols, g, hkv, max_slots, fill)
        check_lists(cols, g, hkv, max_slots, items, cta, n_slots, grid)


def grpo_like_columns(groups=8, prompt_tiles=4, completion_tiles=10):
    """kv-block list lengths of GRPO groups: a prompt block is listed by the
    prompt tiles at and after it and by every completion tile of its group; a
    completion block by about two tiles of its own completion."""
    cols = []
    for _ in range(groups):
        n = prompt_tiles + completion_tiles
        cols += [n - j for j in range(prompt_tiles)]
        cols += [2] * completion_tiles
    return np.array(cols, np.int32)


def test_exact_fill_evens_out_the_ctas(lib):
    cols = grpo_like_columns()
    g, hkv = 7, 2
    fill = pack(lib, cols, g, hkv, 256, True)
    lpt = pack(lib, cols, g, hkv, 256, False)
    check_lists(cols, g, hkv, 256, *fill)
    check_lists(cols, g, hkv, 256, *lpt)
    lf, ll = loads(fill[0], fill[1], fill[3]), loads(lpt[0], lpt[1], lpt[3])
    mean = (g * hkv * cols.sum() + 2 * hkv * len(cols)) / CTAS
    assert fill[3] == CTAS and fill[2] > 0  # every CTA has work; long columns were cut
    assert lf.max() <= 1.05 * mean + 4
    assert lf.max() <= ll.max()


def test_exact_fill_balance_on_random_columns(lib):
    rng = np.random.default_rng(11)
    checked = 0
    for _ in range(80):
        nk = int(rng.integers(40, 300))
        g, hkv = int(rng.integers(1, 8)), int(rng.integers(1, 4))
        cols = rng.integers(0, nk, nk)
        total = g * hkv * int(cols.sum())
        if total < 40 * CTAS:
            continue
        items, cta, n_slots, grid = pack(lib, cols, g, hkv, 100000, True)
        check_lists(cols, g, hkv, 100000, items, cta, n_slots, grid)
        mean = (total + 2 * hkv * nk) / CTAS
        assert loads(items, cta, grid).max() <= 1.10 * mean
        checked += 1
    assert checked >= 20


def test_exact_fill_falls_back_without_slots(lib):
    """Too few partial-sum slots for the cuts: the packing is the
    longest-first one, item for item."""
    cols = grpo_like_columns()
    for max_slots in (0, 4):
        a = pack(lib, cols, 7, 2, max_slots, True)
        b = pack(lib, cols, 7, 2, max_slots, False)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2:] == b[2:]


def test_small_problem_uses_longest_first(lib):
    """Under four steps per CTA on average the exact fill is not used: the
    packing is the longest-first one (which still cuts a column longer than
    its chunk of at least four steps)."""
    cols = np.array([3, 1, 0, 2], np.int32)
    a = pack(lib, cols, 2, 1, 100000, True)
    b = pack(lib, cols, 2, 1, 100000, False)
    check_lists(cols, 2, 1, 100000, *a)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2:] == b[2:]
    assert a[2] == 2  # the six-step column in two chunks


def test_bad_arguments_rejected(lib):
    cols = np.array([1, 2], np.int32)
    items = np.zeros((8, 5), np.int32)
    cta = np.zeros(CTAS + 1, np.int32)
    n = [ctypes.c_int32() for _ in range(3)]
    refs = [ctypes.byref(x) for x in n]
    assert lib.pt_debug_pack_dkdv(cols.ctypes.data, 2, 0, 1, 0, CTAS, 0, items.ctypes.data, 8, cta.ctypes.data,
                                  *refs) == pt.PT_ERR_INVALID_ARG
    neg = np.array([1, -1], np.int32)
    assert lib.pt_debug_pack_dkdv(neg.ctypes.data, 2, 1, 1, 0, CTAS, 0, items.ctypes.data, 8, cta.ctypes.data,
                                  *refs) == pt.PT_ERR_INVALID_ARG
    # too little room for the items: refused, the count still reported
    big = np.full(40, 40, np.int32)
    assert lib.pt_debug_pack_dkdv(big.ctypes.data, 40, 4, 2, 0, CTAS, 0, items.ctypes.data, 8, cta.ctypes.data,
                                  *refs) == pt.PT_ERR_INVALID_ARG
    assert n[0].value == 80


def pack_dq(lib, rows, hq, ctas=CTAS):
    rows = np.ascontiguousarray(rows, np.int32)
    cap = max(1, int((rows > 0).sum()) * hq)
    items = np.zeros((cap, 4), np.int32)
    rec = np.zeros((ctas, 4), np.int32)
    n_items, grid, n_empty = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = lib.pt_debug_pack_dq(rows.ctypes.data, len(rows), hq, ctas, items.ctypes.data, cap, rec.ctypes.data,
                              ctypes.byref(n_items), ctypes.byref(grid), ctypes.byref(n_empty))
    assert rc == pt.PT_OK, rc
    return items[:n_items.value], rec[:grid.value], n_empty.value


@pytest.mark.parametrize("ctas", [1, 7, CTAS])
def test_dq_items_cover_every_row_once(lib, ctas):
    rng = np.random.default_rng(ctas)
    for _ in range(40):
        nq = int(rng.integers(1, 200))
        hq = int(rng.integers(1, 9))
        rows = rng.integers(0, nq + 1, nq)
        rows[rng.random(nq) < 0.2] = 0
        items, rec, n_empty = pack_dq(lib, rows, hq, ctas)
        offsets = np.concatenate([[0], np.cumsum(rows)[:-1]])
        want = {(t, h): (int(offsets[t]), int(rows[t])) for t in range(nq) if rows[t] > 0 for h in range(hq)}
        got = {(int(t), int(h)): (int(e0), int(n)) for t, h, e0, n in items}
        assert len(got) == len(items) and got == want
        assert n_empty == int((rows == 0).sum())
        assert len(rec) == max(1, min(ctas, len(items)))
        assert rec[0, 0] == 0 and rec[-1, 1] == len(items) and np.all(rec[1:, 0] == rec[:-1, 1])
        for x, y, blocks, _ in rec:
            assert blocks == items[x:y, 3].sum()
        # longest first: every CTA's items in non-increasing order of length
        for x, y, _, _ in rec:
            assert np.all(np.diff(items[x:y, 3]) <= 0)


def test_dq_items_balanced(lib):
    """Longest-first packing of many items: no CTA more than one item's
    length (plus its fixed cost) above the mean."""
    rng = np.random.default_rng(5)
    rows = rng.integers(1, 40, 230)
    items, rec, _ = pack_dq(lib, rows, 8)
    load = np.array([rec_b[2] + 2 * (rec_b[1] - rec_b[0]) for rec_b in rec])
    assert load.max() <= load.mean() + rows.max() + 2

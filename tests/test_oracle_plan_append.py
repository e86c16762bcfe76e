"""Pins for the oracle's work split (plan) and its kv_append.

Plan: units are (row, KV head, page) tiles in that order; in the uniform
split, of C chunks asked for, Ce = min(C, T) are used, chunk k covering
[floor(k T / Ce), floor((k + 1) T / Ce)), so none is empty; a segment (row,
head) is split into pieces by the chunks it meets.  Pinned to hand-derived
fixtures and to a brute-force enumeration of every unit.  The segment-aligned
split is pinned to hand-derived cases and to its structure.

Append (tinyllm, "The repository currently provides": block table per active
sequence; "Known limitations": 16-token pages): row i's new token goes to page
block_table[i][(L_i - 1) // 16], slot (L_i - 1) % 16, stored with the f16 or
q8_0 encoder; nothing else in the pool changes."""
import json
import os

import numpy as np
import pytest

import oracle as O
from conftest import GOLDEN
from paged_kv_decode_09_gb300 import workloads as W


def _golden():
    with open(os.path.join(GOLDEN, "plan_tiny.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: f"C{c['chunks']}_{len(c['seq_lens'])}rows")
def test_plan_golden(case):
    rps, first, last, T = O.plan(np.array(case["seq_lens"], np.int32), case["n_kv"], case["chunks"])
    assert T == case["total"]
    np.testing.assert_array_equal(rps, case["row_page_start"])
    np.testing.assert_array_equal(first, case["seg_first_chunk"])
    np.testing.assert_array_equal(last, case["seg_last_chunk"])


def _pages_read(L, window):
    """Pages of a row holding an attended token: tokens max(0, L - window)..L-1
    (all L for window 0), by brute force over the tokens."""
    first = max(0, L - window) if window > 0 else 0
    return sorted({t // 16 for t in range(first, max(L, 0))})


def _enumerate(seq_lens, n_kv, C, window=0):
    """Brute force: list every unit with its (segment, chunk) and derive the
    chunks each segment meets."""
    units = []  # (segment, chunk) per unit, in unit order
    for i, L in enumerate(seq_lens):
        npg = len(_pages_read(L, window))
        for h in range(n_kv):
            for p in range(npg):
                units.append(i * n_kv + h)
    T = len(units)
    Ce = min(C, T)
    chunk_of = []
    for k in range(Ce):
        n = (k + 1) * T // Ce - k * T // Ce
        assert n >= 1  # no empty chunk
        chunk_of += [k] * n
    J = len(seq_lens) * n_kv
    first, last = [-1] * J, [-1] * J
    for x, j in enumerate(units):
        if first[j] < 0:
            first[j] = chunk_of[x]
        last[j] = chunk_of[x]
    return T, first, last


@pytest.mark.parametrize("seed", range(8))
def test_plan_matches_unit_enumeration(seed):
    rng = np.random.default_rng(seed)
    rows = int(rng.integers(1, 12))
    lens = rng.integers(0, 200, rows).astype(np.int32)
    lens[rng.integers(0, rows)] = 0
    n_kv = int(rng.choice([1, 2, 8]))
    for C in (1, 3, 7, 152, 1000):
        rps, first, last, T = O.plan(lens, n_kv, C)
        T2, f2, l2 = _enumerate(lens.tolist(), n_kv, C)
        assert T == T2
        np.testing.assert_array_equal(first, f2)
        np.testing.assert_array_equal(last, l2)
        np.testing.assert_array_equal(np.diff(rps), (np.maximum(lens, 0) + 15) // 16)


@pytest.mark.parametrize("seed", range(6))
def test_windowed_plan_matches_unit_enumeration(seed):
    """With a sliding window a row's units are the pages holding its last W
    tokens; page p of the row's units is block-table entry floor(a / 16) + p."""
    rng = np.random.default_rng(100 + seed)
    rows = int(rng.integers(1, 10))
    lens = rng.integers(0, 300, rows).astype(np.int32)
    n_kv = int(rng.choice([1, 2, 8]))
    for window in (1, 15, 16, 17, 64, 100, 299, 1000):
        for C in (1, 5, 152):
            rps, first, last, T = O.plan(lens, n_kv, C, window=window)
            T2, f2, l2 = _enumerate(lens.tolist(), n_kv, C, window)
            assert T == T2
            np.testing.assert_array_equal(first, f2)
            np.testing.assert_array_equal(last, l2)
            pages = [_pages_read(int(L), window) for L in lens]
            np.testing.assert_array_equal(np.diff(rps), [len(p) for p in pages])
            for L, p in zip(lens, pages):  # contiguous run starting at floor(a / 16)
                if p:
                    assert p == list(range(max(0, int(L) - window) // 16, p[-1] + 1))


# The segment-aligned split (f16 and bf16 KV).  For a cap of t units a
# chunk, a row of npg >= t pages cuts each KV head's segment into
# c = ceil(npg / t) chunks (chunk q: pages [floor(q npg / c), floor((q+1) npg / c))),
# a shorter row groups m = floor(t / npg) whole segments a chunk; t is the
# first cap from ceil(T / C) to floor(1.1 T / C) whose chunks number at most
# C; with a single cap in that range, or none fitting, the split is uniform.

def test_aligned_split_hand_worked():
    """Rows of 470 and 70 tokens = 30 and 5 pages, 2 KV heads, 5 chunks:
    T = 70, caps 14 .. 15.  Cap 14: row 0 needs 2 * ceil(30 / 14) = 6 > 5.
    Cap 15: 2 * 2 chunks of 15 pages for row 0, and row 1 (5 < 15) groups
    floor(15 / 5) = 3 >= 2 heads in one chunk: 5 chunks."""
    lens = np.array([470, 70], np.int32)
    lo, hi = O.chunk_ranges(lens, 2, 5, aligned=True)
    np.testing.assert_array_equal(lo, [0, 15, 30, 45, 60])
    np.testing.assert_array_equal(hi, [15, 30, 45, 60, 70])
    rps, first, last, T = O.plan(lens, 2, 5, aligned=True)
    assert T == 70
    np.testing.assert_array_equal(first, [0, 2, 4, 4])
    np.testing.assert_array_equal(last, [1, 3, 4, 4])
    # the uniform split of the same call: [0,14) [14,28) [28,42) [42,56) [56,70)
    rps, first, last, T = O.plan(lens, 2, 5, aligned=False)
    np.testing.assert_array_equal(first, [0, 2, 4, 4])
    np.testing.assert_array_equal(last, [2, 4, 4, 4])


def test_aligned_split_whole_segments_of_a_long_and_a_short_row():
    """30 and 3 pages, 8 KV heads, 9 chunks: T = 264, caps 30 .. 32.  Cap 30:
    row 0 gives each head one chunk (30 >= 30, ceil(30 / 30) = 1), row 1
    groups floor(30 / 3) = 10 >= 8 heads in one chunk: 9 chunks."""
    lens = np.array([480, 48], np.int32)
    lo, hi = O.chunk_ranges(lens, 8, 9, aligned=True)
    np.testing.assert_array_equal(lo, [0, 30, 60, 90, 120, 150, 180, 210, 240])
    np.testing.assert_array_equal(hi, [30, 60, 90, 120, 150, 180, 210, 240, 264])
    rps, first, last, T = O.plan(lens, 8, 9, aligned=True)
    np.testing.assert_array_equal(first, list(range(8)) + [8] * 8)
    np.testing.assert_array_equal(last, list(range(8)) + [8] * 8)


def _same_plan(lens, n_kv, C):
    for a, b in zip(O.plan(lens, n_kv, C, aligned=True), O.plan(lens, n_kv, C, aligned=False)):
        np.testing.assert_array_equal(a, b)
    lo, hi = O.chunk_ranges(lens, n_kv, C, aligned=True)
    T = n_kv * int(sum((int(L) + 15) // 16 for L in lens))
    np.testing.assert_array_equal(lo, [k * T // C for k in range(C)])


def test_aligned_split_falls_back_when_no_cap_fits():
    """30 and 4 pages, 8 KV heads, 10 chunks: T = 272, caps 28 .. 29.  Row 0
    alone needs 8 * ceil(30 / 28) = 8 * ceil(30 / 29) = 16 > 10 chunks."""
    _same_plan(np.array([480, 64], np.int32), 8, 10)


def test_aligned_split_needs_room_above_the_even_share():
    """6, 1 and 1 pages, 2 KV heads, 6 chunks: T = 16, ceil(T / C) = 3 but
    floor(1.1 T / C) = 2: a single cap (none above the even share), so the
    split is uniform although cap 3 would need only 6 chunks."""
    _same_plan(np.array([90, 5, 1], np.int32), 2, 6)


@pytest.mark.parametrize("seed", range(10))
def test_aligned_split_structure(seed):
    """Whatever split comes out tiles [0, T) with non-empty chunks, at most C
    of them; when it is not the uniform one, every chunk lies inside one
    segment or is whole segments of one row, a segment split over several
    chunks starts and ends on chunk boundaries, and no chunk holds more than
    max(ceil(T / C), floor(1.1 T / C)) units."""
    rng = np.random.default_rng(300 + seed)
    rows = int(rng.integers(1, 40))
    lens = rng.integers(0, 3000, rows).astype(np.int32)
    lens[rng.integers(0, rows, 2)] = 0
    n_kv = int(rng.choice([1, 2, 4, 8]))
    for C in (1, 4, 37, 152, 456, 5000):
        rps, first, last, T = O.plan(lens, n_kv, C, aligned=True)
        lo, hi = O.chunk_ranges(lens, n_kv, C, aligned=True)
        if T == 0:
            assert len(lo) == 0
            continue
        assert lo[0] == 0 and hi[-1] == T and np.all(hi > lo) and np.all(lo[1:] == hi[:-1])
        assert len(lo) <= C
        ulo, uhi = O.chunk_ranges(lens, n_kv, C, aligned=False)
        if len(lo) == len(ulo) and np.array_equal(lo, ulo):
            continue  # the uniform split (possibly also what alignment gives)
        npg = np.diff(rps)
        seg_start = np.concatenate([[0], np.cumsum(np.repeat(npg, n_kv))])
        seg_row = np.repeat(np.arange(rows), n_kv)
        bounds = set(lo.tolist()) | {T}
        for a, b in zip(lo, hi):
            j0 = np.searchsorted(seg_start, a, "right") - 1
            j1 = np.searchsorted(seg_start, b, "left") - 1
            if j0 != j1:  # several segments: all whole, of one row
                assert seg_start[j0] == a and seg_start[j1 + 1] == b
                assert seg_row[j0] == seg_row[j1]
        for j in range(rows * n_kv):
            if first[j] >= 0 and first[j] != last[j]:
                assert seg_start[j] in bounds and seg_start[j + 1] in bounds
        assert 11 * T // (10 * C) > -(-T // C)  # room above the even share
        assert np.max(hi - lo) <= 11 * T // (10 * C)


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0])
def test_append_writes_one_slot_with_encoder_bytes(dtype):
    rng = np.random.default_rng(21)
    rows, n_kv, D, num_pages = 4, 2, 128, 12
    lens = np.array([1, 17, 32, 5], np.int32)   # slot 0 of page 0, slot 0 of page 1, slot 15, slot 4
    bt = np.full((rows, 3), -1, np.int32)
    bt[:, :2] = rng.permutation(num_pages)[:8].reshape(rows, 2)
    q8 = dtype == W.Q8_0
    kd = rng.integers(0, 2**15, (num_pages, n_kv, 16, D)).astype(np.uint16)
    if q8:
        kd = rng.integers(-127, 128, (num_pages, n_kv, 16, D)).astype(np.int8)
    vd = kd.copy()
    ks = rng.integers(0, 2**14, (num_pages, n_kv, 16, D // 32)).astype(np.uint16) if q8 else None
    vs = ks.copy() if q8 else None
    before = [a.copy() for a in (kd, vd) + ((ks, vs) if q8 else ())]
    k_new = rng.standard_normal((rows, n_kv, D)).astype(np.float32)
    v_new = rng.standard_normal((rows, n_kv, D)).astype(np.float32)
    O.kv_append(dtype, k_new, v_new, bt, lens, num_pages, kd, vd, ks, vs)
    touched = np.zeros((num_pages, 16), bool)
    for i, L in enumerate(lens):
        page, slot = bt[i, (L - 1) // 16], (L - 1) % 16
        touched[page, slot] = True
        for h in range(n_kv):
            if q8:
                ck, sk = O.q8_0_encode(k_new[i, h])
                cv, sv = O.q8_0_encode(v_new[i, h])
                np.testing.assert_array_equal(kd[page, h, slot], ck)
                np.testing.assert_array_equal(ks[page, h, slot], sk)
                np.testing.assert_array_equal(vd[page, h, slot], cv)
                np.testing.assert_array_equal(vs[page, h, slot], sv)
            else:
                np.testing.assert_array_equal(kd[page, h, slot], O.f16_encode(k_new[i, h]))
                np.testing.assert_array_equal(vd[page, h, slot], O.f16_encode(v_new[i, h]))
    # explicit page/slot addressing of the worked rows
    assert touched[bt[0, 0], 0] and touched[bt[1, 1], 0] and touched[bt[2, 1], 15]
    assert touched[bt[3, 0], 4]
    for arr, old in zip((kd, vd) + ((ks, vs) if q8 else ()), before):
        keep = ~touched
        np.testing.assert_array_equal(arr[keep[:, None, :].repeat(n_kv, 1)],
                                      old[keep[:, None, :].repeat(n_kv, 1)])


def test_append_rejects_page_outside_pool():
    bt = np.array([[7]], np.int32)
    kd = np.zeros((4, 1, 16, 32), np.uint16)
    with pytest.raises(ValueError):
        O.kv_append(W.F16, np.zeros((1, 1, 32), np.float32), np.zeros((1, 1, 32), np.float32),
                    bt, np.array([3], np.int32), 4, kd, kd.copy())


def test_append_f32_stores_the_values_unrounded():
    """f32 KV (tinyllm, "The repository currently provides": BF16/F32 KV
    caching) keeps the fp32 inputs as they are: the slot holds k_new and v_new
    bit for bit, in the K and V arrays respectively, and nothing else moves."""
    rng = np.random.default_rng(23)
    rows, n_kv, D, num_pages = 3, 2, 64, 8
    lens = np.array([1, 18, 32], np.int32)
    bt = rng.permutation(num_pages)[:6].reshape(rows, 2).astype(np.int32)
    kd = rng.standard_normal((num_pages, n_kv, 16, D)).astype(np.float32)
    vd = rng.standard_normal((num_pages, n_kv, 16, D)).astype(np.float32)
    k0, v0 = kd.copy(), vd.copy()
    k_new = rng.standard_normal((rows, n_kv, D)).astype(np.float32)
    v_new = rng.standard_normal((rows, n_kv, D)).astype(np.float32)
    O.kv_append(O.F32, k_new, v_new, bt, lens, num_pages, kd, vd)
    for i, L in enumerate(lens):
        page, slot = bt[i, (L - 1) // 16], (L - 1) % 16
        np.testing.assert_array_equal(kd[page, :, slot].view(np.uint32), k_new[i].view(np.uint32))
        np.testing.assert_array_equal(vd[page, :, slot].view(np.uint32), v_new[i].view(np.uint32))
        k0[page, :, slot], v0[page, :, slot] = k_new[i], v_new[i]
    np.testing.assert_array_equal(kd, k0)
    np.testing.assert_array_equal(vd, v0)

"""Pins for the oracle's work split (plan) and its kv_append.

Plan: units are (row, KV head, page) tiles in that order; of C chunks asked
for, Ce = min(C, T) are used, chunk k covering [floor(k T / Ce),
floor((k + 1) T / Ce)), so none is empty; a segment (row, head) is split into
pieces by the chunks it meets.  Pinned to hand-derived fixtures and to a
brute-force enumeration of every unit.

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

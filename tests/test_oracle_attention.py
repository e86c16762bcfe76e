"""Pins for the oracle's decode attention, partial states and merge.

Definition (tinyllm, "The repository currently provides": GQA attention with
contiguous and paged-reference cache paths; "Known limitations": the paged
reference gathers a row's pages, then runs dense attention):
    out[i][g] = sum_t softmax_t(scale <q[i][g], K[i][g // G][t]>) V[i][g // G][t].
The oracle is pinned to a separately written brute force that works on dense
per-row arrays (no block table, no max subtraction, exact fsum dot products),
to closed forms (one token, constant V, zero query or zero scale, two tokens),
and to invariants (contiguous vs paged pages, page permutations, GQA head map,
splitting a row into partial states and merging them)."""
import math

import numpy as np
import pytest

import oracle as O
from helpers import stored_values_dense

PAGE = 16


def _random_stored(rng, dtype, shape):
    """Random stored K or V values [..., D]: (data, scales)."""
    x = rng.standard_normal(shape).astype(np.float32)
    return O.encode_pool(dtype, x)


def _scatter_rows(rng, dtype, dense_k, dense_v, lens, n_kv, D, extra_pages=3, order=None):
    """Place dense per-row stored tokens [rows] of ([n_kv][L][D] data, scales)
    into a pool of 16-token pages; returns (pool arrays, block_table, num_pages)."""
    npg = [(L + PAGE - 1) // PAGE for L in lens]
    num_pages = sum(npg) + extra_pages
    ids = np.arange(num_pages) if order == "contiguous" else rng.permutation(num_pages)
    stride = max(max(npg), 1)
    bt = np.full((len(lens), stride), -1, np.int32)
    q8 = dtype == O.Q8_0
    nan16 = 0x7FC0 if dtype == O.BF16 else 0x7E00  # NaN in the stored 16-bit format
    if dtype == O.F32:
        kd = np.full((num_pages, n_kv, PAGE, D), np.nan, np.float32)
    else:
        kd = np.full((num_pages, n_kv, PAGE, D), nan16 if not q8 else 127,
                     np.uint16 if not q8 else np.int8)
    vd = kd.copy()
    ks = np.full((num_pages, n_kv, PAGE, D // 32), 0x7E00, np.uint16) if q8 else None
    vs = ks.copy() if q8 else None
    at = 0
    for i, L in enumerate(lens):
        for p in range(npg[i]):
            bt[i, p] = ids[at]
            at += 1
        for t in range(L):
            page, slot = bt[i, t // PAGE], t % PAGE
            kd[page, :, slot] = dense_k[i][0][:, t]
            vd[page, :, slot] = dense_v[i][0][:, t]
            if q8:
                ks[page, :, slot] = dense_k[i][1][:, t]
                vs[page, :, slot] = dense_v[i][1][:, t]
    return (kd, vd, ks, vs), bt, num_pages


def _case(seed, dtype, lens, n_q, n_kv, D, order=None):
    rng = np.random.default_rng(seed)
    dk = [_random_stored(rng, dtype, (n_kv, L, D)) for L in lens]
    dv = [_random_stored(rng, dtype, (n_kv, L, D)) for L in lens]
    q = rng.standard_normal((len(lens), n_q, D)).astype(np.float32)
    pool, bt, num_pages = _scatter_rows(rng, dtype, dk, dv, lens, n_kv, D, order=order)
    return q, dk, dv, pool, bt, num_pages


def _brute(dtype, q, dk, dv, lens, n_q, n_kv, scale):
    """Dense brute force in Python floats: exp without max subtraction."""
    G = n_q // n_kv
    rows, _, D = q.shape
    out = np.zeros((rows, n_q, D))
    for i, L in enumerate(lens):
        K = stored_values_dense(dtype, dk[i][0], dk[i][1])  # [n_kv][L][D]
        V = stored_values_dense(dtype, dv[i][0], dv[i][1])
        for g in range(n_q):
            h = g // G
            w = [math.exp(scale * math.fsum(float(a) * float(b) for a, b in zip(q[i, g], K[h, t])))
                 for t in range(L)]
            den = math.fsum(w)
            for d in range(D):
                out[i, g, d] = math.fsum(w[t] * V[h, t, d] for t in range(L)) / den
    return out


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0, O.BF16, O.F32])
@pytest.mark.parametrize("shape", [(4, 4, 32), (4, 2, 64), (8, 2, 128), (2, 2, 32)])
def test_against_dense_brute_force(dtype, shape):
    n_q, n_kv, D = shape
    lens = [1, 16, 17, 40] if D <= 64 else [3, 33]
    q, dk, dv, pool, bt, num_pages = _case(hash((dtype, shape)) % 1000, dtype, lens, n_q, n_kv, D)
    scale = 1.0 / math.sqrt(D)
    got = O.decode_attention(dtype, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv, scale)
    ref = _brute(dtype, q, dk, dv, lens, n_q, n_kv, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0, O.BF16, O.F32])
def test_contiguous_equals_paged(dtype):
    lens, n_q, n_kv, D = [5, 16, 47, 70], 4, 2, 128
    a = _case(3, dtype, lens, n_q, n_kv, D, order="contiguous")
    b = _case(3, dtype, lens, n_q, n_kv, D)
    assert not np.array_equal(a[4], b[4])  # different physical pages
    sl = np.array(lens, np.int32)
    oa = O.decode_attention(dtype, a[0], *a[3], a[4], sl, a[5], n_kv, 0.088)
    ob = O.decode_attention(dtype, b[0], *b[3], b[4], sl, b[5], n_kv, 0.088)
    np.testing.assert_array_equal(oa, ob)


def test_page_permutation_invariance():
    lens, n_q, n_kv, D = [30, 64, 9], 4, 4, 64
    q, dk, dv, (kd, vd, ks, vs), bt, num_pages = _case(4, O.F16, lens, n_q, n_kv, D)
    sl = np.array(lens, np.int32)
    base = O.decode_attention(O.F16, q, kd, vd, None, None, bt, sl, num_pages, n_kv, 0.125)
    perm = np.random.default_rng(5).permutation(num_pages)  # new page id of old page p
    kd2, vd2 = np.empty_like(kd), np.empty_like(vd)
    kd2[perm], vd2[perm] = kd, vd
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    got = O.decode_attention(O.F16, q, kd2, vd2, None, None, bt2, sl, num_pages, n_kv, 0.125)
    np.testing.assert_array_equal(base, got)


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0, O.BF16, O.F32])
def test_single_token_returns_v(dtype):
    q, dk, dv, pool, bt, num_pages = _case(6, dtype, [1, 1], 4, 2, 128)
    out = O.decode_attention(dtype, q, *pool, bt, np.array([1, 1], np.int32), num_pages, 2, 0.3)
    for i in range(2):
        V = stored_values_dense(dtype, dv[i][0], dv[i][1])
        for g in range(4):
            np.testing.assert_array_equal(out[i, g], V[g // 2, 0])


def test_constant_v_returns_v():
    rng = np.random.default_rng(8)
    lens, n_kv, D = [37], 2, 64
    dk = [_random_stored(rng, O.F16, (n_kv, 37, D))]
    v_tok = _random_stored(rng, O.F16, (n_kv, 1, D))[0]
    dv = [(np.repeat(v_tok, 37, axis=1), None)]
    pool, bt, num_pages = _scatter_rows(rng, O.F16, dk, dv, lens, n_kv, D)
    q = rng.standard_normal((1, 4, D)).astype(np.float32) * 3
    out = O.decode_attention(O.F16, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv, 0.2)
    V = v_tok.view(np.float16).astype(np.float64)[:, 0]
    for g in range(4):
        np.testing.assert_allclose(out[0, g], V[g // 2], rtol=1e-14, atol=0)


@pytest.mark.parametrize("which", ["zero_q", "zero_scale"])
def test_uniform_weights_give_mean_of_v(which):
    lens, n_q, n_kv, D = [23, 50], 4, 2, 32
    q, dk, dv, pool, bt, num_pages = _case(9, O.Q8_0, lens, n_q, n_kv, D)
    scale = 0.7
    if which == "zero_q":
        q = np.zeros_like(q)
    else:
        scale = 0.0
    out = O.decode_attention(O.Q8_0, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv, scale)
    for i in range(2):
        V = stored_values_dense(O.Q8_0, dv[i][0], dv[i][1])
        for g in range(n_q):
            np.testing.assert_allclose(out[i, g], V[g // 2].mean(axis=0), rtol=0, atol=1e-14)


def test_two_token_closed_form():
    q, dk, dv, pool, bt, num_pages = _case(10, O.F16, [2], 2, 1, 128)
    scale = 1 / math.sqrt(128)
    out = O.decode_attention(O.F16, q, *pool, bt, np.array([2], np.int32), num_pages, 1, scale)
    K = stored_values_dense(O.F16, dk[0][0], None)[0]
    V = stored_values_dense(O.F16, dv[0][0], None)[0]
    for g in range(2):
        s = scale * (K @ q[0, g].astype(np.float64))
        w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
        np.testing.assert_allclose(out[0, g], w0 * V[0] + (1 - w0) * V[1], rtol=0, atol=1e-14)


def test_gqa_head_map_contiguous_groups():
    """Query head g reads KV head g // G: give every KV head its own constant V."""
    rng = np.random.default_rng(12)
    n_q, n_kv, D, L = 8, 4, 32, 20
    dk = [_random_stored(rng, O.F16, (n_kv, L, D))]
    vals = (np.arange(n_kv, dtype=np.float32) + 1)[:, None, None] * np.ones((n_kv, L, D), np.float32)
    dv = [(O.f16_encode(vals), None)]
    pool, bt, num_pages = _scatter_rows(rng, O.F16, dk, dv, [L], n_kv, D)
    q = rng.standard_normal((1, n_q, D)).astype(np.float32)
    out = O.decode_attention(O.F16, q, *pool, bt, np.array([L], np.int32), num_pages, n_kv, 0.5)
    for g in range(n_q):
        np.testing.assert_allclose(out[0, g], g // 2 + 1, rtol=1e-15)


def test_equal_queries_in_a_group_give_equal_outputs():
    q, dk, dv, pool, bt, num_pages = _case(13, O.Q8_0, [29], 4, 1, 64)
    q[0, 1] = q[0, 0]
    out = O.decode_attention(O.Q8_0, q, *pool, bt, np.array([29], np.int32), num_pages, 1, 0.1)
    np.testing.assert_array_equal(out[0, 0], out[0, 1])
    assert not np.array_equal(out[0, 0], out[0, 2])


def test_peaked_scores_select_one_token():
    """A key aligned with a large query dominates: out -> that token's V."""
    rng = np.random.default_rng(14)
    L, D = 40, 64
    dk = [_random_stored(rng, O.F16, (1, L, D))]
    dv = [_random_stored(rng, O.F16, (1, L, D))]
    pool, bt, num_pages = _scatter_rows(rng, O.F16, dk, dv, [L], 1, D)
    K = stored_values_dense(O.F16, dk[0][0], None)[0]
    q = (K[23] * 50).astype(np.float32)[None, None]
    out = O.decode_attention(O.F16, q, *pool, bt, np.array([L], np.int32), num_pages, 1, 1.0)
    V = stored_values_dense(O.F16, dv[0][0], None)[0]
    np.testing.assert_allclose(out[0, 0], V[23], atol=1e-12)


def test_empty_row_gives_zeros_and_bad_page_raises():
    q, dk, dv, pool, bt, num_pages = _case(15, O.F16, [5, 3], 2, 1, 32)
    out = O.decode_attention(O.F16, q, *pool, bt, np.array([0, 3], np.int32), num_pages, 1, 0.2)
    assert np.all(out[0] == 0) and np.all(np.isfinite(out[1]))
    bad = bt.copy()
    bad[1, 0] = num_pages
    with pytest.raises(ValueError):
        O.decode_attention(O.F16, q, *pool, bad, np.array([5, 3], np.int32), num_pages, 1, 0.2)


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0])
def test_partials_merge_to_full_attention(dtype):
    lens, n_q, n_kv, D = [75], 4, 2, 128
    q, dk, dv, pool, bt, num_pages = _case(16, dtype, lens, n_q, n_kv, D)
    scale = 1 / math.sqrt(D)
    full = O.decode_attention(dtype, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv, scale)
    for g in range(n_q):
        for cuts in ([0, 75], [0, 16, 75], [0, 1, 2, 40, 75], [0, 30, 31, 74, 75]):
            parts = [O.attention_partial(dtype, q[0], *pool, bt, num_pages, n_kv, 0, g, scale, a, b)
                     for a, b in zip(cuts[:-1], cuts[1:])]
            m2 = np.array([p[0] for p in parts])
            l = np.array([p[1] for p in parts])
            acc = np.array([p[2] for p in parts])
            # the partial states themselves: base-2 softmax pieces of the same scores
            assert np.all(l >= 1.0) and np.all(l <= np.diff(cuts))
            merged = O.combine(m2, l, acc)
            np.testing.assert_allclose(merged, full[0, g], rtol=0, atol=2e-6)


def test_merge_is_invariant_to_rescaled_partials():
    rng = np.random.default_rng(17)
    m2 = rng.standard_normal(5).astype(np.float32) * 4
    l = rng.uniform(1, 10, 5).astype(np.float32)
    acc = rng.standard_normal((5, 16)).astype(np.float32)
    a = O.combine(m2, l, acc)
    # shifting one partial's reference point by c multiplies its l and acc by 2^-c
    m2b, lb, accb = m2.copy(), l.copy(), acc.copy()
    m2b[2] += 3
    lb[2] /= 8
    accb[2] /= 8
    np.testing.assert_allclose(O.combine(m2b, lb, accb), a, rtol=1e-12)
    # one partial: out = acc / l
    np.testing.assert_allclose(O.combine(m2[:1], l[:1], acc[:1]),
                               acc[0].astype(np.float64) / np.float64(l[0]), rtol=1e-15)


# ---------------------------------------------------------------------------
# Sliding window (LeatEngine, "Capabilities": sliding-window KV caches).  Reading:
# with W > 0 a row of L tokens attends to [max(0, L - W), L).

def _brute_window(dtype, q, dk, dv, lens, n_q, n_kv, scale, window):
    """Dense brute force over each row's last `window` tokens."""
    G = n_q // n_kv
    rows, _, D = q.shape
    out = np.zeros((rows, n_q, D))
    for i, L in enumerate(lens):
        a = max(0, L - window)
        K = stored_values_dense(dtype, dk[i][0], dk[i][1])
        V = stored_values_dense(dtype, dv[i][0], dv[i][1])
        for g in range(n_q):
            h = g // G
            w = [math.exp(scale * math.fsum(float(x) * float(y) for x, y in zip(q[i, g], K[h, t])))
                 for t in range(a, L)]
            den = math.fsum(w)
            for d in range(D):
                out[i, g, d] = math.fsum(w[t - a] * V[h, t, d] for t in range(a, L)) / den
    return out


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0])
@pytest.mark.parametrize("window", [1, 5, 16, 17, 39])
def test_window_against_dense_brute_force(dtype, window):
    lens, n_q, n_kv, D = [1, 16, 17, 40], 4, 2, 32
    q, dk, dv, pool, bt, num_pages = _case(31 + window, dtype, lens, n_q, n_kv, D)
    got = O.decode_attention(dtype, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv, 0.2,
                             window=window)
    ref = _brute_window(dtype, q, dk, dv, lens, n_q, n_kv, 0.2, window)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0])
def test_window_at_least_the_length_is_full_attention(dtype):
    lens, n_q, n_kv, D = [3, 33, 64], 4, 2, 64
    q, dk, dv, pool, bt, num_pages = _case(41, dtype, lens, n_q, n_kv, D)
    sl = np.array(lens, np.int32)
    full = O.decode_attention(dtype, q, *pool, bt, sl, num_pages, n_kv, 0.1)
    for window in (64, 65, 10**6):
        np.testing.assert_array_equal(
            O.decode_attention(dtype, q, *pool, bt, sl, num_pages, n_kv, 0.1, window=window), full)


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0])
def test_window_one_returns_the_newest_v(dtype):
    lens, n_q, n_kv, D = [1, 20, 48], 4, 2, 64
    q, dk, dv, pool, bt, num_pages = _case(43, dtype, lens, n_q, n_kv, D)
    out = O.decode_attention(dtype, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv, 0.5,
                             window=1)
    for i, L in enumerate(lens):
        V = stored_values_dense(dtype, dv[i][0], dv[i][1])
        for g in range(n_q):
            np.testing.assert_array_equal(out[i, g], V[g // 2, L - 1])


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0])
def test_window_equals_full_attention_of_the_truncated_rows(dtype):
    """The last W tokens re-paged from slot 0 as rows of their own give the
    same result, bit for bit (same values, same order of summation)."""
    lens, n_q, n_kv, D, window = [9, 30, 70, 100], 4, 2, 64, 37
    q, dk, dv, pool, bt, num_pages = _case(47, dtype, lens, n_q, n_kv, D)
    got = O.decode_attention(dtype, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv, 0.15,
                             window=window)
    cut = [min(L, window) for L in lens]

    def tail(parts, L):
        data, sc = parts
        return (data[:, L - min(L, window):], None if sc is None else sc[:, L - min(L, window):])

    dk2 = [tail(dk[i], L) for i, L in enumerate(lens)]
    dv2 = [tail(dv[i], L) for i, L in enumerate(lens)]
    pool2, bt2, np2 = _scatter_rows(np.random.default_rng(48), dtype, dk2, dv2, cut, n_kv, D)
    want = O.decode_attention(dtype, q, *pool2, bt2, np.array(cut, np.int32), np2, n_kv, 0.15)
    np.testing.assert_array_equal(got, want)

"""Pins for the oracle's several-queries-per-row attention and append
(chunked prefill and speculative verification: Leone, "What ships";
LeatEngine, "Capabilities").

Reading: a row of L tokens whose last q_len are new has one query per new
token; query j sits at position P = L - q_len + j and attends causally to
[max(0, P + 1 - W), P + 1) under a window W (all of [0, P + 1) without one).
Pinned to: the single-query oracle (q_len = 1 is the same call; query j is
single-query attention over length P + 1, bit for bit), a dense causal brute
force, causality (poisoning every token after P leaves query j unchanged),
and for the append, q_len single appends with growing lengths."""
import math

import numpy as np
import pytest

import oracle as O
from helpers import stored_values_dense
from test_oracle_attention import _case


def _mq_case(seed, dtype, lens, q_len, n_q, n_kv, D):
    q1, dk, dv, pool, bt, num_pages = _case(seed, dtype, lens, n_q, n_kv, D)
    rng = np.random.default_rng(seed + 1000)
    q = rng.standard_normal((len(lens), q_len, n_q, D)).astype(np.float32)
    return q, dk, dv, pool, bt, num_pages


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0, O.BF16, O.F32])
def test_one_query_is_the_single_query_call(dtype):
    lens, n_q, n_kv, D = [3, 17, 40], 4, 2, 64
    q, dk, dv, pool, bt, num_pages = _mq_case(5, dtype, lens, 1, n_q, n_kv, D)
    sl = np.array(lens, np.int32)
    for window in (0, 7):
        mq = O.decode_attention_mq(dtype, q, *pool, bt, sl, num_pages, n_kv, 0.2, window=window)
        single = O.decode_attention(dtype, q[:, 0], *pool, bt, sl, num_pages, n_kv, 0.2,
                                    window=window)
        np.testing.assert_array_equal(mq[:, 0], single)


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0, O.BF16, O.F32])
@pytest.mark.parametrize("window", [0, 5, 16, 33])
def test_each_query_is_single_query_attention_over_its_prefix(dtype, window):
    lens, q_len, n_q, n_kv, D = [8, 20, 47, 64], 6, 4, 2, 64
    q, dk, dv, pool, bt, num_pages = _mq_case(7, dtype, lens, q_len, n_q, n_kv, D)
    sl = np.array(lens, np.int32)
    mq = O.decode_attention_mq(dtype, q, *pool, bt, sl, num_pages, n_kv, 0.15, window=window)
    for j in range(q_len):
        prefix = sl - q_len + j + 1
        want = O.decode_attention(dtype, q[:, j], *pool, bt, prefix, num_pages, n_kv, 0.15,
                                  window=window)
        np.testing.assert_array_equal(mq[:, j], want)


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0])
def test_dense_causal_brute_force(dtype):
    lens, q_len, n_q, n_kv, D = [4, 19, 33], 4, 4, 2, 32
    q, dk, dv, pool, bt, num_pages = _mq_case(9, dtype, lens, q_len, n_q, n_kv, D)
    got = O.decode_attention_mq(dtype, q, *pool, bt, np.array(lens, np.int32), num_pages, n_kv,
                                0.3)
    G = n_q // n_kv
    for i, L in enumerate(lens):
        K = stored_values_dense(dtype, dk[i][0], dk[i][1])
        V = stored_values_dense(dtype, dv[i][0], dv[i][1])
        for j in range(q_len):
            P = L - q_len + j
            for g in range(n_q):
                h = g // G
                w = [math.exp(0.3 * math.fsum(float(a) * float(b) for a, b in zip(q[i, j, g], K[h, t])))
                     for t in range(P + 1)]
                den = math.fsum(w)
                want = [math.fsum(w[t] * V[h, t, d] for t in range(P + 1)) / den for d in range(D)]
                np.testing.assert_allclose(got[i, j, g], want, rtol=0, atol=1e-12)


def test_causality_later_tokens_do_not_matter():
    lens, q_len, n_q, n_kv, D = [30, 45], 5, 4, 2, 64
    q, dk, dv, (kd, vd, ks, vs), bt, num_pages = _mq_case(11, O.F16, lens, q_len, n_q, n_kv, D)
    sl = np.array(lens, np.int32)
    base = O.decode_attention_mq(O.F16, q, kd, vd, None, None, bt, sl, num_pages, n_kv, 0.2)
    for j in range(q_len):
        kd2, vd2 = kd.copy(), vd.copy()
        for i, L in enumerate(lens):  # NaN into every token after query j's position
            for t in range(L - q_len + j + 1, L):
                kd2[bt[i, t // 16], :, t % 16] = 0x7E00
                vd2[bt[i, t // 16], :, t % 16] = 0x7E00
        got = O.decode_attention_mq(O.F16, q, kd2, vd2, None, None, bt, sl, num_pages, n_kv, 0.2)
        np.testing.assert_array_equal(got[:, :j + 1], base[:, :j + 1])
        if j + 1 < q_len:
            assert np.isnan(got[:, j + 1:]).any()  # later queries do see the poisoned tokens


@pytest.mark.parametrize("dtype", [O.F16, O.Q8_0, O.BF16, O.F32])
def test_multi_token_append_is_sequential_appends(dtype):
    rng = np.random.default_rng(13)
    rows, q_len, n_kv, D, num_pages = 3, 5, 2, 64, 12
    lens = np.array([5, 20, 33], np.int32)  # the lengths after the step
    bt = rng.permutation(num_pages)[:9].reshape(rows, 3).astype(np.int32)
    q8 = dtype == O.Q8_0
    shape = (num_pages, n_kv, 16, D)
    kd = np.zeros(shape, np.int8 if q8 else np.float32 if dtype == O.F32 else np.uint16)
    ks = np.zeros((num_pages, n_kv, 16, D // 32), np.uint16) if q8 else None
    pools = [[kd.copy(), kd.copy(), None if ks is None else ks.copy(), None if ks is None else ks.copy()]
             for _ in range(2)]
    k_new = rng.standard_normal((rows, q_len, n_kv, D)).astype(np.float32)
    v_new = rng.standard_normal((rows, q_len, n_kv, D)).astype(np.float32)
    O.kv_append_mq(dtype, k_new, v_new, bt, lens, num_pages, *pools[0])
    for j in range(q_len):
        O.kv_append(dtype, k_new[:, j], v_new[:, j], bt, lens - q_len + j + 1, num_pages, *pools[1])
    for a, b in zip(*pools):
        if a is not None:
            np.testing.assert_array_equal(a, b)

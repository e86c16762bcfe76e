"""Several queries per row (Leone, "What ships": chunked prefill and exact
speculative verification; LeatEngine, "Capabilities": chunked prefill,
speculative decoding) on the GPU against the FP64 oracle, through the C ABI.

Reading: a row of L tokens whose last q_len are new has one query per new
token; query j sits at position P = L - q_len + j and attends causally to
[max(0, P + 1 - W), P + 1).  Checked for f16, q8_0 and bf16, GQA groups 1, 2
and 4, q_len from 1 up to several passes of the kernel, with and without a
window; with every slot no row holds poisoned with NaN (and, for the windowed
cases, every page wholly before the first query's window), through the fused
step (the q_len new tokens stored, bit-exact against the oracle's append,
then attended), at several chunk counts, and at the 8B shapes.  Bounds as in
the other attention tests: <= 2e-3 and <= 1e-4 * max(1, max|ref|)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (ATOL_STATED, BF16_NAN, F16_NAN, F32_NAN, device_pool, encode_pool,
                     host_arrays, tight_tol, to_dev)
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LENGTHS = [13, 17, 33, 100, 16, 250, 0, 31, 64, 14]  # none in (0, 13): every q_len fits


def _wl(dtype, n_q=16, n_kv=8, lengths=LENGTHS, seed=0):
    wl = W.draw("tiny", seed=seed, lengths=lengths)
    wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": dtype, "n_q_heads": n_q,
                         "n_kv_heads": n_kv})
    return wl


def _check(out, ref):
    assert np.all(np.isfinite(out)), "non-finite output: a poisoned slot was read"
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL_STATED, err
    assert err <= tight_tol(ref), err
    return err


def _poison(wl, host, positions_of_row):
    """NaN into the slots positions_of_row(i, L) of every row (f16/bf16/f32
    data, q8_0 scales)."""
    kd, vd, ks, vs = [None if a is None else a.copy() for a in host]
    nan = {W.F16: F16_NAN, W.BF16: BF16_NAN, W.F32: F32_NAN}.get(wl.cfg.dtype)
    for i, L in enumerate(wl.seq_lens):
        for t in positions_of_row(i, int(L)):
            page, slot = wl.block_table[i, t // W.PAGE], t % W.PAGE
            if nan is not None:
                kd[page, :, slot] = nan
                vd[page, :, slot] = nan
            else:
                ks[page, :, slot] = F16_NAN
                vs[page, :, slot] = F16_NAN
    return kd, vd, ks, vs


def _before_window(q_len, window):
    """Pages wholly before the first query's window [L - q_len + 1 - W, ...)."""
    def pos(i, L):
        if window <= 0 or L == 0:
            return []
        first_page = max(0, L - q_len + 1 - window) // W.PAGE
        return range(first_page * W.PAGE)
    return pos


def _oracle(wl, host, q, window=0, seq_lens=None):
    return O.decode_attention_mq(wl.cfg.dtype, q, *host, wl.block_table,
                                 wl.seq_lens if seq_lens is None else seq_lens, wl.num_pages,
                                 wl.cfg.n_kv_heads, wl.scale, window=window)


def _attend(wl, pool, q, num_chunks=0, seq_lens=None):
    sl = wl.seq_lens if seq_lens is None else seq_lens
    out = api.paged_decode_attention_mq(pool, 0, to_dev(q), to_dev(wl.block_table), to_dev(sl),
                                        wl.scale, num_chunks=num_chunks)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
@pytest.mark.parametrize("q_len", [1, 2, 3, 5, 8, 13])
@pytest.mark.parametrize("group", [1, 2, 4])
def test_mq_matches_oracle(dtype, q_len, group):
    wl = _wl(dtype, n_q=8 * group, n_kv=8)
    q, _, _ = W.mq_inputs(wl, q_len)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    out = _attend(wl, pool, q)
    assert pool.read_status() == 0
    _check(out, _oracle(wl, host, q))


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
@pytest.mark.parametrize("q_len,window", [(1, 1), (2, 1), (4, 5), (8, 16), (3, 17), (8, 40),
                                          (13, 100), (5, 1000)])
def test_mq_window_matches_oracle_and_skips_earlier_pages(dtype, q_len, window):
    wl = _wl(dtype, n_q=32, n_kv=8)
    q, _, _ = W.mq_inputs(wl, q_len, seed=1)
    host = encode_pool(wl)
    ref = _oracle(wl, host, q, window=window)  # from the unpoisoned pool
    pool = device_pool(wl, _poison(wl, host, _before_window(q_len, window)))
    pool.set_window(0, window)
    out = _attend(wl, pool, q)
    assert pool.read_status() == 0
    _check(out, ref)


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
@pytest.mark.parametrize("q_len", [2, 3, 6])  # G = 4: 8, 12 and 24 columns (each kernel)
def test_mq_split_invariance(dtype, q_len):
    wl = _wl(dtype, n_q=32, n_kv=8)
    q, _, _ = W.mq_inputs(wl, q_len, seed=2)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    ref = _oracle(wl, host, q)
    outs = [_attend(wl, pool, q, num_chunks=c) for c in (1, 3, 64, 1000)]
    for o in outs:
        _check(o, ref)
        assert float(np.max(np.abs(o - outs[0]))) <= 1e-6


@pytest.mark.parametrize("dtype,rows", [(W.F16, 1300), (W.F16, 2048), (W.BF16, 1000), (W.BF16, 1100)])
def test_mq_many_rows(dtype, rows):
    """32 columns with many short rows of mixed lengths (many pieces per CTA,
    whole and split).  The tensor-core kernel keeps its plan tables in shared
    memory beside its rings: f16 takes every row count the API allows (2048),
    bf16 (larger Q^T and P buffers) up to 1029 rows; calls of more rows take
    the team kernels.  Both sides of the bf16 limit."""
    lengths = [8 + (7 * i) % 29 for i in range(rows)]
    cfg = W.Config(**{**W.CONFIGS["tiny"].__dict__, "rows": rows, "n_q_heads": 32,
                      "dtype": dtype, "pool": ("spare", 0.10)})
    wl = W.draw(cfg, seed=3, lengths=lengths)
    q, _, _ = W.mq_inputs(wl, 8, seed=3)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    out = _attend(wl, pool, q)
    assert pool.read_status() == 0
    _check(out, _oracle(wl, host, q))


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
@pytest.mark.parametrize("q_len,window", [(1, 0), (4, 0), (7, 0), (8, 30)])
def test_mq_decode_step_appends_then_attends(dtype, q_len, window):
    """pkv_decode_step_mq: the q_len new tokens of every row land bit-exact
    where the oracle's append puts them (their slots start as NaN), and the
    queries attend over the pool that holds them."""
    wl = _wl(dtype, n_q=32, n_kv=8, lengths=[13, 17, 33, 100, 16, 250, 0, 31, 64, 8])
    q, k_new, v_new = W.mq_inputs(wl, q_len, seed=3)
    host = _poison(wl, encode_pool(wl), lambda i, L: range(max(0, L - q_len), L))
    want = [None if a is None else a.copy() for a in host]
    O.kv_append_mq(dtype, k_new, v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    pool = device_pool(wl, host)
    pool.set_window(0, window)
    out = api.decode_step_mq(pool, 0, to_dev(q), to_dev(k_new), to_dev(v_new),
                             to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    got = host_arrays(pool)
    for a, b in zip(got, want):
        if b is not None:
            np.testing.assert_array_equal(a, b)
    _check(out.cpu().numpy(), _oracle(wl, want, q, window=window))


def test_mq_q_len_one_equals_single_query_path():
    wl = W.draw("qwen3_0p6b_layer")
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    q1 = to_dev(wl.q)
    single = api.paged_decode_attention(pool, 0, q1, to_dev(wl.block_table),
                                        to_dev(wl.seq_lens), wl.scale)
    multi = api.paged_decode_attention_mq(pool, 0, q1[:, None].contiguous(),
                                          to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale)
    torch.cuda.synchronize()
    ref = O.decode_attention(W.F16, wl.q, *host, wl.block_table, wl.seq_lens, wl.num_pages,
                             wl.cfg.n_kv_heads, wl.scale)
    _check(single.cpu().numpy(), ref)
    _check(multi[:, 0].cpu().numpy(), ref)


def test_mq_short_row_reports_bad_length():
    """A row with fewer tokens than queries: zeros and PKV_DEV_BAD_LENGTH;
    the other rows are unaffected."""
    wl = _wl(W.F16, n_q=32, n_kv=8, lengths=[13, 17, 1, 100, 0, 3, 4])
    q_len = 4
    lens = wl.seq_lens.copy()
    q, _, _ = W.mq_inputs(wl, q_len)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    out = _attend(wl, pool, q)
    assert pool.read_status() == 2  # PKV_DEV_BAD_LENGTH
    bad = [2, 5]  # L = 1 and 3 < q_len
    assert np.all(out[bad] == 0)
    lens[bad] = 0
    _check(out, _oracle(wl, host, q, seq_lens=lens))  # zeros where the oracle has zeros


@pytest.mark.parametrize("cfg_name,q_len", [("llama8b_f16", 4), ("llama8b_bf16", 3),
                                            ("llama8b_q8_0", 2), ("llama8b_f32", 5)])
def test_mq_full_size(cfg_name, q_len):
    """The 8B shapes: every row of f16 and bf16, every fourth row of q8_0."""
    wl = W.draw(cfg_name)
    q, k_new, v_new = W.mq_inputs(wl, q_len)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    out = _attend(wl, pool, q)
    assert pool.read_status() == 0
    rows = np.arange(0, wl.rows, 4 if wl.cfg.dtype == W.Q8_0 else 1)
    ref = O.decode_attention_mq(wl.cfg.dtype, q[rows], *host, wl.block_table[rows],
                                wl.seq_lens[rows], wl.num_pages, wl.cfg.n_kv_heads, wl.scale)
    _check(out[rows], ref)


def test_mq_validation():
    wl = _wl(W.F16, n_q=16, n_kv=8)
    pool = device_pool(wl, encode_pool(wl))
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    for q_len in (0, 65):
        q = torch.zeros((wl.rows, max(q_len, 1), 16, 128), device="cuda")
        if q_len == 0:
            q = q[:, :0]
        with pytest.raises((api.PkvError, ValueError)):
            api.paged_decode_attention_mq(pool, 0, q.contiguous(), bt, sl, wl.scale)
    with pytest.raises(ValueError):  # 3-D q
        api.paged_decode_attention_mq(pool, 0, torch.zeros((wl.rows, 16, 128), device="cuda"),
                                      bt, sl, wl.scale)


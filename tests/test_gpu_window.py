"""Sliding-window decode (LeatEngine, "Capabilities": sliding-window KV caches) on
the GPU against the FP64 oracle, through the C ABI.

Reading: with window W a row of L tokens attends to [max(0, L - W), L), and
the kernel reads only the pages that hold those tokens.  Checked for f16 and
q8_0 at windows that start mid-page, on a page boundary, span one token and
exceed the row; with the pages wholly before each row's window poisoned with
NaN (a read of one would show); through the fused decode step; through the
two-launch split + combine; and the plan against the oracle's.  Bounds as in
the other attention tests: <= 2e-3 and <= 1e-4 * max(1, max|ref|)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (ATOL_STATED, F16_NAN, device_pool, encode_pool, oracle_decode, split_aligned,
                     tight_tol, to_dev)
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

WINDOWS = [1, 16, 17, 100, 1000, 4096]


def _check(out, ref):
    assert np.all(np.isfinite(out)), "non-finite output: a poisoned slot was read"
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL_STATED, err
    assert err <= tight_tol(ref), err
    return err


def _poison_before_window(wl, host, window):
    """NaN into every page of a row that lies wholly before its window (f16
    data or q8_0 scales): those pages must not be read."""
    kd, vd, ks, vs = [None if a is None else a.copy() for a in host]
    for i, L in enumerate(wl.seq_lens):
        first = max(0, int(L) - window) // W.PAGE
        for p in range(first):
            page = wl.block_table[i, p]
            if wl.cfg.dtype == W.F16:
                kd[page] = F16_NAN
                vd[page] = F16_NAN
            else:
                ks[page] = F16_NAN
                vs[page] = F16_NAN
    return kd, vd, ks, vs


def _attend(wl, pool, layer=0, num_chunks=0):
    out = api.paged_decode_attention(pool, layer, to_dev(wl.q), to_dev(wl.block_table),
                                     to_dev(wl.seq_lens), wl.scale, num_chunks=num_chunks)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("window", WINDOWS)
def test_window_f16_matches_oracle_and_skips_earlier_pages(window):
    wl = W.draw("llama8b_f16")
    host = encode_pool(wl)
    ref = oracle_decode(wl, host, window=window)  # from the unpoisoned pool
    pool = device_pool(wl, _poison_before_window(wl, host, window))
    pool.set_window(0, window)
    assert pool.window(0) == window
    _check(_attend(wl, pool), ref)


@pytest.mark.parametrize("window", [17, 1000])
def test_window_q8_0_matches_oracle_and_skips_earlier_pages(window):
    wl = W.draw("llama8b_q8_0")
    host = encode_pool(wl)
    pool = device_pool(wl, _poison_before_window(wl, host, window))
    pool.set_window(0, window)
    out = _attend(wl, pool)
    rows = np.arange(0, wl.rows, 4)
    ref = O.decode_attention(W.Q8_0, wl.q[rows], *host, wl.block_table[rows], wl.seq_lens[rows],
                             wl.num_pages, wl.cfg.n_kv_heads, wl.scale, window=window)
    _check(out[rows], ref)


@pytest.mark.parametrize("cfg_name", ["tiny", "qwen3_0p6b_layer"])
def test_window_per_layer(cfg_name):
    """Each layer keeps its own window; a layer without one attends to all."""
    wl = W.draw(cfg_name)
    host = encode_pool(wl)
    pool = device_pool(wl, host, num_layers=2, layer=1)
    pool.set_window(0, 33)  # another layer's window does not apply to layer 1
    _check(_attend(wl, pool, layer=1), oracle_decode(wl, host))
    pool.set_window(1, 20)
    _check(_attend(wl, pool, layer=1), oracle_decode(wl, host, window=20))


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
def test_window_split_invariance(dtype):
    """Windows starting mid-page, rows shorter than the window, an empty row."""
    wl = W.draw("tiny", lengths=[1, 17, 33, 100, 16, 250, 0, 31])
    wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": dtype})
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    pool.set_window(0, 40)
    ref = oracle_decode(wl, host, window=40)
    outs = [_attend(wl, pool, num_chunks=c) for c in (1, 3, 64, 1000)]
    for o in outs:
        _check(o, ref)
        assert float(np.max(np.abs(o - outs[0]))) <= 1e-6


def test_window_decode_step_appends_then_attends():
    """pkv_decode_step with a window: the new token lands in the last page
    (always inside the window) and attention covers the last W tokens."""
    wl = W.draw("skewed")
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host)
    pool.set_window(0, 300)
    out = api.decode_step(pool, 0, to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new),
                          to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(W.F16, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    _check(out.cpu().numpy(), oracle_decode(wl, want, window=300))


def test_window_split_combine_and_plan():
    wl = W.draw("llama8b_f16")
    cfg = wl.cfg
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    window = 777
    pool.set_window(0, window)
    chunks = 50
    ws = api.Workspace(pool, cfg.n_q_heads, wl.rows, chunks)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    out = torch.full_like(q, float("nan"))
    api.paged_decode_split(pool, 0, q, bt, sl, wl.scale, out, ws)
    api.paged_decode_combine(sl, cfg.n_q_heads, cfg.n_kv_heads, wl.bt_stride, chunks, ws.tensor,
                             out, window=window, kv_dtype=pool.dtype)
    torch.cuda.synchronize()
    _check(out.cpu().numpy(), oracle_decode(wl, host, window=window))
    rps, first, last = api.paged_decode_plan(sl, cfg.n_kv_heads, wl.bt_stride, chunks,
                                             window=window, kv_dtype=pool.dtype)
    o_rps, o_first, o_last, _ = O.plan(wl.seq_lens, cfg.n_kv_heads, chunks, window=window,
                                       aligned=split_aligned(pool.dtype))
    np.testing.assert_array_equal(rps.cpu().numpy(), o_rps)
    np.testing.assert_array_equal(first.cpu().numpy(), o_first)
    np.testing.assert_array_equal(last.cpu().numpy(), o_last)


def test_window_validation():
    wl = W.draw("tiny")
    pool = api.KVPool(2, wl.num_pages, wl.cfg.n_kv_heads, wl.cfg.dtype)
    with pytest.raises(api.PkvError):
        pool.set_window(0, -1)
    with pytest.raises(api.PkvError):
        pool.set_window(2, 16)
    assert pool.window(1) == 0

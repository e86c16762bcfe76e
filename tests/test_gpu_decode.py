"""paged_decode_attention (and the fused decode step) on the GPU against the
FP64 oracle, through the C ABI.

Every workload shape (tiny, Qwen3-0.6B layer, 8B f16, 8B q8_0, skewed batch)
runs at its full size, and the oracle checks every output.  Unused pool slots are poisoned with NaN,
so any read outside a row's tokens shows up.  Bounds: max abs error <= 2e-3
(the stated bound) and <= 1e-4 * max(1, max|ref|) (internal)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (ATOL_STATED, device_pool, encode_pool, host_arrays, oracle_decode,
                     tight_tol, to_dev)
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu


_HOST_POOLS = {}


def _host_pool(wl, include_appended=True):
    """encode_pool of a full-size workload, kept for the module's other tests
    (encoding the 8B q8_0 pool takes a while; the arrays are only read)."""
    key = (wl.cfg.name, include_appended)
    if key not in _HOST_POOLS:
        _HOST_POOLS[key] = encode_pool(wl, include_appended=include_appended)
    return _HOST_POOLS[key]


def _check(out, ref):
    assert np.all(np.isfinite(out)), "non-finite output: a poisoned slot was read"
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL_STATED, err
    assert err <= tight_tol(ref), err
    return err


def _run(wl, pool, layer=0, num_chunks=0, q=None, seq_lens=None):
    q = wl.q if q is None else q
    sl = wl.seq_lens if seq_lens is None else seq_lens
    out = api.paged_decode_attention(pool, layer, to_dev(q), to_dev(wl.block_table), to_dev(sl),
                                     wl.scale, num_chunks=num_chunks)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("cfg_name", ["tiny", "qwen3_0p6b_layer", "llama8b_f16", "llama8b_bf16",
                                      "llama8b_f32"])
def test_attention_matches_oracle(cfg_name):
    wl = W.draw(cfg_name)
    host = encode_pool(wl)
    pool = device_pool(wl, host, num_layers=2, layer=1)
    ref = oracle_decode(wl, host)
    _check(_run(wl, pool, layer=1), ref)


def test_attention_q8_0_full_batch_every_row():
    """The 8B q8_0 batch at full size (32 rows up to 32768 tokens) in the
    launch configuration the benchmark times; the oracle checks every row."""
    wl = W.draw("llama8b_q8_0")
    host = _host_pool(wl)
    pool = device_pool(wl, host)
    out = _run(wl, pool)
    _check(out, oracle_decode(wl, host))


@pytest.mark.parametrize("cfg_name", ["llama8b_f16", "llama8b_q8_0"])
def test_benchmarked_decode_step(cfg_name):
    """The call the benchmark times: pkv_decode_step on the full 8B batch at
    the default chunk count, the new token of every row stored by the fused
    append.  The pool must then equal the oracle's append bit for bit, and the
    output must match the oracle's attention over it."""
    wl = W.draw(cfg_name)
    host = _host_pool(wl, include_appended=False)
    pool = device_pool(wl, host)
    out = api.decode_step(pool, 0, to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new),
                          to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(wl.cfg.dtype, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages,
                *want)
    got = host_arrays(pool, 0)
    for g, w in zip(got, want):
        if w is not None:
            assert np.array_equal(g, w), "fused append differs from the oracle's encoding"
    _check(out.cpu().numpy(), oracle_decode(wl, want))


def test_skewed_decode_step_appends_then_attends():
    """64 rows, one at 40960 tokens: pkv_decode_step appends each row's new
    token and attends over lengths that include it."""
    wl = W.draw("skewed")
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host)
    out = api.decode_step(pool, 0, to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new),
                          to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(W.F16, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    _check(out.cpu().numpy(), oracle_decode(wl, want))


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
def test_split_invariance(dtype):
    """Any chunk count gives the same output: 1 chunk (no merge), many chunks
    (every (row, head) split, one page per piece at the extreme)."""
    wl = W.draw("tiny", lengths=[1, 17, 33, 100, 16, 250, 0, 31])
    wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": dtype})
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    ref = oracle_decode(wl, host)
    outs = [_run(wl, pool, num_chunks=c) for c in (1, 2, 7, 64, 455, 4000, 0)]
    for o in outs:
        _check(o, ref)
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-6)
    assert np.all(outs[0][6] == 0)  # the empty row


@pytest.mark.parametrize("group,n_kv", [(1, 4), (2, 8), (4, 8), (4, 2)])
@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
def test_gqa_groups(group, n_kv, dtype):
    cfg = W.Config("gqa", 5, ("uniform", 1, 300), n_kv * group, n_kv, 128, dtype,
                   ("spare", 0.3), 40 + group)
    wl = W.draw(cfg)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    _check(_run(wl, pool, num_chunks=37), oracle_decode(wl, host))


@pytest.mark.parametrize("cfg_name", ["llama8b_f16", "llama8b_f32", "llama8b_bf16",
                                      "llama8b_q8_0"])
def test_peaked_scores(cfg_name):
    """q scaled by 8: near one-hot softmax, so one wrong key or value would
    dominate the output."""
    wl = W.draw(cfg_name)
    host = _host_pool(wl)
    pool = device_pool(wl, host)
    q = (wl.q * 8).astype(np.float32)
    _check(_run(wl, pool, q=q), oracle_decode(wl, host, q=q))


def test_single_token_rows_return_v():
    wl = W.draw("tiny", lengths=[1, 1, 1])
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    out = _run(wl, pool, num_chunks=5)
    ref = oracle_decode(wl, host)
    np.testing.assert_array_equal(out.astype(np.float64), ref)  # softmax of one token is 1


def test_out_of_range_lengths_and_pages_are_flagged_not_read():
    wl = W.draw("tiny")
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    sl = wl.seq_lens.copy()
    sl[2] = wl.bt_stride * 16 + 40     # beyond the block table: clamped
    bt = wl.block_table.copy()
    bt[3, 2] = -7                       # outside the pool: page 0 read instead
    out = api.paged_decode_attention(pool, 0, to_dev(wl.q), to_dev(bt), to_dev(sl), wl.scale)
    torch.cuda.synchronize()
    st = pool.read_status()
    assert st & api.DEV_BAD_LENGTH and st & api.DEV_BAD_PAGE
    assert out.shape == wl.q.shape


def test_host_validation_errors():
    wl = W.draw("tiny")
    pool = api.KVPool(1, wl.num_pages, 8, W.F16)
    q = to_dev(wl.q)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    ws = api.Workspace(pool, 16, 4)
    with pytest.raises(api.PkvError) as e:   # GQA group 3
        api.paged_decode_attention(pool, 0, torch.zeros(4, 24, 128, device="cuda"), bt, sl, 0.1)
    assert e.value.status == 2
    small = api.Workspace(pool, 16, 4)
    small.nbytes = 256
    with pytest.raises(api.PkvError) as e:
        api.paged_decode_attention(pool, 0, q, bt, sl, 0.1, workspace=small)
    assert e.value.status == 4
    out = api.paged_decode_attention(pool, 0, q, bt, sl, 0.1, workspace=ws)
    assert out.shape == q.shape


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
def test_fused_step_append_is_bit_exact(dtype):
    """pkv_decode_step stores each row's token inside the attention kernel:
    the pool afterwards must equal the oracle's append byte for byte."""
    from helpers import host_arrays
    wl = W.draw("skewed")
    wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": dtype})
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host, num_layers=2, layer=1)
    out = api.decode_step(pool, 1, to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new),
                          to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale, num_chunks=333)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(dtype, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    for g, w in zip(host_arrays(pool, 1), want):
        if w is not None:
            np.testing.assert_array_equal(g, w)
    rows = np.arange(0, wl.rows, 7)
    ref = O.decode_attention(dtype, wl.q[rows], *want, wl.block_table[rows], wl.seq_lens[rows],
                             wl.num_pages, wl.cfg.n_kv_heads, wl.scale)
    _check(out.cpu().numpy()[rows], ref)


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
def test_split_then_combine_equals_merged(dtype):
    wl = W.draw("llama8b_f16")
    wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": dtype})
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    merged = api.paged_decode_attention(pool, 0, q, bt, sl, wl.scale).cpu().numpy()
    ws = api.Workspace(pool, wl.cfg.n_q_heads, wl.rows)
    out = torch.full_like(q, float("nan"))
    api.paged_decode_split(pool, 0, q, bt, sl, wl.scale, out, ws)
    api.paged_decode_combine(sl, wl.cfg.n_q_heads, wl.cfg.n_kv_heads, wl.bt_stride,
                             ws.num_chunks, ws.tensor, out, kv_dtype=pool.dtype)
    torch.cuda.synchronize()
    # the two merges batch the pieces differently: same sums, other rounding order
    np.testing.assert_allclose(out.cpu().numpy(), merged, rtol=0, atol=1e-6)
    _check(merged, oracle_decode(wl, host))


def test_workspace_reuse_across_calls_and_shapes():
    """The arrival counters return to zero after every call: one workspace
    serves many calls, with different batches and chunk splits."""
    wl = W.draw("qwen3_0p6b_layer")
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    ws = api.Workspace(pool, wl.cfg.n_q_heads, wl.rows, 97)
    ref = oracle_decode(wl, host)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    for rep in range(3):
        out = api.paged_decode_attention(pool, 0, q, bt, sl, wl.scale, workspace=ws)
        _check(out.cpu().numpy(), ref)
        sub = api.paged_decode_attention(pool, 0, q[:3].contiguous(), bt[:3].contiguous(),
                                         sl[:3].contiguous(), wl.scale, workspace=ws)
        _check(sub.cpu().numpy(), ref[:3])
    assert _flags_clear(ws, wl.rows)


def _flags_clear(ws, max_rows, n_kv=8):
    """The merge's flags (down from the end of the workspace) are all zero."""
    slots = ws.num_chunks + max_rows * n_kv
    up = (slots * 8 + 255) // 256 * 256
    return int(ws.tensor[ws.nbytes - up:ws.nbytes].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("chunks", [456, 97])
def test_workspace_reuse_across_batch_sizes(chunks):
    """A workspace sized for the largest batch serves batches of every size in
    any order, as in continuous batching: rows come and go between steps.  A
    small call's partial states must not be read as a later large call's
    arrival counters or ready flags."""
    wl = W.draw("skewed")
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    ws = api.Workspace(pool, wl.cfg.n_q_heads, wl.rows, chunks)
    ref = oracle_decode(wl, host)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    for rows in (64, 4, 64, 17, 64, 1, 40, 64):
        out = api.paged_decode_attention(pool, 0, q[:rows].contiguous(), bt[:rows].contiguous(),
                                         sl[:rows].contiguous(), wl.scale, workspace=ws,
                                         num_chunks=chunks)
        torch.cuda.synchronize()
        _check(out.cpu().numpy(), ref[:rows])
    assert pool.read_status() == 0
    assert _flags_clear(ws, wl.rows)

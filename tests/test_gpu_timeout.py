"""The attention kernels' give-up path on a real GPU, without a hang or a fault.

Every wait of a kernel on a tile copy is bounded: when it runs out, the CTA
stops reading, records PKV_DEV_TIMEOUT in the pool's status word, waits for
the copies it still has in flight (they do land) and returns.  The limit of
those waits is a pool setting (kv_pool_set_wait_limit); at 0 a warp gives up
at the first copy that has not landed when it looks.  With one chunk, one CTA
streams thousands of tiles through rings of two stages per warp, so a warp
soon waits for a copy issued a few hundred nanoseconds earlier: the wait gives
up.  The tests check that the status bit is set, that the call returns, and
that the same context then computes the right result with the default limit
and a zeroed workspace.  No wait here is left without an end: the copies are
real and complete, and the drain keeps the default limit."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import ATOL_STATED, device_pool, encode_pool, oracle_decode, tight_tol, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _workload(dtype, lengths=(4096, 300)):
    cfg = W.Config("timeout", len(lengths), ("fixed", tuple(lengths)), 32, 8, 128, dtype,
                   ("spare", 0.1), 11)
    return W.draw(cfg)


def _check(out, ref):
    assert np.all(np.isfinite(out))
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL_STATED and err <= tight_tol(ref), err


@pytest.mark.parametrize("chunks", [1, 0])
@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0])
def test_single_query_wait_gives_up_then_recovers(dtype, chunks):
    wl = _workload(dtype)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    ws = api.Workspace(pool, wl.cfg.n_q_heads, wl.rows, chunks)
    pool.set_wait_limit(0)
    api.paged_decode_attention(pool, 0, q, bt, sl, wl.scale, workspace=ws, num_chunks=chunks)
    torch.cuda.synchronize()  # the call returned: no wait was left hanging
    assert pool.read_status() & api.DEV_TIMEOUT
    # the context is intact: default limit, zeroed workspace, right answer
    pool.set_wait_limit(api.DEFAULT_WAIT_NS)
    ws.tensor.zero_()
    out = api.paged_decode_attention(pool, 0, q, bt, sl, wl.scale, workspace=ws, num_chunks=chunks)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    _check(out.cpu().numpy(), oracle_decode(wl, host))


@pytest.mark.parametrize("dtype,q_len", [(W.F16, 2), (W.F16, 4), (W.F16, 8), (W.Q8_0, 2),
                                         (W.Q8_0, 4), (W.BF16, 4), (W.F32, 2)])
def test_several_query_wait_gives_up_then_recovers(dtype, q_len):
    """q_len 2 runs the kernel whose warps read their own pages; wider steps run
    the kernels whose warps share every page (full and empty barriers)."""
    wl = _workload(dtype)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    q_np = W.mq_inputs(wl, q_len)[0]
    q, bt, sl = to_dev(q_np), to_dev(wl.block_table), to_dev(wl.seq_lens)
    ws = api.WorkspaceMQ(pool, wl.cfg.n_q_heads, wl.rows, q_len, 1)
    pool.set_wait_limit(0)
    api.paged_decode_attention_mq(pool, 0, q, bt, sl, wl.scale, workspace=ws, num_chunks=1)
    torch.cuda.synchronize()
    assert pool.read_status() & api.DEV_TIMEOUT
    pool.set_wait_limit(api.DEFAULT_WAIT_NS)
    ws.tensor.zero_()
    out = api.paged_decode_attention_mq(pool, 0, q, bt, sl, wl.scale, workspace=ws, num_chunks=1)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    ref = O.decode_attention_mq(dtype, q_np, *host, wl.block_table, wl.seq_lens, wl.num_pages,
                                wl.cfg.n_kv_heads, wl.scale)
    _check(out.cpu().numpy(), ref)


def test_fused_step_wait_gives_up_without_touching_other_layers():
    """The fused step with the 0 limit on the 8B f16 batch at the default chunk
    count (many CTAs, segments split over chunks): the status bit is set, and
    another layer of the pool keeps its contents."""
    wl = W.draw("llama8b_f16")
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host, num_layers=2, layer=1)
    before = pool.k_data[0].clone()
    args = (to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new), to_dev(wl.block_table),
            to_dev(wl.seq_lens), wl.scale)
    ws = api.Workspace(pool, wl.cfg.n_q_heads, wl.rows)
    pool.set_wait_limit(0)
    api.decode_step(pool, 1, *args, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() & api.DEV_TIMEOUT
    assert torch.equal(pool.k_data[0].view(torch.int16), before.view(torch.int16))
    pool.set_wait_limit(api.DEFAULT_WAIT_NS)
    ws.tensor.zero_()
    # the step again with the default limit: it stores the same new tokens
    # (whether or not the first call got to them) and attends
    out = api.decode_step(pool, 1, *args, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(W.F16, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    _check(out.cpu().numpy(), oracle_decode(wl, want))

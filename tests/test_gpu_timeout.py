"""The attention kernels' give-up path on a real GPU, without a hang or a fault.

Every wait of a kernel on a shared-memory barrier is bounded: when one runs
out, the CTA stops reading, records PKV_DEV_TIMEOUT in the pool's status
word, waits for the copies it still has in flight (they do land) and
returns.  The pool's test hook (kv_pool_set_test_stall) makes each warp,
once it has queued its first tile copies, wait a few microseconds on a
barrier that nothing completes: that wait runs out every time, as a wait on
a copy that never lands would, and the kernel takes the same path.

The calls run the full 8B batches at the default chunk count (every CTA with
copies in flight when it gives up, segments split over chunks) through every
attention kernel: one query per row, and several queries per row with warps
reading their own pages or sharing them.  The tests check that the status bit
is set, that the call returns, and that the same context then computes the
oracle's result with the hook off and a zeroed workspace."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import ATOL_STATED, device_pool, encode_pool, oracle_decode, tight_tol, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STALL_NS = 2000  # how long each warp waits on the barrier nothing completes

_HOST = {}


def _setup(name, include_appended=True):
    """The full-size workload, its oracle-encoded pool (kept for the module's
    other tests; only read) and a device pool holding it."""
    wl = W.draw(name)
    key = (name, include_appended)
    if key not in _HOST:
        _HOST[key] = encode_pool(wl, include_appended=include_appended)
    host = _HOST[key]
    return wl, host, device_pool(wl, host)


def _check(out, ref):
    assert np.all(np.isfinite(out))
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL_STATED and err <= tight_tol(ref), err


def _rows(wl, n=3):
    """The longest rows (the oracle checks these after recovery)."""
    return np.sort(np.argsort(wl.seq_lens)[::-1][:n])


@pytest.mark.parametrize("name", ["llama8b_f16", "llama8b_q8_0", "llama8b_bf16", "llama8b_f32"])
def test_single_query_wait_gives_up_then_recovers(name):
    wl, host, pool = _setup(name)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    ws = api.Workspace(pool, wl.cfg.n_q_heads, wl.rows)
    pool.set_test_stall(STALL_NS)
    api.paged_decode_attention(pool, 0, q, bt, sl, wl.scale, workspace=ws)
    torch.cuda.synchronize()  # the call returned: no wait was left hanging
    assert pool.read_status() & api.DEV_TIMEOUT
    # the context is intact: default limit, zeroed workspace, right answer
    pool.set_test_stall(0)
    ws.tensor.zero_()
    out = api.paged_decode_attention(pool, 0, q, bt, sl, wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    r = _rows(wl)
    ref = O.decode_attention(wl.cfg.dtype, wl.q[r], *host, wl.block_table[r], wl.seq_lens[r],
                             wl.num_pages, wl.cfg.n_kv_heads, wl.scale)
    _check(out.cpu().numpy()[r], ref)


@pytest.mark.parametrize("name,q_len", [("llama8b_f16", 2), ("llama8b_f16", 4), ("llama8b_f16", 8),
                                        ("llama8b_q8_0", 2), ("llama8b_q8_0", 4),
                                        ("llama8b_bf16", 4), ("llama8b_f32", 2)])
def test_several_query_wait_gives_up_then_recovers(name, q_len):
    """q_len 2 runs the kernel whose warps read their own pages; wider steps run
    the kernels whose warps share every page (full and empty barriers)."""
    wl, host, pool = _setup(name)
    q_np = W.mq_inputs(wl, q_len)[0]
    q, bt, sl = to_dev(q_np), to_dev(wl.block_table), to_dev(wl.seq_lens)
    ws = api.WorkspaceMQ(pool, wl.cfg.n_q_heads, wl.rows, q_len)
    pool.set_test_stall(STALL_NS)
    api.paged_decode_attention_mq(pool, 0, q, bt, sl, wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() & api.DEV_TIMEOUT
    pool.set_test_stall(0)
    ws.tensor.zero_()
    out = api.paged_decode_attention_mq(pool, 0, q, bt, sl, wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    r = _rows(wl, 2)
    ref = O.decode_attention_mq(wl.cfg.dtype, q_np[r], *host, wl.block_table[r], wl.seq_lens[r],
                                wl.num_pages, wl.cfg.n_kv_heads, wl.scale)
    _check(out.cpu().numpy()[r], ref)


def test_fused_step_wait_gives_up_without_touching_other_layers():
    """The fused step with the 0 limit: the status bit is set, and another
    layer of the pool keeps its contents."""
    wl = W.draw("llama8b_f16")
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host, num_layers=2, layer=1)
    before = pool.k_data[0].clone()
    args = (to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new), to_dev(wl.block_table),
            to_dev(wl.seq_lens), wl.scale)
    ws = api.Workspace(pool, wl.cfg.n_q_heads, wl.rows)
    pool.set_test_stall(STALL_NS)
    api.decode_step(pool, 1, *args, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() & api.DEV_TIMEOUT
    assert torch.equal(pool.k_data[0].view(torch.int16), before.view(torch.int16))
    pool.set_test_stall(0)
    ws.tensor.zero_()
    # the step again with the default limit: it stores the same new tokens
    # (whether or not the first call got to them) and attends
    out = api.decode_step(pool, 1, *args, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(W.F16, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    _check(out.cpu().numpy(), oracle_decode(wl, want))

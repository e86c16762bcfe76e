"""The segment-aligned work split on the GPU, in cases chosen (with the oracle's
plan) so that it differs from the uniform split and holds both kinds of chunk:
parts of long rows' segments, and several whole segments of a short row; some
launched CTAs get no chunk.  For f16 and bf16 KV (the formats that take it):
the device plan equals the oracle's bit for bit, the fused step (append, then
attention merged in-kernel) and the two-launch form (split, combine) match the
FP64 oracle within <= 2e-3 and <= 1e-4 * max(1, max|ref|), and the fused
step's pool equals the oracle's append bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import ATOL_STATED, device_pool, encode_pool, host_arrays, tight_tol, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [  # (lengths, chunks): 8 KV heads, 32 query heads
    ([1500, 70, 30, 2900, 5, 400, 16, 17, 800, 33], 121),
    ([4000, 9, 9, 9, 9, 9, 9, 9, 2500, 120], 113),
    ([3000, 500, 48, 1, 2048, 1024], 57),
]


def _workload(lengths, dtype):
    base = W.CONFIGS["llama8b_f16"]
    cfg = W.Config(**{**base.__dict__, "name": "aligned_case", "rows": len(lengths),
                      "lengths": ("fixed", tuple(lengths)), "dtype": dtype})
    return W.draw(cfg, lengths=lengths)


def _check(out, ref):
    assert np.all(np.isfinite(out))
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL_STATED, err
    assert err <= tight_tol(ref), err


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_aligned_split_step_and_plan(case, dtype):
    lengths, chunks = CASES[case]
    wl = _workload(lengths, dtype)
    cfg = wl.cfg
    # the case exercises the aligned split: it differs from the uniform one,
    # some chunk holds several whole segments and some segment spans chunks
    lo, hi = O.chunk_ranges(wl.seq_lens, cfg.n_kv_heads, chunks, aligned=True)
    ulo, _ = O.chunk_ranges(wl.seq_lens, cfg.n_kv_heads, chunks, aligned=False)
    assert len(lo) != len(ulo) or not np.array_equal(lo, ulo)
    o_rps, o_first, o_last, _ = O.plan(wl.seq_lens, cfg.n_kv_heads, chunks, aligned=True)
    assert np.any(o_first != o_last)

    sl, bt = to_dev(wl.seq_lens), to_dev(wl.block_table)
    rps, first, last = api.paged_decode_plan(sl, cfg.n_kv_heads, wl.bt_stride, chunks,
                                             kv_dtype=dtype)
    np.testing.assert_array_equal(rps.cpu().numpy(), o_rps)
    np.testing.assert_array_equal(first.cpu().numpy(), o_first)
    np.testing.assert_array_equal(last.cpu().numpy(), o_last)

    # fused step with the appended tokens, merged in-kernel
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host)
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(dtype, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    ref = O.decode_attention(dtype, wl.q, *want, wl.block_table, wl.seq_lens, wl.num_pages,
                             cfg.n_kv_heads, wl.scale)
    ws = api.Workspace(pool, cfg.n_q_heads, wl.rows, chunks)
    out = api.decode_step(pool, 0, to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new), bt, sl,
                          wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    for g, w in zip(host_arrays(pool), want):
        if w is not None:
            np.testing.assert_array_equal(g, w)
    _check(out.cpu().numpy(), ref)

    # the two-launch form on the same pool (the tokens are stored now)
    out2 = torch.full_like(out, float("nan"))
    api.paged_decode_split(pool, 0, to_dev(wl.q), bt, sl, wl.scale, out2, ws)
    api.paged_decode_combine(sl, cfg.n_q_heads, cfg.n_kv_heads, wl.bt_stride, chunks, ws.tensor,
                             out2, kv_dtype=dtype)
    torch.cuda.synchronize()
    _check(out2.cpu().numpy(), ref)

"""paged_decode_attention_static: the decode entry point for callers that
cannot allocate device memory while decoding (a server whose memory is all
reserved up front by its KV pool and caching allocator, or code where a
cudaMalloc is not allowed or would stall the device).  Its scratch is a
fixed array inside the library.

Checked through the C ABI against paged_decode_attention with a caller
workspace, on two calls in a row, with the tolerance of the split-invariance
tests; and the size limit is checked to fail with a clear error.  This file is
collected last so that a run stopping at its first failure has already run
every other test; it needs nothing from them."""
import ctypes

import numpy as np
import pytest
import torch

from helpers import device_pool, encode_pool, oracle_decode, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 1e-6  # as between chunk splits of the same call


def _static_fn():
    f = api.lib().paged_decode_attention_static
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, i, vp, vp, i, vp, i, i, ctypes.c_float, vp, i, vp]
    f.restype = i
    return f


def _call_static(pool, q, bt, sl, n_q, scale, out, chunks=0):
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return _static_fn()(pool.handle, 0, P(q), P(bt), bt.shape[1], P(sl), sl.shape[0], n_q,
                        ctypes.c_float(scale), P(out), chunks,
                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("cfg_name", ["llama8b_f16", "skewed", "llama8b_q8_0"])
def test_static_scratch_matches_workspace_entry_point(cfg_name):
    wl = W.draw(cfg_name)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    ref = api.paged_decode_attention(pool, 0, q, bt, sl, wl.scale).cpu().numpy()
    for call in range(2):  # two calls in a row share the array
        out = torch.full_like(q, float("nan"))
        st = _call_static(pool, q, bt, sl, wl.cfg.n_q_heads, wl.scale, out)
        assert st == 0, api.lib().pkv_last_error_message().decode()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - ref))) <= TOL, f"call {call}"
    assert pool.read_status() == 0
    if cfg_name == "llama8b_f16":  # and the result is the attention itself
        assert float(np.max(np.abs(ref - oracle_decode(wl, host)))) <= 2e-3


def test_static_scratch_rejects_calls_that_do_not_fit():
    wl = W.draw("llama8b_f16")
    pool = api.KVPool(1, wl.num_pages, 8, W.F16)
    rows = 1000  # 1000 rows x 8 KV heads of partial slots need ~17 MiB > 8 MiB
    q = torch.zeros(rows, 32, 128, device="cuda")
    bt = torch.zeros(rows, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(rows, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    st = _call_static(pool, q, bt, sl, 32, 0.1, out, chunks=304)
    assert st == 4  # PKV_ERR_WORKSPACE
    assert b"static array" in api.lib().pkv_last_error_message()


def _scratch_bytes():
    """PKV_STATIC_SCRATCH_BYTES as include/pkv.h defines it."""
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "pkv.h")).read()
    m = re.search(r"#define PKV_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    return int(m.group(1)) << int(m.group(2))


def _largest_fitting_rows(pool, n_q):
    """The most rows whose workspace, at the default chunk count for that
    many rows, fits the static array."""
    best = 0
    for rows in range(1, api.MAX_ROWS + 1):
        need = api.workspace_bytes(rows, n_q, pool.n_kv, api.default_chunks(pool, n_q, rows))
        if need > _scratch_bytes():
            break
        best = rows
    return best


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0])
def test_static_scratch_size_limit_is_exact(dtype):
    """At the largest row count that fits, the call succeeds and matches the
    workspace entry point; with one row more it is refused."""
    cfg = W.Config("limit", 1, ("fixed", (1,)), 32, 8, 128, dtype, ("spare", 0.1), 21)
    probe = api.KVPool(1, 64, 8, dtype)
    n = _largest_fitting_rows(probe, 32)
    assert 0 < n < api.MAX_ROWS
    lengths = [1 + (7 * i) % 40 for i in range(n + 1)]  # short rows, 1 to 40 tokens
    wl = W.draw(cfg, lengths=lengths)
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    q, bt, sl = to_dev(wl.q), to_dev(wl.block_table), to_dev(wl.seq_lens)
    qn, sln = q[:n].contiguous(), sl[:n].contiguous()
    btn = bt[:n].contiguous()
    ref = api.paged_decode_attention(pool, 0, qn, btn, sln, wl.scale).cpu().numpy()
    out = torch.full_like(qn, float("nan"))
    assert _call_static(pool, qn, btn, sln, 32, wl.scale, out) == 0
    torch.cuda.synchronize()
    assert float(np.max(np.abs(out.cpu().numpy() - ref))) <= TOL
    out1 = torch.zeros_like(q)
    assert _call_static(pool, q, bt, sl, 32, wl.scale, out1) == 4  # PKV_ERR_WORKSPACE
    assert pool.read_status() == 0

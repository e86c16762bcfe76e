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


@pytest.mark.parametrize("cfg_name", ["llama8b_f16", "skewed"])
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

"""kv_append on the GPU against the oracle's append: bit-exact f16 stores and
q8_0 codes and scales (Leone, "What ships"; LeatEngine, "Run"), through the C
ABI.  Also the rows that write nothing and the device-side bounds checks."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import device_pool, encode_pool, host_arrays, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _append_case(cfg_name, dtype=None, scale_new=1.0, layer=1, layers=3):
    wl = W.draw(cfg_name)
    if dtype is not None:
        wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": dtype})
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host, num_layers=layers, layer=layer)
    k_new = (wl.k_new * scale_new).astype(np.float32)
    v_new = (wl.v_new * scale_new).astype(np.float32)
    api.kv_append(pool, layer, to_dev(k_new), to_dev(v_new), to_dev(wl.block_table),
                  to_dev(wl.seq_lens))
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    got = host_arrays(pool, layer)
    want = [None if a is None else a.copy() for a in host]
    O.kv_append(wl.cfg.dtype, k_new, v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    return wl, pool, got, want


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0, W.BF16, W.F32])
@pytest.mark.parametrize("cfg_name", ["tiny", "skewed"])
def test_append_bit_exact(cfg_name, dtype):
    _, pool, got, want = _append_case(cfg_name, dtype)
    for g, w in zip(got, want):
        if w is not None:
            np.testing.assert_array_equal(g, w)
    # other layers untouched
    other = host_arrays(pool, 0)
    assert np.array_equal(other[0].view(np.uint8), host_arrays(pool, 2)[0].view(np.uint8))


@pytest.mark.parametrize("scale_new", [1e-3, 1e3, 3e4])
def test_append_q8_wide_ranges_and_ties(scale_new):
    _, _, got, want = _append_case("tiny", W.Q8_0, scale_new=scale_new)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)


def test_append_q8_exact_ties():
    """Values x/d = k + 1/2 exactly (d = 1): ties must go away from zero."""
    wl = W.draw("tiny")
    wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": W.Q8_0})
    rng = np.random.default_rng(5)
    k_new = (rng.integers(-126, 126, wl.k_new.shape) + 0.5).astype(np.float32)
    k_new[..., ::32] = 127.0  # amax 127 in every block -> d = 1
    v_new = -k_new
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host)
    api.kv_append(pool, 0, to_dev(k_new), to_dev(v_new), to_dev(wl.block_table),
                  to_dev(wl.seq_lens))
    got = host_arrays(pool)
    want = [a.copy() for a in host]
    O.kv_append(W.Q8_0, k_new, v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)


def test_append_skips_empty_rows_and_flags_bad_pages():
    wl = W.draw("tiny")
    host = encode_pool(wl, include_appended=False)
    pool = device_pool(wl, host)
    before = host_arrays(pool)
    sl = wl.seq_lens.copy()
    sl[0] = 0                       # writes nothing
    bt = wl.block_table.copy()
    bt[1, (sl[1] - 1) // 16] = wl.num_pages + 5   # outside the pool: skipped, flagged
    api.kv_append(pool, 0, to_dev(wl.k_new), to_dev(wl.v_new), to_dev(bt), to_dev(sl))
    assert pool.read_status() & api.DEV_BAD_PAGE
    after = host_arrays(pool)
    want = [a.copy() for a in before[:2]]
    sl2 = sl.copy()
    sl2[1] = 0   # the oracle: row 1 skipped too
    O.kv_append(W.F16, wl.k_new, wl.v_new, wl.block_table, sl2, wl.num_pages, *want)
    np.testing.assert_array_equal(after[0], want[0])
    np.testing.assert_array_equal(after[1], want[1])
    assert pool.read_status() == 0  # reading cleared it


def test_append_rejects_bad_host_arguments():
    wl = W.draw("tiny")
    pool = api.KVPool(1, wl.num_pages, 8, W.F16)
    with pytest.raises(api.PkvError) as e:
        api.kv_append(pool, 1, to_dev(wl.k_new), to_dev(wl.v_new), to_dev(wl.block_table),
                      to_dev(wl.seq_lens))
    assert e.value.status == 1  # layer outside the pool

"""Seeded random cases on the GPU against the FP64 oracle, through the C ABI:
shapes the fixed workloads do not reach (1, 3 or 5 KV heads, lengths on and
around page boundaries, empty rows, windows shorter and longer than rows,
several queries per row with a window, every KV format), each case once with
the append fused into the step.  Bounds as in the other attention tests:
<= 2e-3 and <= 1e-4 * max(1, max|ref|); the pool after a fused step equals the
oracle's append bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import ATOL_STATED, device_pool, encode_pool, host_arrays, tight_tol, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DTYPES = [W.F16, W.Q8_0, W.BF16, W.F32]


def _case(seed):
    rng = np.random.default_rng([77, seed])
    n_kv = int(rng.choice([1, 2, 3, 5, 8]))
    group = int(rng.choice([1, 2, 4]))
    dtype = DTYPES[seed % len(DTYPES)]
    rows = int(rng.integers(1, 12))
    # lengths: a mix of on-page-boundary, one-off-boundary, short and long
    lens = []
    for _ in range(rows):
        kind = rng.integers(0, 4)
        if kind == 0:
            lens.append(16 * int(rng.integers(1, 40)))
        elif kind == 1:
            lens.append(16 * int(rng.integers(1, 40)) + int(rng.choice([-1, 1])))
        elif kind == 2:
            lens.append(int(rng.integers(0, 20)))
        else:
            lens.append(int(rng.integers(20, 1500)))
    window = int(rng.choice([0, 0, 1, 7, 16, 33, 300, 5000]))
    q_len = int(rng.choice([1, 1, 2, 3, 5, 8]))
    lens = [0 if 0 < L < q_len else L for L in lens]  # every row holds its queries
    if sum(lens) == 0:
        lens[0] = max(q_len, 1)
    pages = sum(W.pages_for(L) for L in lens)
    cfg = W.Config(f"fuzz{seed}", rows, ("fixed", tuple(lens)), n_kv * group, n_kv, 128, dtype,
                   ("fixed", pages + int(rng.integers(1, 9))), 1000 + seed)
    return W.draw(cfg), window, q_len


def _check(out, ref):
    assert np.all(np.isfinite(out)), "non-finite output: a poisoned slot was read"
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL_STATED, err
    assert err <= tight_tol(ref), err


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_attention(seed):
    wl, window, q_len = _case(seed)
    dtype = wl.cfg.dtype
    host = encode_pool(wl)
    pool = device_pool(wl, host)
    pool.set_window(0, window)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    if q_len == 1:
        out = api.paged_decode_attention(pool, 0, to_dev(wl.q), bt, sl, wl.scale)
        ref = O.decode_attention(dtype, wl.q, *host, wl.block_table, wl.seq_lens, wl.num_pages,
                                 wl.cfg.n_kv_heads, wl.scale, window=window)
    else:
        q, _, _ = W.mq_inputs(wl, q_len, seed=seed)
        out = api.paged_decode_attention_mq(pool, 0, to_dev(q), bt, sl, wl.scale)
        ref = O.decode_attention_mq(dtype, q, *host, wl.block_table, wl.seq_lens, wl.num_pages,
                                    wl.cfg.n_kv_heads, wl.scale, window=window)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    _check(out.cpu().numpy(), ref)


@pytest.mark.parametrize("seed", range(24, 40))
def test_fuzz_fused_step(seed):
    wl, window, q_len = _case(seed)
    dtype = wl.cfg.dtype
    if q_len == 1:
        host = encode_pool(wl, include_appended=False)
    else:  # the last q_len slots of every row start as NaN: the step writes them
        host = encode_pool(wl)
        nan = {W.F16: np.uint16(0x7E00), W.BF16: np.uint16(0x7FC0), W.F32: np.float32(np.nan)}
        kd, vd, ks, vs = [None if a is None else a.copy() for a in host]
        for i, L in enumerate(wl.seq_lens):
            for t in range(max(0, int(L) - q_len), int(L)):
                page, slot = wl.block_table[i, t // W.PAGE], t % W.PAGE
                if dtype == W.Q8_0:
                    ks[page, :, slot] = np.uint16(0x7E00)
                    vs[page, :, slot] = np.uint16(0x7E00)
                else:
                    kd[page, :, slot] = nan[dtype]
                    vd[page, :, slot] = nan[dtype]
        host = (kd, vd, ks, vs)
    pool = device_pool(wl, host)
    pool.set_window(0, window)
    want = [None if a is None else a.copy() for a in host]
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    if q_len == 1:
        out = api.decode_step(pool, 0, to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new), bt, sl,
                              wl.scale)
        O.kv_append(dtype, wl.k_new, wl.v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
        ref = O.decode_attention(dtype, wl.q, *want, wl.block_table, wl.seq_lens, wl.num_pages,
                                 wl.cfg.n_kv_heads, wl.scale, window=window)
    else:
        q, k_new, v_new = W.mq_inputs(wl, q_len, seed=seed)
        out = api.decode_step_mq(pool, 0, to_dev(q), to_dev(k_new), to_dev(v_new), bt, sl,
                                 wl.scale)
        O.kv_append_mq(dtype, k_new, v_new, wl.block_table, wl.seq_lens, wl.num_pages, *want)
        ref = O.decode_attention_mq(dtype, q, *want, wl.block_table, wl.seq_lens, wl.num_pages,
                                    wl.cfg.n_kv_heads, wl.scale, window=window)
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    for g, w in zip(host_arrays(pool), want):
        if w is not None:
            np.testing.assert_array_equal(g, w)
    _check(out.cpu().numpy(), ref)

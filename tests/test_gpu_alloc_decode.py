"""The host page allocator driving real decode steps on the GPU.

Sequences are admitted with prompts (kv_append of every prompt token), then
decode step by step: reserve 1, build the batch's block tables and lengths
(pkv_alloc_batch with extra = 1), pkv_decode_step, commit 1.  Midway one
sequence is forked: the child shares the parent's complete pages and writes
its non-aligned suffix again (tinyllm, "Known limitations": only complete
pages are shared, a non-aligned suffix is recomputed), then both decode with
different tokens.  A host copy of the pool receives the same appends through
the oracle; the device pool must equal it byte for byte (so no shared page
was ever written), and every step's attention must match the oracle's."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import ATOL_STATED, host_arrays, tight_tol, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N_KV, N_Q, D, PAGES, STRIDE = 8, 32, 128, 96, 24


def _empty_host(dtype):
    if dtype == W.F16:
        z = np.zeros((PAGES, N_KV, 16, D), np.uint16)
        return [z, z.copy(), None, None]
    z = np.zeros((PAGES, N_KV, 16, D), np.int8)
    s = np.zeros((PAGES, N_KV, 16, D // 32), np.uint16)
    return [z, z.copy(), s, s.copy()]


def _append_both(pool, host, dtype, k, v, bt, sl):
    api.kv_append(pool, 0, to_dev(k), to_dev(v), to_dev(bt), to_dev(sl))
    O.kv_append(dtype, k, v, bt, sl, PAGES, *host)


@pytest.mark.parametrize("dtype", [W.F16, W.Q8_0])
def test_allocator_drives_decode_with_a_fork(dtype):
    rng = np.random.default_rng(7 + dtype)
    pool = api.KVPool(1, PAGES, N_KV, dtype)
    for t in (pool.k_data, pool.v_data) + ((pool.k_scales, pool.v_scales) if dtype else ()):
        t.zero_()
    if dtype == W.Q8_0:  # code 0 (the host mirror's zeros) is the stored byte 128
        pool.k_data.fill_(128)
        pool.v_data.fill_(128)
    host = _empty_host(dtype)
    alloc = api.PageAllocator(PAGES, 8, STRIDE)
    prompts = [37, 16, 70, 5]
    seqs = [alloc.open() for _ in prompts]
    for s, P in zip(seqs, prompts):  # prompt tokens: one pseudo-row per token
        alloc.reserve(s, P)
        row = alloc.block_table(s, STRIDE)
        bt = np.repeat(row[None], P, axis=0)
        sl = np.arange(1, P + 1, dtype=np.int32)
        k = rng.standard_normal((P, N_KV, D)).astype(np.float32)
        v = rng.standard_normal((P, N_KV, D)).astype(np.float32)
        _append_both(pool, host, dtype, k, v, bt, sl)
        alloc.commit(s, P)
    scale = 1.0 / np.sqrt(D)
    for step in range(12):
        if step == 5:  # fork sequence 0 (committed 42: 2 complete pages shared, 10 rewritten)
            parent = seqs[0]
            committed, _, _ = alloc.info(parent)
            child = alloc.fork(parent)
            c_len, _, c_pages = alloc.info(child)
            assert c_len == 16 * (committed // 16) and c_pages == committed // 16
            suffix = committed - c_len
            alloc.reserve(child, suffix)
            # the parent's suffix tokens, read back from the host mirror, written again
            p_row = alloc.block_table(parent, STRIDE)
            c_row = alloc.block_table(child, STRIDE)
            pos = np.arange(c_len, committed)
            if dtype == W.F16:
                k = host[0][p_row[pos // 16], :, pos % 16].view(np.float16).astype(np.float32)
                v = host[1][p_row[pos // 16], :, pos % 16].view(np.float16).astype(np.float32)
            else:
                def deq(codes, sc):
                    return (codes.astype(np.float32) *
                            np.repeat(sc.view(np.float16).astype(np.float32), 32, axis=-1))
                k = deq(host[0][p_row[pos // 16], :, pos % 16], host[2][p_row[pos // 16], :, pos % 16])
                v = deq(host[1][p_row[pos // 16], :, pos % 16], host[3][p_row[pos // 16], :, pos % 16])
            bt = np.repeat(c_row[None], suffix, axis=0)
            _append_both(pool, host, dtype, np.ascontiguousarray(k), np.ascontiguousarray(v), bt,
                         (pos + 1).astype(np.int32))
            alloc.commit(child, suffix)
            seqs.append(child)
            _, _, shared = alloc.stats()
            assert shared == committed // 16
        for s in seqs:
            alloc.reserve(s, 1)
        bt, sl = alloc.batch(seqs, 1, STRIDE)
        rows = len(seqs)
        q = rng.standard_normal((rows, N_Q, D)).astype(np.float32)
        k = rng.standard_normal((rows, N_KV, D)).astype(np.float32)
        v = rng.standard_normal((rows, N_KV, D)).astype(np.float32)
        out = api.decode_step(pool, 0, to_dev(q), to_dev(k), to_dev(v), to_dev(bt), to_dev(sl),
                              scale)
        torch.cuda.synchronize()
        assert pool.read_status() == 0
        O.kv_append(dtype, k, v, bt, sl, PAGES, *host)
        ref = O.decode_attention(dtype, q, *host, bt, sl, PAGES, N_KV, scale)
        got = out.cpu().numpy().astype(np.float64)
        err = float(np.max(np.abs(got - ref)))
        assert err <= ATOL_STATED and err <= tight_tol(ref), (step, err)
        for s in seqs:
            alloc.commit(s, 1)
    dev = host_arrays(pool)
    for a, b in zip(dev, host):
        if b is not None:
            np.testing.assert_array_equal(a, b)  # the device pool is the oracle's, byte for byte

"""The plan and combine steps on the GPU against the oracle.

Plan: bit-exact row page offsets and per-segment chunk ranges, for the split
of q8_0 and f32 pools (uniform) and of f16 and bf16 pools (segment-aligned
when it balances).
Combine: the GPU merge of partial states that the ORACLE computed (base 2:
m2 = max log2(e) scale <q, K_t>, l = sum 2^(s2_t - m2), acc = sum 2^(..) V_t)
against the oracle's merge of the same fp32 partials."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import encode_pool, split_aligned, to_dev
from paged_kv_decode_09_gb300 import api
from paged_kv_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(6))
def test_plan_bit_exact(seed):
    rng = np.random.default_rng(seed)
    rows = int(rng.integers(1, 300))
    lens = rng.integers(0, 5000, rows).astype(np.int32)
    lens[rng.integers(0, rows, 3)] = 0
    n_kv = int(rng.choice([1, 2, 8]))
    stride = int((lens.max() + 15) // 16) + 1
    for chunks in (1, 5, 152, 456, 100000):
        for kv_dtype in (W.F16, W.Q8_0):
            rps, first, last = api.paged_decode_plan(to_dev(lens), n_kv, stride, chunks,
                                                     kv_dtype=kv_dtype)
            o_rps, o_first, o_last, _ = O.plan(lens, n_kv, chunks, aligned=split_aligned(kv_dtype))
            np.testing.assert_array_equal(rps.cpu().numpy(), o_rps)
            np.testing.assert_array_equal(first.cpu().numpy(), o_first)
            np.testing.assert_array_equal(last.cpu().numpy(), o_last)


@pytest.mark.parametrize("lens,chunks", [([111, 70, 18, 596], 24), ([693, 10, 18, 71], 20),
                                         ([95, 678, 186, 81], 24)])
def test_plan_where_the_splits_differ(lens, chunks):
    """Cases whose aligned split is not the uniform one (the oracle says so)."""
    lens = np.array(lens, np.int32)
    lo, _ = O.chunk_ranges(lens, 8, chunks, aligned=True)
    ulo, _ = O.chunk_ranges(lens, 8, chunks, aligned=False)
    assert len(lo) != len(ulo) or not np.array_equal(lo, ulo)
    for kv_dtype in (W.F16, W.BF16, W.F32, W.Q8_0):
        rps, first, last = api.paged_decode_plan(to_dev(lens), 8, 64, chunks, kv_dtype=kv_dtype)
        _, o_first, o_last, _ = O.plan(lens, 8, chunks, aligned=split_aligned(kv_dtype))
        np.testing.assert_array_equal(first.cpu().numpy(), o_first)
        np.testing.assert_array_equal(last.cpu().numpy(), o_last)


@pytest.mark.parametrize("lengths,chunks,kv_dtype", [
    ([100, 37, 1, 64], 9, W.F16), ([100, 37, 1, 64], 200, W.F16),
    ([111, 70, 18, 596], 24, W.F16), ([111, 70, 18, 596], 24, W.Q8_0),
    ([111, 70, 18, 596], 24, W.BF16), ([693, 10, 18, 71], 20, W.F32)])
def test_combine_of_oracle_partials(lengths, chunks, kv_dtype):
    """chunks = 200 > 120 units: only 120 chunks are used, one unit each;
    slots no piece owns hold garbage that the merge must not read.  The
    combine follows the split of the pool's format (the partials are those of
    f16 pages either way)."""
    wl = W.draw("tiny", lengths=lengths)
    cfg = wl.cfg
    G = cfg.group
    host = encode_pool(wl)
    aligned = split_aligned(kv_dtype)
    rps, first, last, T = O.plan(wl.seq_lens, cfg.n_kv_heads, chunks, aligned=aligned)
    lo, hi = O.chunk_ranges(wl.seq_lens, cfg.n_kv_heads, chunks, aligned=aligned)
    slots = chunks + wl.rows * cfg.n_kv_heads
    part_ml = np.full((slots, G, 2), 1e30, np.float32)    # garbage in unwritten slots
    part_acc = np.full((slots, G, 128), np.nan, np.float32)
    want = np.zeros((wl.rows, cfg.n_q_heads, 128))
    merged = np.zeros(wl.rows * cfg.n_kv_heads, bool)
    for i in range(wl.rows):
        npg = rps[i + 1] - rps[i]
        for h in range(cfg.n_kv_heads):
            j = i * cfg.n_kv_heads + h
            if first[j] == last[j]:
                continue  # one piece: not the combine's business
            merged[j] = True
            seg0 = cfg.n_kv_heads * rps[i] + h * npg
            pieces = []
            for k in range(first[j], last[j] + 1):
                a = max(lo[k], seg0) - seg0
                b = min(hi[k], seg0 + npg) - seg0
                assert a < b
                pieces.append(k + j)
                t0, t1 = a * 16, min(b * 16, int(wl.seq_lens[i]))
                for g in range(G):
                    m2, l, acc = O.attention_partial(cfg.dtype, wl.q[i], *host, wl.block_table,
                                                     wl.num_pages, cfg.n_kv_heads, i, h * G + g,
                                                     wl.scale, t0, t1)
                    part_ml[k + j, g] = (m2, l)
                    part_acc[k + j, g] = acc
            for g in range(G):
                s = pieces
                want[i, h * G + g] = O.combine(part_ml[s, g, 0], part_ml[s, g, 1], part_acc[s, g])
    assert merged.sum() >= 5 or chunks == 200
    nbytes = api.workspace_bytes(wl.rows, cfg.n_q_heads, cfg.n_kv_heads, chunks)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    # layout: part_ml, part_acc (256-byte aligned), then the merge's flags down from the end
    up = lambda n: (n + 255) // 256 * 256  # noqa: E731
    ml_at = 0
    acc_at = ml_at + up(slots * G * 2 * 4)
    assert acc_at + up(part_acc.nbytes) + up(slots * 2 * 4) == nbytes
    ws[ml_at:ml_at + part_ml.nbytes] = torch.from_numpy(part_ml.view(np.uint8).reshape(-1)).cuda()
    ws[acc_at:acc_at + part_acc.nbytes] = torch.from_numpy(
        part_acc.view(np.uint8).reshape(-1)).cuda()
    out = torch.full((wl.rows, cfg.n_q_heads, 128), 7.0, device="cuda")
    api.paged_decode_combine(to_dev(wl.seq_lens), cfg.n_q_heads, cfg.n_kv_heads, wl.bt_stride,
                             chunks, ws, out, kv_dtype=kv_dtype)
    got = out.cpu().numpy().reshape(wl.rows, cfg.n_kv_heads, G, 128)
    w = want.reshape(wl.rows, cfg.n_kv_heads, G, 128)
    m = merged.reshape(wl.rows, cfg.n_kv_heads)
    np.testing.assert_allclose(got[m], w[m], rtol=0, atol=1e-6)
    assert np.all(got[~m] == 7.0)  # untouched where one piece holds the segment

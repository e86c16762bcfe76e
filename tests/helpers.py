"""Test-side helpers: build host pools from seeded workloads with the oracle's
encoder, poison unused slots, and small utilities shared by the tests.

Pool arrays per layer (the library's documented layout): data
[num_pages][n_kv][16][D] (uint16 f16 / bf16 bits, float32, or q8_0 codes), q8_0 scales
[num_pages][n_kv][16][D/32] (uint16 f16 bits).  The oracle holds q8_0 codes as int8; the
library stores them offset-binary (code + 128, the int8 byte with its top bit flipped):
device_pool and host_arrays convert."""
from __future__ import annotations

import numpy as np

import oracle as O
from paged_kv_decode_09_gb300 import workloads as W

F16_NAN = np.uint16(0x7E00)
BF16_NAN = np.uint16(0x7FC0)
F32_NAN = np.float32(np.nan)


def encode_pool(wl: W.Workload, layer: int = 0, include_appended: bool = True,
                poison: bool = True):
    """(k_data, v_data, k_scales, v_scales) host arrays of one layer's pool.

    Context values come from the seeded generator and are stored by the
    oracle's encoder.  Slots that hold no token (and, with
    include_appended=False, the slot the step will append into) are poisoned
    with f16 NaN (f16 data, or the q8_0 block scales), so that a kernel reading
    one produces NaN."""
    cfg = wl.cfg
    k, v = W.context_values(wl, layer)
    kd, ks = O.encode_pool(cfg.dtype, k)
    vd, vs = O.encode_pool(cfg.dtype, v)
    if poison:
        unused = ~W.used_slots(wl, include_appended=include_appended)  # [pages][16]
        sel = np.broadcast_to(unused[:, None, :], (wl.num_pages, cfg.n_kv_heads, W.PAGE))
        if cfg.dtype == W.F16:
            kd[sel] = F16_NAN
            vd[sel] = F16_NAN
        elif cfg.dtype == W.BF16:
            kd[sel] = BF16_NAN
            vd[sel] = BF16_NAN
        elif cfg.dtype == W.F32:
            kd[sel] = F32_NAN
            vd[sel] = F32_NAN
        else:
            ks[sel] = F16_NAN
            vs[sel] = F16_NAN
            kd[sel] = 127
            vd[sel] = 127
    return kd, vd, ks, vs


def oracle_decode(wl: W.Workload, pool, seq_lens=None, q=None, scale=None, window=0):
    kd, vd, ks, vs = pool
    return O.decode_attention(wl.cfg.dtype, wl.q if q is None else q, kd, vd, ks, vs,
                              wl.block_table, wl.seq_lens if seq_lens is None else seq_lens,
                              wl.num_pages, wl.cfg.n_kv_heads,
                              wl.scale if scale is None else scale, window=window)


def stored_values_dense(dtype, data, scales):
    """float64 values of pool elements [..., D] using numpy's own float16
    widening (a route independent of the oracle's)."""
    if dtype == W.F16:
        return data.view(np.float16).astype(np.float64)
    if dtype == W.BF16:  # the high half of a binary32
        return (data.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == W.F32:
        return data.astype(np.float64)
    sc = scales.view(np.float16).astype(np.float64)
    return np.repeat(sc, 32, axis=-1) * data.astype(np.float64)


def max_abs_err(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


# ------------------------------------------------------------- device side ----
def stored_codes(codes):
    """int8 q8_0 codes as the pool's offset-binary bytes."""
    return np.ascontiguousarray(codes).view(np.uint8) ^ np.uint8(0x80)


def int8_codes(stored):
    """The pool's offset-binary q8_0 bytes as int8 codes."""
    return (np.ascontiguousarray(stored).view(np.uint8) ^ np.uint8(0x80)).view(np.int8)


def device_pool(wl: W.Workload, host_pool, num_layers: int = 1, layer: int = 0):
    """A library KVPool on cuda:0 holding the host pool arrays in `layer`
    (other layers are filled with f16 NaN / NaN scales)."""
    import torch
    from paged_kv_decode_09_gb300 import api
    cfg = wl.cfg
    pool = api.KVPool(num_layers, wl.num_pages, cfg.n_kv_heads, cfg.dtype, device="cuda")
    kd, vd, ks, vs = host_pool
    if cfg.dtype in (W.F16, W.BF16):  # 16-bit patterns copied as int16
        nan = 0x7E00 if cfg.dtype == W.F16 else 0x7FC0
        for t in (pool.k_data, pool.v_data):
            t.view(torch.int16).fill_(nan)
        pool.k_data[layer].view(torch.int16).copy_(torch.from_numpy(kd.view(np.int16)))
        pool.v_data[layer].view(torch.int16).copy_(torch.from_numpy(vd.view(np.int16)))
    elif cfg.dtype == W.F32:
        for t in (pool.k_data, pool.v_data):
            t.fill_(float("nan"))
        pool.k_data[layer].copy_(torch.from_numpy(np.ascontiguousarray(kd, np.float32)))
        pool.v_data[layer].copy_(torch.from_numpy(np.ascontiguousarray(vd, np.float32)))
    else:
        for t in (pool.k_scales, pool.v_scales):
            t.view(torch.int16).fill_(0x7E00)
        pool.k_data.fill_(127)
        pool.v_data.fill_(127)
        pool.k_data[layer].copy_(torch.from_numpy(stored_codes(kd)))
        pool.v_data[layer].copy_(torch.from_numpy(stored_codes(vd)))
        pool.k_scales[layer].copy_(torch.from_numpy(ks.view(np.float16)))
        pool.v_scales[layer].copy_(torch.from_numpy(vs.view(np.float16)))
    return pool


def split_aligned(dtype) -> bool:
    """Whether attention calls on a pool of this KV format may use the segment-aligned split
    (the oracle plan's `aligned` flag): the 16-bit formats."""
    return dtype in (W.F16, W.BF16)


def host_arrays(pool, layer: int = 0):
    """(k_data, v_data, k_scales, v_scales) numpy copies of one layer of a device pool."""
    import torch
    if pool.dtype in (W.F16, W.BF16):
        return (pool.k_data[layer].cpu().view(torch.int16).numpy().view(np.uint16),
                pool.v_data[layer].cpu().view(torch.int16).numpy().view(np.uint16), None, None)
    if pool.dtype == W.F32:
        return pool.k_data[layer].cpu().numpy(), pool.v_data[layer].cpu().numpy(), None, None
    return (int8_codes(pool.k_data[layer].cpu().numpy()), int8_codes(pool.v_data[layer].cpu().numpy()),
            pool.k_scales[layer].cpu().view(torch.int16).numpy().view(np.uint16),
            pool.v_scales[layer].cpu().view(torch.int16).numpy().view(np.uint16))


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


# Tolerances of the attention parity tests: the stated bound (2e-3 max abs
# against the FP64 oracle) and a tighter internal one.  fp32 accumulation over
# a few thousand tokens with O(1) logits errs by ~1e-6; 1e-4 leaves margin
# while still failing on a single dropped or misplaced token of a short row.
ATOL_STATED = 2e-3


def tight_tol(ref):
    return 1e-4 * max(1.0, float(np.max(np.abs(ref))))

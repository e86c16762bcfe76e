"""FP64 CPU oracle for one paged-KV decode step (ctypes wrapper of pkv_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product package.  It
shares no code with the CUDA path.  Every function states the definition it
evaluates; the C source cites the pages it follows:

* tinyllm, "The repository currently provides" / "Known limitations": a
  physical pool of 16-token KV pages reached through a per-row block table; the
  paged-reference decode gathers a row's pages and runs dense attention.
* Leone, "What ships"; LeatEngine, "Run": f16 and q8_0 KV storage.

Pool layout per layer (a reading; the pages fix none): data
``[num_pages][n_kv][16][D]`` (f16 or bf16 bits as uint16, float32, or int8
codes), q8_0 scales ``[num_pages][n_kv][16][D/32]`` (f16 bits as uint16).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

F16, Q8_0, BF16, F32 = 0, 1, 2, 3
PAGE = 16
QBLOCK = 32

_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(np.int8, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p
_i = ctypes.c_int


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    with _lock:
        if _lib is None:
            # PKV_ORACLE_LIB points the wrapper at another build of the oracle;
            # the mutation tests use it to load deliberately broken copies.
            path = os.environ.get("PKV_ORACLE_LIB") or _build.build()
            L = ctypes.CDLL(path)
            L.oracle_num_threads.restype = _i
            L.oracle_set_num_threads.argtypes = [_i]
            L.oracle_set_num_threads.restype = None
            L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f64.restype = ctypes.c_double
            L.oracle_f16_from_f32.argtypes = [ctypes.c_float]
            L.oracle_f16_from_f32.restype = ctypes.c_uint16
            L.oracle_q8_0_encode_block.argtypes = [_f32p, _i8p, ctypes.POINTER(ctypes.c_uint16)]
            L.oracle_q8_0_encode_block.restype = ctypes.c_float
            L.oracle_q8_0_encode.argtypes = [_f32p, ctypes.c_int64, _i8p, _u16p]
            L.oracle_q8_0_encode.restype = None
            L.oracle_f16_encode.argtypes = [_f32p, ctypes.c_int64, _u16p]
            L.oracle_f16_encode.restype = None
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
            L.oracle_bf16_from_f32.restype = ctypes.c_uint16
            L.oracle_bf16_encode.argtypes = [_f32p, ctypes.c_int64, _u16p]
            L.oracle_bf16_encode.restype = None
            L.oracle_kv_append.argtypes = [_i, _i, _i, _i, _f32p, _f32p, _i32p, _i, _i32p, _i,
                                           _vp, _vp, _vp, _vp]
            L.oracle_kv_append.restype = _i
            L.oracle_decode_attention.argtypes = [_i, _i, _i, _i, _i, _f32p, _vp, _vp, _vp, _vp,
                                                  _i32p, _i, _i32p, _i, ctypes.c_double, _i,
                                                  _f64p]
            L.oracle_decode_attention.restype = _i
            L.oracle_decode_attention_mq.argtypes = [_i, _i, _i, _i, _i, _i, _f32p, _vp, _vp, _vp,
                                                     _vp, _i32p, _i, _i32p, _i, ctypes.c_double,
                                                     _i, _f64p]
            L.oracle_decode_attention_mq.restype = _i
            L.oracle_kv_append_mq.argtypes = [_i, _i, _i, _i, _i, _f32p, _f32p, _i32p, _i, _i32p,
                                              _i, _vp, _vp, _vp, _vp]
            L.oracle_kv_append_mq.restype = _i
            L.oracle_attention_partial.argtypes = [
                _i, _i, _i, _i, _f32p, _vp, _vp, _vp, _vp, _i32p, _i, _i, _i, _i,
                ctypes.c_double, _i, _i, ctypes.POINTER(ctypes.c_double),
                ctypes.POINTER(ctypes.c_double), _f64p]
            L.oracle_attention_partial.restype = _i
            L.oracle_combine.argtypes = [_i, _f32p, _f32p, _f32p, _i, _f64p]
            L.oracle_combine.restype = None
            L.oracle_plan.argtypes = [_i, _i32p, _i, _i, _i, _i, _i32p, _i32p, _i32p, _i64p]
            L.oracle_plan.restype = _i
            L.oracle_chunk_ranges.argtypes = [_i, _i32p, _i, _i, _i, _i, _i64p, _i64p, _i64p]
            L.oracle_chunk_ranges.restype = _i
            _lib = L
    return _lib


def num_threads() -> int:
    """Threads the oracle's parallel loop uses (OpenMP), 1 without OpenMP."""
    return lib().oracle_num_threads()


def set_num_threads(n: int):
    """Threads for the oracle's parallel loops from now on (timing only)."""
    lib().oracle_set_num_threads(int(n))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ f16 ----
def f16_from_f32(x: float) -> int:
    """Bits of the binary16 nearest to fp32 x, ties to even."""
    return int(lib().oracle_f16_from_f32(float(np.float32(x))))


def f16_to_f64(bits: int) -> float:
    """Exact value of a binary16 bit pattern."""
    return float(lib().oracle_f16_to_f64(int(bits) & 0xFFFF))


def f16_encode(x: np.ndarray) -> np.ndarray:
    """Elementwise binary16 bits (uint16) of an fp32 array, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f16_encode(x.reshape(-1), x.size, out.reshape(-1))
    return out


def f16_decode(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of a uint16 array of binary16 bits."""
    f = np.vectorize(lambda b: lib().oracle_f16_to_f64(int(b)), otypes=[np.float64])
    return f(np.asarray(bits, np.uint16))


def bf16_from_f32(x: float) -> int:
    """Bits of the bfloat16 nearest to fp32 x, ties to even."""
    return int(lib().oracle_bf16_from_f32(float(np.float32(x))))


def bf16_to_f64(bits: int) -> float:
    """Exact value of a bfloat16 bit pattern."""
    return float(lib().oracle_bf16_to_f64(int(bits) & 0xFFFF))


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """Elementwise bfloat16 bits (uint16) of an fp32 array, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_bf16_encode(x.reshape(-1), x.size, out.reshape(-1))
    return out


# ----------------------------------------------------------------- q8_0 ----
def q8_0_encode_block(x: np.ndarray):
    """(codes int8[32], scale bits uint16, fp32 d) of one 32-value block."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (QBLOCK,)
    codes = np.empty(QBLOCK, np.int8)
    sb = ctypes.c_uint16(0)
    d = lib().oracle_q8_0_encode_block(x, codes, ctypes.byref(sb))
    return codes, int(sb.value), float(np.float32(d))


def q8_0_encode(x: np.ndarray):
    """(codes int8, scale bits uint16 [..., D/32]) of an fp32 array [..., D]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape[-1] % QBLOCK == 0
    codes = np.empty(x.shape, np.int8)
    scales = np.empty(x.shape[:-1] + (x.shape[-1] // QBLOCK,), np.uint16)
    lib().oracle_q8_0_encode(x.reshape(-1), x.size, codes.reshape(-1), scales.reshape(-1))
    return codes, scales


def encode_pool(dtype: int, values: np.ndarray):
    """Store fp32 values [pages][n_kv][16][D] in the pool dtype: (data, scales).

    f16 / bf16: data uint16 bits, scales None.  f32: the fp32 values as given,
    scales None.  q8_0: data int8 codes, scales uint16 [pages][n_kv][16][D/32]."""
    if dtype == F16:
        return f16_encode(values), None
    if dtype == BF16:
        return bf16_encode(values), None
    if dtype == F32:
        return np.array(values, dtype=np.float32, copy=True), None
    return q8_0_encode(values)


# ---------------------------------------------------------- decode step ----
def kv_append(dtype, k_new, v_new, block_table, seq_lens, num_pages, k_data, v_data,
              k_scales=None, v_scales=None):
    """Write row i's new K/V token (fp32 [rows][n_kv][D]) into the pool arrays
    (modified in place) at position seq_lens[i]-1: page block_table[i][pos//16],
    slot pos % 16."""
    k_new = np.ascontiguousarray(k_new, np.float32)
    v_new = np.ascontiguousarray(v_new, np.float32)
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    rows, n_kv, D = k_new.shape
    for a in (k_data, v_data, k_scales, v_scales):
        assert a is None or a.flags.c_contiguous
    st = lib().oracle_kv_append(dtype, rows, n_kv, D, k_new.reshape(-1), v_new.reshape(-1),
                                bt.reshape(-1), bt.shape[1], sl, num_pages, _ptr(k_data),
                                _ptr(v_data), _ptr(k_scales), _ptr(v_scales))
    if st:
        raise ValueError(f"oracle_kv_append: status {st}")


def decode_attention(dtype, q, k_data, v_data, k_scales, v_scales, block_table, seq_lens,
                     num_pages, n_kv, scale, window=0):
    """out[i][g] = softmax_t(scale <q[i][g], K[i][g//G][t]>) V over the row's
    tokens max(0, L - window) <= t < L (all L for window 0), L = seq_lens[i],
    in float64 [rows][n_q][D]; zeros for rows with seq_lens[i] <= 0."""
    q = np.ascontiguousarray(q, np.float32)
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    rows, n_q, D = q.shape
    for a in (k_data, v_data, k_scales, v_scales):
        assert a is None or a.flags.c_contiguous
    out = np.zeros((rows, n_q, D), np.float64)
    st = lib().oracle_decode_attention(dtype, rows, n_q, n_kv, D, q.reshape(-1), _ptr(k_data),
                                       _ptr(v_data), _ptr(k_scales), _ptr(v_scales),
                                       bt.reshape(-1), bt.shape[1], sl, num_pages,
                                       float(scale), int(window), out.reshape(-1))
    if st:
        raise ValueError(f"oracle_decode_attention: status {st}")
    return out


def decode_attention_mq(dtype, q, k_data, v_data, k_scales, v_scales, block_table, seq_lens,
                        num_pages, n_kv, scale, window=0):
    """Several queries per row: q [rows][q_len][n_q][D]; query j of row i sits
    at position L - q_len + j (L = seq_lens[i]) and attends causally to
    [max(0, P + 1 - window), P + 1).  float64 [rows][q_len][n_q][D]."""
    q = np.ascontiguousarray(q, np.float32)
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    rows, q_len, n_q, D = q.shape
    out = np.zeros((rows, q_len, n_q, D), np.float64)
    st = lib().oracle_decode_attention_mq(dtype, rows, q_len, n_q, n_kv, D, q.reshape(-1),
                                          _ptr(k_data), _ptr(v_data), _ptr(k_scales),
                                          _ptr(v_scales), bt.reshape(-1), bt.shape[1], sl,
                                          num_pages, float(scale), int(window), out.reshape(-1))
    if st:
        raise ValueError(f"oracle_decode_attention_mq: status {st}")
    return out


def kv_append_mq(dtype, k_new, v_new, block_table, seq_lens, num_pages, k_data, v_data,
                 k_scales=None, v_scales=None):
    """Store q_len new tokens per row (k_new, v_new [rows][q_len][n_kv][D]) at
    positions L - q_len + j, in place."""
    k_new = np.ascontiguousarray(k_new, np.float32)
    v_new = np.ascontiguousarray(v_new, np.float32)
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    rows, q_len, n_kv, D = k_new.shape
    st = lib().oracle_kv_append_mq(dtype, rows, q_len, n_kv, D, k_new.reshape(-1),
                                   v_new.reshape(-1), bt.reshape(-1), bt.shape[1], sl, num_pages,
                                   _ptr(k_data), _ptr(v_data), _ptr(k_scales), _ptr(v_scales))
    if st:
        raise ValueError(f"oracle_kv_append_mq: status {st}")


def attention_partial(dtype, q_row, k_data, v_data, k_scales, v_scales, block_table, num_pages,
                      n_kv, row, g, scale, t0, t1):
    """Base-2 partial state (m2, l, acc[D]) of row `row`, query head g over
    tokens [t0, t1): s2_t = log2(e) scale <q, K_t>, m2 = max s2_t,
    l = sum 2^(s2_t - m2), acc = sum 2^(s2_t - m2) V_t."""
    q_row = np.ascontiguousarray(q_row, np.float32)
    bt = np.ascontiguousarray(block_table, np.int32)
    n_q, D = q_row.shape
    m2, l = ctypes.c_double(), ctypes.c_double()
    acc = np.zeros(D, np.float64)
    st = lib().oracle_attention_partial(dtype, n_q, n_kv, D, q_row.reshape(-1), _ptr(k_data),
                                        _ptr(v_data), _ptr(k_scales), _ptr(v_scales),
                                        bt.reshape(-1), bt.shape[1], num_pages, row, g,
                                        float(scale), t0, t1, ctypes.byref(m2),
                                        ctypes.byref(l), acc)
    if st:
        raise ValueError(f"oracle_attention_partial: status {st}")
    return m2.value, l.value, acc


def combine(m2, l, acc):
    """Merge base-2 partials (fp32 m2[n], l[n], acc[n][D]) of disjoint token
    ranges: out = sum_s 2^(m2_s - M) acc_s / sum_s 2^(m2_s - M) l_s."""
    m2 = np.ascontiguousarray(m2, np.float32)
    l = np.ascontiguousarray(l, np.float32)
    acc = np.ascontiguousarray(acc, np.float32)
    n, D = acc.shape
    out = np.zeros(D, np.float64)
    lib().oracle_combine(n, m2, l, acc.reshape(-1), D, out)
    return out


def chunk_ranges(seq_lens, n_kv, num_chunks, window=0, aligned=False):
    """(lo, hi): unit ranges [lo[k], hi[k]) of the chunks that hold units, in the split
    `plan` describes."""
    sl = np.ascontiguousarray(seq_lens, np.int32)
    lo = np.zeros(num_chunks, np.int64)
    hi = np.zeros(num_chunks, np.int64)
    used = np.zeros(1, np.int64)
    st = lib().oracle_chunk_ranges(sl.shape[0], sl, n_kv, num_chunks, int(window),
                                   int(bool(aligned)), lo, hi, used)
    if st:
        raise ValueError(f"oracle_chunk_ranges: status {st}")
    return lo[:used[0]], hi[:used[0]]


def plan(seq_lens, n_kv, num_chunks, window=0, aligned=False):
    """Work split of one decode call (see oracle_plan in the C source); `aligned`: the call
    allows the segment-aligned split (f16 and bf16 KV):
    (row_page_start[rows+1], seg_first_chunk[rows*n_kv], seg_last_chunk[...], T)."""
    sl = np.ascontiguousarray(seq_lens, np.int32)
    rows = sl.shape[0]
    rps = np.zeros(rows + 1, np.int32)
    first = np.zeros(max(rows * n_kv, 1), np.int32)
    last = np.zeros(max(rows * n_kv, 1), np.int32)
    total = np.zeros(1, np.int64)
    st = lib().oracle_plan(rows, sl, n_kv, num_chunks, int(window), int(bool(aligned)), rps, first,
                           last, total)
    if st:
        raise ValueError(f"oracle_plan: status {st}")
    return rps, first[:rows * n_kv], last[:rows * n_kv], int(total[0])

"""ctypes binding of libpkv.so (C ABI in include/pkv.h).

Argument marshalling only: every function checks tensor dtypes, shapes and
devices, passes raw device pointers and the current torch CUDA stream to the
C entry point of the same name, and raises PkvError on a non-zero status.  All
compute runs in the library's CUDA kernels; there is no CPU fallback, and a
missing library raises on first use.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

F16, Q8_0, BF16, F32 = 0, 1, 2, 3
_TORCH_DTYPE = {F16: torch.float16, Q8_0: torch.uint8, BF16: torch.bfloat16, F32: torch.float32}
PAGE = 16
HEAD_DIM = 128
Q8_BLOCK = 32
MAX_ROWS = 2048
DEFAULT_WAIT_NS = 1 << 30

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")
_lock = threading.Lock()
_lib = None

STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_CAPACITY", 4: "PKV_ERR_WORKSPACE", 5: "PKV_ERR_CUDA"}
DEV_BAD_PAGE, DEV_BAD_LENGTH, DEV_TIMEOUT = 1, 2, 4


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "kv_pool_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "kv_pool_create": ([ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp], _i),
    "kv_pool_destroy": ([_vp], None),
    "kv_pool_read_status": ([_vp, _vp, ctypes.POINTER(ctypes.c_int32)], _i),
    "kv_append": ([_vp, _i, _vp, _vp, _vp, _i, _vp, _i, _vp], _i),
    "paged_decode_default_chunks": ([_vp, _i, _i, ctypes.POINTER(_i)], _i),
    "paged_decode_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "paged_decode_attention": ([_vp, _i, _vp, _vp, _i, _vp, _i, _i, ctypes.c_float, _vp, _vp,
                                _sz, _i, _vp], _i),
    "paged_decode_split": ([_vp, _i, _vp, _vp, _i, _vp, _i, _i, ctypes.c_float, _vp, _vp,
                            _sz, _i, _vp], _i),
    "paged_decode_plan": ([_vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp], _i),
    "paged_decode_combine": ([_vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp], _i),
    "kv_pool_set_window": ([_vp, _i, _i], _i),
    "kv_pool_set_test_stall": ([_vp, ctypes.c_ulonglong], _i),
    "pkv_alloc_create": ([ctypes.POINTER(_vp), _i, _i, _i], _i),
    "pkv_alloc_destroy": ([_vp], None),
    "pkv_alloc_open": ([_vp, ctypes.POINTER(_i)], _i),
    "pkv_alloc_reserve": ([_vp, _i, _i], _i),
    "pkv_alloc_commit": ([_vp, _i, _i], _i),
    "pkv_alloc_reserve_many": ([_vp, _vp, _i, _i], _i),
    "pkv_alloc_commit_many": ([_vp, _vp, _i, _i], _i),
    "pkv_alloc_unreserve": ([_vp, _i, _i], _i),
    "pkv_alloc_fork": ([_vp, _i, ctypes.POINTER(_i)], _i),
    "pkv_alloc_release": ([_vp, _i], _i),
    "pkv_alloc_seq_info": ([_vp, _i, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)],
                           _i),
    "pkv_alloc_block_table": ([_vp, _i, _vp, _i], _i),
    "pkv_alloc_batch": ([_vp, _vp, _i, _i, _vp, _i, _vp], _i),
    "pkv_alloc_stats": ([_vp, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)], _i),
    "pkv_alloc_page_refs": ([_vp, _i, ctypes.POINTER(_i)], _i),
    "kv_pool_get_window": ([_vp, _i, ctypes.POINTER(_i)], _i),
    "pkv_decode_step": ([_vp, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, ctypes.c_float, _vp, _vp,
                         _sz, _i, _vp], _i),
    "paged_decode_workspace_bytes_mq": ([_i, _i, _i, _i, _i], _sz),
    "paged_decode_default_chunks_mq": ([_vp, _i, _i, _i, ctypes.POINTER(_i)], _i),
    "paged_decode_attention_mq": ([_vp, _i, _vp, _vp, _i, _vp, _i, _i, _i, ctypes.c_float, _vp,
                                   _vp, _sz, _i, _vp], _i),
    "pkv_decode_step_mq": ([_vp, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, ctypes.c_float,
                            _vp, _vp, _sz, _i, _vp], _i),
    "pkv_status_string": ([_i], ctypes.c_char_p),
    "pkv_last_error_message": ([], ctypes.c_char_p),
}


def lib():
    """The loaded libpkv.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise PkvError(-1, "libpkv", f"{_LIB_PATH} is missing: run "
                               "paged_kv_decode_09_gb300.build.build() (nvcc, sm_103a) first")
            L = ctypes.CDLL(_LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pkv_status_string(status).decode()


def _check(status: int, where: str):
    if status != 0:
        raise PkvError(status, where, lib().pkv_last_error_message().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


class KVPool:
    """A caller-owned paged KV pool (torch tensors) and its library descriptor.

    k_data / v_data: [layers][pages][n_kv][16][128] float16 (f16), uint8 (q8_0
    codes stored offset-binary: code + 128), bfloat16 (bf16) or float32 (f32);
    k_scales / v_scales (q8_0): [layers][pages][n_kv][16][4] float16;
    status: int32 [1] device status word."""

    def __init__(self, num_layers, num_pages, n_kv_heads, dtype=F16, head_dim=HEAD_DIM,
                 device="cuda", tensors=None):
        self.num_layers, self.num_pages, self.n_kv = num_layers, num_pages, n_kv_heads
        self.dtype, self.head_dim = dtype, head_dim
        self.device = torch.device(device)
        if self.device.index is None:
            self.device = torch.device(self.device.type, torch.cuda.current_device())
        shape = (num_layers, num_pages, n_kv_heads, PAGE, head_dim)
        sshape = (num_layers, num_pages, n_kv_heads, PAGE, head_dim // Q8_BLOCK)
        if tensors is None:
            tdt = _TORCH_DTYPE[dtype]
            tensors = [torch.empty(shape, dtype=tdt, device=self.device),
                       torch.empty(shape, dtype=tdt, device=self.device)]
            if dtype == Q8_0:
                tensors += [torch.empty(sshape, dtype=torch.float16, device=self.device),
                            torch.empty(sshape, dtype=torch.float16, device=self.device)]
        self.k_data, self.v_data = tensors[0], tensors[1]
        self.k_scales = tensors[2] if dtype == Q8_0 else None
        self.v_scales = tensors[3] if dtype == Q8_0 else None
        tdt = _TORCH_DTYPE[dtype]
        for name in ("k_data", "v_data"):
            _need(getattr(self, name), tdt, name, shape, self.device)
        if dtype == Q8_0:
            for name in ("k_scales", "v_scales"):
                _need(getattr(self, name), torch.float16, name, sshape, self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        h = ctypes.c_void_p()
        _check(lib().kv_pool_create(ctypes.byref(h), num_layers, num_pages, n_kv_heads, head_dim,
                                    dtype, _ptr(self.k_data), _ptr(self.v_data),
                                    _ptr(self.k_scales), _ptr(self.v_scales), _ptr(self.status)),
               "kv_pool_create")
        self.handle = h

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.kv_pool_destroy(h)
            self.handle = None

    def set_window(self, layer: int, window: int):
        """Sliding window of `layer` (0: none): attention on the layer reads
        each row's last `window` tokens only."""
        _check(lib().kv_pool_set_window(self.handle, layer, window), "kv_pool_set_window")

    def set_test_stall(self, stall_ns: int):
        """Test hook (kv_pool_set_test_stall in pkv.h): with stall_ns > 0 the
        attention kernels stall on a barrier nothing completes, give up after
        stall_ns and take their timeout path; 0 turns it off."""
        _check(lib().kv_pool_set_test_stall(self.handle, int(stall_ns)), "kv_pool_set_test_stall")

    def window(self, layer: int) -> int:
        w = ctypes.c_int(0)
        _check(lib().kv_pool_get_window(self.handle, layer, ctypes.byref(w)), "kv_pool_get_window")
        return w.value

    def read_status(self, stream=None) -> int:
        """Synchronise and return (and clear) the device status word."""
        out = ctypes.c_int32(0)
        _check(lib().kv_pool_read_status(self.handle, _stream(stream), ctypes.byref(out)),
               "kv_pool_read_status")
        return out.value

    @staticmethod
    def bytes(num_layers, num_pages, n_kv_heads, dtype, which=0, head_dim=HEAD_DIM) -> int:
        return lib().kv_pool_bytes(num_layers, num_pages, n_kv_heads, head_dim, dtype, which)


def default_chunks(pool: KVPool, n_q_heads: int, max_rows: int) -> int:
    c = ctypes.c_int(0)
    _check(lib().paged_decode_default_chunks(pool.handle, n_q_heads, max_rows, ctypes.byref(c)),
           "paged_decode_default_chunks")
    return c.value


def workspace_bytes(max_rows: int, n_q_heads: int, n_kv_heads: int, num_chunks: int,
                    head_dim: int = HEAD_DIM) -> int:
    n = lib().paged_decode_workspace_bytes(max_rows, n_q_heads, n_kv_heads, head_dim, num_chunks)
    if n == 0 and max_rows > 0:
        raise PkvError(1, "paged_decode_workspace_bytes", "invalid sizes")
    return n


class Workspace:
    """Device scratch for paged_decode_attention: arrival counters and partial
    states.  Zero-filled here, as the library requires before first use."""

    def __init__(self, pool: KVPool, n_q_heads: int, max_rows: int, num_chunks: int = 0):
        self.num_chunks = num_chunks or default_chunks(pool, n_q_heads, max_rows)
        self.nbytes = workspace_bytes(max_rows, n_q_heads, pool.n_kv, self.num_chunks)
        self.tensor = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=pool.device)


def _rows(block_table, seq_lens, device):
    _need(block_table, torch.int32, "block_table", device=device)
    _need(seq_lens, torch.int32, "seq_lens", device=device)
    if block_table.dim() != 2 or seq_lens.dim() != 1 or block_table.shape[0] != seq_lens.shape[0]:
        raise ValueError("block_table must be [rows][stride] and seq_lens [rows]")
    return seq_lens.shape[0], block_table.shape[1]


def kv_append(pool: KVPool, layer: int, k_new, v_new, block_table, seq_lens, stream=None):
    rows, stride = _rows(block_table, seq_lens, pool.device)
    shape = (rows, pool.n_kv, pool.head_dim)
    _need(k_new, torch.float32, "k_new", shape, pool.device)
    _need(v_new, torch.float32, "v_new", shape, pool.device)
    _check(lib().kv_append(pool.handle, layer, _ptr(k_new), _ptr(v_new), _ptr(block_table),
                           stride, _ptr(seq_lens), rows, _stream(stream)), "kv_append")


def paged_decode_attention(pool: KVPool, layer: int, q, block_table, seq_lens, scale: float,
                           out=None, workspace: Workspace | None = None, num_chunks: int = 0,
                           stream=None):
    rows, stride = _rows(block_table, seq_lens, pool.device)
    _need(q, torch.float32, "q", device=pool.device)
    if q.dim() != 3 or q.shape[0] != rows or q.shape[2] != pool.head_dim:
        raise ValueError("q must be [rows][n_q_heads][128]")
    n_q = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float32, "out", q.shape, pool.device)
    if workspace is None:
        workspace = Workspace(pool, n_q, max(rows, 1), num_chunks)
    chunks = num_chunks or workspace.num_chunks
    _check(lib().paged_decode_attention(pool.handle, layer, _ptr(q), _ptr(block_table), stride,
                                        _ptr(seq_lens), rows, n_q, float(scale), _ptr(out),
                                        _ptr(workspace.tensor), workspace.nbytes, chunks,
                                        _stream(stream)), "paged_decode_attention")
    return out


def decode_step(pool: KVPool, layer: int, q, k_new, v_new, block_table, seq_lens, scale: float,
                out=None, workspace: Workspace | None = None, num_chunks: int = 0, stream=None):
    """Append each row's new token, then attend (pkv_decode_step, one launch)."""
    rows, stride = _rows(block_table, seq_lens, pool.device)
    _need(q, torch.float32, "q", device=pool.device)
    shape = (rows, pool.n_kv, pool.head_dim)
    _need(k_new, torch.float32, "k_new", shape, pool.device)
    _need(v_new, torch.float32, "v_new", shape, pool.device)
    n_q = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float32, "out", q.shape, pool.device)
    if workspace is None:
        workspace = Workspace(pool, n_q, max(rows, 1), num_chunks)
    chunks = num_chunks or workspace.num_chunks
    _check(lib().pkv_decode_step(pool.handle, layer, _ptr(q), _ptr(k_new), _ptr(v_new),
                                 _ptr(block_table), stride, _ptr(seq_lens), rows, n_q,
                                 float(scale), _ptr(out), _ptr(workspace.tensor),
                                 workspace.nbytes, chunks, _stream(stream)), "pkv_decode_step")
    return out


class WorkspaceMQ:
    """Device scratch for the several-query calls (32 partial-state columns per
    slot), zero-filled as the library requires before first use.  The default
    chunk count depends on q_len (it selects the kernel)."""

    def __init__(self, pool: KVPool, n_q_heads: int, max_rows: int, q_len: int,
                 num_chunks: int = 0):
        if not num_chunks:
            c = ctypes.c_int(0)
            _check(lib().paged_decode_default_chunks_mq(pool.handle, n_q_heads, max_rows, q_len,
                                                        ctypes.byref(c)),
                   "paged_decode_default_chunks_mq")
            num_chunks = c.value
        self.num_chunks = num_chunks
        self.nbytes = lib().paged_decode_workspace_bytes_mq(max_rows, n_q_heads, pool.n_kv,
                                                            pool.head_dim, num_chunks)
        if self.nbytes == 0 and max_rows > 0:
            raise PkvError(1, "paged_decode_workspace_bytes_mq", "invalid sizes")
        self.tensor = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=pool.device)


def _mq_args(pool, q, block_table, seq_lens, out, workspace, num_chunks):
    rows, stride = _rows(block_table, seq_lens, pool.device)
    _need(q, torch.float32, "q", device=pool.device)
    if q.dim() != 4 or q.shape[0] != rows or q.shape[3] != pool.head_dim:
        raise ValueError("q must be [rows][q_len][n_q_heads][128]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float32, "out", q.shape, pool.device)
    if workspace is None:
        workspace = WorkspaceMQ(pool, q.shape[2], max(rows, 1), max(q.shape[1], 1), num_chunks)
    return rows, stride, out, workspace, num_chunks or workspace.num_chunks


def paged_decode_attention_mq(pool: KVPool, layer: int, q, block_table, seq_lens, scale: float,
                              out=None, workspace: WorkspaceMQ | None = None, num_chunks: int = 0,
                              stream=None):
    """Several queries per row: q [rows][q_len][n_q][128]; query j of a row of
    L tokens sits at position L - q_len + j and attends causally."""
    rows, stride, out, workspace, chunks = _mq_args(pool, q, block_table, seq_lens, out,
                                                    workspace, num_chunks)
    _check(lib().paged_decode_attention_mq(pool.handle, layer, _ptr(q), _ptr(block_table), stride,
                                           _ptr(seq_lens), rows, q.shape[1], q.shape[2],
                                           float(scale), _ptr(out), _ptr(workspace.tensor),
                                           workspace.nbytes, chunks, _stream(stream)),
           "paged_decode_attention_mq")
    return out


def decode_step_mq(pool: KVPool, layer: int, q, k_new, v_new, block_table, seq_lens,
                   scale: float, out=None, workspace: WorkspaceMQ | None = None,
                   num_chunks: int = 0, stream=None):
    """Store each row's q_len new tokens (k_new, v_new [rows][q_len][n_kv][128])
    at positions L - q_len .. L - 1, then attend (pkv_decode_step_mq)."""
    rows, stride, out, workspace, chunks = _mq_args(pool, q, block_table, seq_lens, out,
                                                    workspace, num_chunks)
    shape = (rows, q.shape[1], pool.n_kv, pool.head_dim)
    _need(k_new, torch.float32, "k_new", shape, pool.device)
    _need(v_new, torch.float32, "v_new", shape, pool.device)
    _check(lib().pkv_decode_step_mq(pool.handle, layer, _ptr(q), _ptr(k_new), _ptr(v_new),
                                    _ptr(block_table), stride, _ptr(seq_lens), rows, q.shape[1],
                                    q.shape[2], float(scale), _ptr(out), _ptr(workspace.tensor),
                                    workspace.nbytes, chunks, _stream(stream)),
           "pkv_decode_step_mq")
    return out


def paged_decode_split(pool: KVPool, layer: int, q, block_table, seq_lens, scale: float, out,
                       workspace: Workspace, stream=None):
    """The decode kernel without the in-kernel merge; partial states stay in
    the workspace for paged_decode_combine."""
    rows, stride = _rows(block_table, seq_lens, pool.device)
    _need(q, torch.float32, "q", device=pool.device)
    _need(out, torch.float32, "out", q.shape, pool.device)
    _check(lib().paged_decode_split(pool.handle, layer, _ptr(q), _ptr(block_table), stride,
                                    _ptr(seq_lens), rows, q.shape[1], float(scale), _ptr(out),
                                    _ptr(workspace.tensor), workspace.nbytes,
                                    workspace.num_chunks, _stream(stream)), "paged_decode_split")
    return out


def paged_decode_plan(seq_lens, n_kv_heads: int, bt_stride: int, num_chunks: int, stream=None,
                      window: int = 0, *, kv_dtype: int):
    """(row_page_start [rows+1], seg_first_chunk, seg_last_chunk [rows*n_kv]) int32 tensors:
    the split an attention call on a pool of KV format kv_dtype uses."""
    _need(seq_lens, torch.int32, "seq_lens")
    rows = seq_lens.shape[0]
    dev = seq_lens.device
    rps = torch.empty(rows + 1, dtype=torch.int32, device=dev)
    first = torch.empty(max(rows * n_kv_heads, 1), dtype=torch.int32, device=dev)
    last = torch.empty_like(first)
    _check(lib().paged_decode_plan(_ptr(seq_lens), rows, n_kv_heads, bt_stride, window, num_chunks,
                                   kv_dtype, _ptr(rps), _ptr(first), _ptr(last), _stream(stream)),
           "paged_decode_plan")
    return rps, first[:rows * n_kv_heads], last[:rows * n_kv_heads]


def paged_decode_combine(seq_lens, n_q_heads: int, n_kv_heads: int, bt_stride: int,
                         num_chunks: int, workspace: torch.Tensor, out, stream=None,
                         window: int = 0, *, kv_dtype: int):
    """Merge partial states held in `workspace` (layout of paged_decode_workspace_bytes) left
    by paged_decode_split on a pool of KV format kv_dtype."""
    _need(seq_lens, torch.int32, "seq_lens")
    _need(workspace, torch.uint8, "workspace")
    _need(out, torch.float32, "out")
    rows = seq_lens.shape[0]
    _check(lib().paged_decode_combine(_ptr(seq_lens), rows, n_q_heads, n_kv_heads, HEAD_DIM,
                                      bt_stride, window, num_chunks, kv_dtype, _ptr(workspace),
                                      workspace.numel(),
                                      _ptr(out), _stream(stream)), "paged_decode_combine")
    return out


class PageAllocator:
    """The library's host page allocator (include/pkv_alloc.h): page ids of a
    pool, sequences with block tables, reserve/commit/unreserve/fork/release.
    Raises PkvError with status PKV_ERR_CAPACITY (3) on overload."""

    def __init__(self, num_pages: int, max_seqs: int, max_pages_per_seq: int):
        import numpy as np  # noqa: F401  (used by batch)
        h = ctypes.c_void_p()
        _check(lib().pkv_alloc_create(ctypes.byref(h), num_pages, max_seqs, max_pages_per_seq),
               "pkv_alloc_create")
        self.handle, self.num_pages, self.max_pages_per_seq = h, num_pages, max_pages_per_seq

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.pkv_alloc_destroy(h)
            self.handle = None

    def open(self) -> int:
        s = ctypes.c_int(0)
        _check(lib().pkv_alloc_open(self.handle, ctypes.byref(s)), "pkv_alloc_open")
        return s.value

    def reserve(self, seq: int, n: int):
        _check(lib().pkv_alloc_reserve(self.handle, seq, n), "pkv_alloc_reserve")

    def commit(self, seq: int, n: int):
        _check(lib().pkv_alloc_commit(self.handle, seq, n), "pkv_alloc_commit")

    def reserve_many(self, seqs, n: int):
        import numpy as np
        ids = np.ascontiguousarray(seqs, np.int32)
        _check(lib().pkv_alloc_reserve_many(self.handle, ids.ctypes.data, len(ids), n),
               "pkv_alloc_reserve_many")

    def commit_many(self, seqs, n: int):
        import numpy as np
        ids = np.ascontiguousarray(seqs, np.int32)
        _check(lib().pkv_alloc_commit_many(self.handle, ids.ctypes.data, len(ids), n),
               "pkv_alloc_commit_many")

    def unreserve(self, seq: int, n: int):
        _check(lib().pkv_alloc_unreserve(self.handle, seq, n), "pkv_alloc_unreserve")

    def fork(self, parent: int) -> int:
        c = ctypes.c_int(0)
        _check(lib().pkv_alloc_fork(self.handle, parent, ctypes.byref(c)), "pkv_alloc_fork")
        return c.value

    def release(self, seq: int):
        _check(lib().pkv_alloc_release(self.handle, seq), "pkv_alloc_release")

    def info(self, seq: int):
        c, r, p = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
        _check(lib().pkv_alloc_seq_info(self.handle, seq, ctypes.byref(c), ctypes.byref(r),
                                        ctypes.byref(p)), "pkv_alloc_seq_info")
        return c.value, r.value, p.value

    def block_table(self, seq: int, stride: int):
        import numpy as np
        row = np.empty(stride, np.int32)
        _check(lib().pkv_alloc_block_table(self.handle, seq, row.ctypes.data, stride),
               "pkv_alloc_block_table")
        return row

    def batch(self, seqs, extra: int, stride: int):
        """(block_table int32 [rows][stride], seq_lens int32 [rows]) host arrays."""
        import numpy as np
        ids = np.ascontiguousarray(seqs, np.int32)
        bt = np.empty((len(ids), stride), np.int32)
        sl = np.empty(len(ids), np.int32)
        _check(lib().pkv_alloc_batch(self.handle, ids.ctypes.data, len(ids), extra, bt.ctypes.data,
                                     stride, sl.ctypes.data), "pkv_alloc_batch")
        return bt, sl

    def stats(self):
        f, u, s = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
        _check(lib().pkv_alloc_stats(self.handle, ctypes.byref(f), ctypes.byref(u),
                                     ctypes.byref(s)), "pkv_alloc_stats")
        return f.value, u.value, s.value

    def page_refs(self, page: int) -> int:
        r = ctypes.c_int(0)
        _check(lib().pkv_alloc_page_refs(self.handle, page, ctypes.byref(r)), "pkv_alloc_page_refs")
        return r.value

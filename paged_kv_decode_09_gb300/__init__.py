"""Paged-KV decode attention for GB300 (sm_103a).

One decode step of attention for a batch of variable-length rows whose K/V live
in a shared pool of 16-token pages reached through per-row block tables, with
GQA and f16 or q8_0 KV storage.  The compute runs in hand-written CUDA kernels
behind a C ABI (``libpkv.so``, declared in ``include/pkv.h``); the ``api``
module is a thin ctypes binding over it that takes device pointers from torch
tensors.

The binding is imported on first attribute access, so that the seeded input
generators in ``workloads`` can be used without loading the CUDA library.  If
the library is missing, every call raises: there is no CPU fallback.
"""
_API_NAMES = {
    "F16", "Q8_0", "PAGE", "PkvError", "KVPool", "kv_append", "paged_decode_attention",
    "paged_decode_plan", "paged_decode_combine", "paged_decode_split", "decode_step", "workspace_bytes",
    "default_chunks", "status_string", "library_path", "Workspace",
}


def __getattr__(name):
    if name in _API_NAMES:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)

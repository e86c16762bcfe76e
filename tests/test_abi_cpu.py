"""The C ABI without a GPU: libpkv.so builds and loads, exports every function
the headers under include/ declare, and rejects bad arguments on the host before any CUDA
call (so these calls are safe on a machine without a device)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_09_gb300 import api, build
    if not os.path.exists(build.LIB):
        if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
            pytest.skip("no nvcc to build libpkv.so")
        build.build()
    else:
        build.build()  # rebuilds only if a source is newer
    return api.lib()


def _declared():
    inc = os.path.join(ROOT, "include")
    text = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                   if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) -
                  {"if", "sizeof", "defined"})


def test_every_declared_function_is_exported(lib):
    names = _declared()
    assert {"kv_pool_create", "kv_append", "paged_decode_attention"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_pool_bytes(lib):
    # f16: 2 bytes per element; q8_0: 1 byte per element + 2 bytes per 32-element block
    assert lib.kv_pool_bytes(2, 10, 8, 128, 0, 0) == 2 * 10 * 8 * 16 * 128 * 2
    assert lib.kv_pool_bytes(2, 10, 8, 128, 0, 1) == 0
    assert lib.kv_pool_bytes(2, 10, 8, 128, 1, 0) == 2 * 10 * 8 * 16 * 128
    assert lib.kv_pool_bytes(2, 10, 8, 128, 1, 1) == 2 * 10 * 8 * 16 * 4 * 2
    assert lib.kv_pool_bytes(0, 10, 8, 128, 0, 0) == 0


def test_workspace_bytes(lib):
    chunks, rows, n_q, n_kv = 456, 8, 32, 8
    slots, G = chunks + rows * n_kv, n_q // n_kv
    flags = (slots * 2 * 4 + 255) // 256 * 256  # a counter and a ready flag per slot index
    ml = (slots * G * 2 * 4 + 255) // 256 * 256
    acc = (slots * G * 128 * 4 + 255) // 256 * 256
    assert lib.paged_decode_workspace_bytes(rows, n_q, n_kv, 128, chunks) == ml + acc + flags
    assert lib.paged_decode_workspace_bytes(rows, 30, 8, 128, chunks) == 0   # 30 % 8 != 0
    assert lib.paged_decode_workspace_bytes(rows, 32, 8, 64, chunks) == 0    # head_dim 64
    assert lib.paged_decode_workspace_bytes(rows, n_q, n_kv, 128, (1 << 24) + 1) == 0  # chunks


def test_plan_and_combine_reject_bad_split_arguments(lib):
    """The plan and the combine describe the split of one KV format: an unknown
    format, or more than 2^24 chunks, is rejected on the host."""
    fake = ctypes.c_void_p(1 << 20)
    assert lib.paged_decode_plan(fake, 1, 8, 4, 0, 16, 7, fake, fake, fake, None) == 1
    assert lib.paged_decode_plan(fake, 1, 8, 4, 0, (1 << 24) + 1, 0, fake, fake, fake,
                                 None) == 2
    assert lib.paged_decode_combine(fake, 1, 32, 8, 128, 4, 0, 16, 9, fake, 1 << 20, fake,
                                    None) == 1
    assert lib.paged_decode_combine(fake, 1, 32, 8, 128, 4, 0, (1 << 24) + 1, 0, fake, 1 << 30,
                                    fake, None) == 2


def test_host_validation_without_device(lib):
    from paged_kv_decode_09_gb300 import api
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    st = lib.kv_pool_create(ctypes.byref(h), 1, 4, 8, 128, 0, None, fake, None, None, None)
    assert st == 1 and b"null" in lib.pkv_last_error_message()
    st = lib.kv_pool_create(ctypes.byref(h), 1, 4, 8, 64, 0, fake, fake, None, None, None)
    assert st == 2
    st = lib.kv_pool_create(ctypes.byref(h), 1, 4, 8, 128, 1, fake, fake, None, None, None)
    assert st == 1  # q8_0 needs scales
    st = lib.kv_pool_create(ctypes.byref(h), 1, 4, 8, 128, 0, ctypes.c_void_p(3), fake, None,
                            None, None)
    assert st == 1  # misaligned
    # a descriptor over fake pointers: creating it touches no device memory
    assert lib.kv_pool_create(ctypes.byref(h), 2, 4, 8, 128, 0, fake, fake, None, None, None) == 0
    bt = ctypes.c_void_p(1 << 21)
    assert lib.kv_append(h, 2, fake, fake, bt, 1, bt, 1, None) == 1          # layer out of range
    assert lib.kv_append(h, 0, ctypes.c_void_p(4), fake, bt, 1, bt, 1, None) == 1  # misaligned
    assert lib.paged_decode_attention(h, 0, fake, bt, 1, bt, 1, 24, 0.1, fake, fake, 1 << 20,
                                      4, None) == 2                          # group 3
    assert lib.paged_decode_attention(h, 0, fake, bt, 1, bt, 4, 16, 0.1, fake, fake, 256,
                                      4, None) == 4                          # workspace too small
    assert lib.paged_decode_attention(h, 0, fake, bt, 1, bt, 5000, 16, 0.1, fake, fake, 256,
                                      4, None) == 2                          # too many rows
    lib.kv_pool_destroy(h)
    assert api.status_string(4) == "PKV_ERR_WORKSPACE"


def test_pool_bytes_bf16_f32(lib):
    assert lib.kv_pool_bytes(2, 10, 8, 128, 2, 0) == 2 * 10 * 8 * 16 * 128 * 2  # bf16
    assert lib.kv_pool_bytes(2, 10, 8, 128, 3, 0) == 2 * 10 * 8 * 16 * 128 * 4  # f32
    assert lib.kv_pool_bytes(2, 10, 8, 128, 3, 1) == 0
    assert lib.kv_pool_bytes(2, 10, 8, 128, 4, 0) == 0  # no such format


def test_workspace_bytes_several_queries(lib):
    # 32 partial-state columns per slot, 4 arrival counters per (row, KV head)
    chunks, rows, n_q, n_kv = 304, 8, 32, 8
    slots = chunks + rows * n_kv
    cnt = (rows * n_kv * 4 * 4 + 255) // 256 * 256
    ml = (slots * 32 * 2 * 4 + 255) // 256 * 256
    acc = (slots * 32 * 128 * 4 + 255) // 256 * 256
    assert lib.paged_decode_workspace_bytes_mq(rows, n_q, n_kv, 128, chunks) == cnt + ml + acc
    assert lib.paged_decode_workspace_bytes_mq(rows, n_q, n_kv, 128, 0) == 0


def test_several_query_host_validation_without_device(lib):
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(1 << 20)
    bt = ctypes.c_void_p(1 << 21)
    assert lib.kv_pool_create(ctypes.byref(h), 1, 4, 8, 128, 0, fake, fake, None, None, None) == 0
    args = (h, 0, fake, bt, 1, bt, 4)
    # q_len outside [1, 64] -> PKV_ERR_UNSUPPORTED, before any CUDA call
    assert lib.paged_decode_attention_mq(*args, 0, 32, 0.1, fake, fake, 1 << 24, 4, None) == 2
    assert lib.paged_decode_attention_mq(*args, 65, 32, 0.1, fake, fake, 1 << 24, 4, None) == 2
    # GQA group 3 -> PKV_ERR_UNSUPPORTED
    assert lib.paged_decode_attention_mq(*args, 2, 24, 0.1, fake, fake, 1 << 24, 4, None) == 2
    # null q -> PKV_ERR_INVALID_ARG
    assert lib.paged_decode_attention_mq(h, 0, None, bt, 1, bt, 4, 2, 32, 0.1, fake, fake,
                                         1 << 24, 4, None) == 1
    # workspace too small -> PKV_ERR_WORKSPACE
    assert lib.paged_decode_attention_mq(*args, 2, 32, 0.1, fake, fake, 256, 4, None) == 4
    # the fused step also needs its new tokens
    assert lib.pkv_decode_step_mq(h, 0, fake, None, fake, bt, 1, bt, 4, 2, 32, 0.1, fake, fake,
                                  1 << 24, 4, None) == 1
    lib.kv_pool_destroy(h)


def test_missing_library_raises(monkeypatch):
    """The product path has no fallback: without libpkv.so every call raises."""
    from paged_kv_decode_09_gb300 import api
    monkeypatch.setattr(api, "_LIB_PATH", os.path.join(ROOT, "no_such_dir", "libpkv.so"))
    monkeypatch.setattr(api, "_lib", None)
    with pytest.raises(api.PkvError, match="missing"):
        api.lib()


def test_q8_0_code_bytes():
    """q8_0 codes sit in the pool offset-binary (code + 128, the int8 byte with its top bit
    flipped): the tests' conversions between the oracle's int8 codes and the stored bytes
    invert each other, keep the codes' order, and the binding's q8_0 data tensors are bytes."""
    import numpy as np
    import torch

    from helpers import int8_codes, stored_codes
    from paged_kv_decode_09_gb300 import api
    codes = np.arange(-128, 128, dtype=np.int8)
    stored = stored_codes(codes)
    assert stored.dtype == np.uint8
    np.testing.assert_array_equal(stored.astype(np.int64), codes.astype(np.int64) + 128)
    assert np.all(np.diff(stored.astype(np.int64)) == 1)  # order kept
    np.testing.assert_array_equal(int8_codes(stored), codes)
    assert stored[codes == 0][0] == 128 and stored[codes == -127][0] == 1 and stored[codes == 127][0] == 255
    assert api._TORCH_DTYPE[api.Q8_0] == torch.uint8

"""The benchmark's algorithmic byte count, on the CPU, against values worked
out by hand: K and V of every needed token read once (2 bytes per value for
f16 and bf16, 4 for f32, 34 per 32 for q8_0), plus fp32 q and out."""
import numpy as np

import bench
from paged_kv_decode_09_gb300 import workloads as W


def _tiny(dtype):
    wl = W.draw("tiny")  # lengths {1, 17, 33, 100}, 16 q heads, 8 KV heads
    wl.cfg = W.Config(**{**wl.cfg.__dict__, "dtype": dtype})
    return wl


def test_tiny_f16_bytes_by_hand():
    # 151 tokens x 8 heads x (K + V) x 128 values x 2 bytes, plus q and out:
    # 4 rows x 16 heads x 128 x 4 bytes, twice
    assert bench.step_bytes(_tiny(W.F16)) == 151 * 8 * 2 * 128 * 2 + 2 * 4 * 16 * 128 * 4


def test_bytes_per_value_of_each_format():
    kv = 151 * 8 * 2 * 128
    qo = 2 * 4 * 16 * 128 * 4
    assert bench.step_bytes(_tiny(W.BF16)) == kv * 2 + qo
    assert bench.step_bytes(_tiny(W.F32)) == kv * 4 + qo
    assert bench.step_bytes(_tiny(W.Q8_0)) == kv * 34 // 32 + qo


def test_window_counts_only_the_attended_tokens():
    wl = _tiny(W.F16)
    # window 20: min(L, 20) per row = 1 + 17 + 20 + 20
    assert bench.attended_tokens(wl, 20) == 58
    assert bench.step_bytes(wl, 20) == 58 * 8 * 2 * 128 * 2 + 2 * 4 * 16 * 128 * 4


def test_several_queries_read_the_union_of_their_windows_once():
    wl = _tiny(W.F16)
    # q_len 4 with window 20: the first query's window starts at L - 4 + 1 - 20,
    # so a row needs min(L, 23) tokens: 1 + 17 + 23 + 23
    assert bench.attended_tokens(wl, 20, 4) == 64
    # without a window every token, once, whatever q_len; q and out grow with q_len
    assert bench.attended_tokens(wl, 0, 4) == 151
    assert bench.step_bytes(wl, 0, 4) == 151 * 8 * 2 * 128 * 2 + 2 * 4 * 4 * 16 * 128 * 4


def test_row_tokens_edges():
    assert bench.row_tokens(0) == 0
    assert bench.row_tokens(5, 100, 1) == 5
    assert bench.row_tokens(500, 100, 1) == 100
    assert bench.row_tokens(500, 100, 8) == 107
    assert bench.row_tokens(np.int32(37)) == 37


def test_source_hash_follows_code_not_comments(tmp_path):
    """A profile stays valid through edits of comments and layout, and not
    through an edit of code: string literals (inline PTX) count as code."""
    base = 'int f(int a) {  // doubles\n  return 2 * a; /* fast */\n}\nconst char* s = "x // y";\n'
    same = '/* header */\nint f(int a)\n{\n    return 2 * a;\n}\nconst char* s = "x // y";  // ptx\n'
    other = 'int f(int a) { return 3 * a; }\nconst char* s = "x // y";\n'
    lit = 'int f(int a) { return 2 * a; }\nconst char* s = "x // z";\n'
    paths = {}
    for name, text in (("base", base), ("same", same), ("other", other), ("lit", lit)):
        paths[name] = tmp_path / f"{name}.cu"
        paths[name].write_text(text)
    h = {k: bench.code_hash([str(p)]) for k, p in paths.items()}
    assert h["base"] == h["same"]
    assert h["base"] != h["other"]
    assert h["base"] != h["lit"]
    assert bench.code_only(base) == 'int f(int a) { return 2 * a; } const char* s = "x // y";'

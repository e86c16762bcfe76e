"""Seeded synthetic workloads for one paged-KV decode step.

This module only draws random numbers, lengths, page permutations and block
tables.  It holds none of the method's arithmetic (no f16 rounding, no q8_0
encoding, no attention): the tests encode context values with the oracle, the
benchmark with the library's own ``kv_append``.  It is the one module that the
CUDA path's tests and the oracle's tests share.

Workload shapes follow the engines on the pages: a shared pool of 16-token
pages with a per-row block table (tinyllm, "Known limitations": 1 GiB default
KV budget with 16-token pages; "The repository currently provides": runner-
owned page pool, block table per active sequence), GQA layer shapes of
Qwen3-0.6B (16 query / 8 KV heads, 28 layers) and Llama-3 / Qwen3 8B (32 / 8),
head_dim 128, f16 or q8_0 KV (Leone, "What ships"; LeatEngine, "Run"), and a
skewed batch whose long row sits at Qwen3-0.6B's 40,960-position limit
(tinyllm, "Known limitations").

Value recipe: q, new K/V and context K/V are N(0, 1) fp32.  Block tables are a
seeded random permutation of the pool's page ids, handed to rows in order;
unused table entries are -1.  Lengths count the attended tokens including the
token appended this step.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PAGE = 16
F16, Q8_0, BF16, F32 = 0, 1, 2, 3
DTYPE_NAMES = {F16: "f16", Q8_0: "q8_0", BF16: "bf16", F32: "f32"}


@dataclass(frozen=True)
class Config:
    name: str
    rows: int
    lengths: tuple          # ("fixed", (..)), ("uniform", lo, hi), ("skewed", long, lo, hi)
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: int
    pool: tuple             # ("fixed", pages), ("budget", bytes, layers), ("spare", frac)
    seed: int
    append: bool = True     # the step appends one token per row before attention
    model_layers: int = 1   # layers of the model shape (used to rotate pools in timing)
    description: str = ""

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


CONFIGS = {
    c.name: c for c in [
        Config("tiny", 4, ("fixed", (1, 17, 33, 100)), 16, 8, 128, F16, ("fixed", 64), 0,
               description="4 rows, seq_lens {1,17,33,100}, 16q/8kv, D=128, f16, 64-page pool"),
        Config("qwen3_0p6b_layer", 8, ("uniform", 256, 2048), 16, 8, 128, F16,
               ("budget", 1 << 30, 28), 1, model_layers=28,
               description="Qwen3-0.6B layer: 8 rows, L~U[256,2048], 16q/8kv, f16, "
                           "1 GiB pool over 28 layers"),
        Config("llama8b_f16", 8, ("uniform", 1024, 8192), 32, 8, 128, F16, ("spare", 0.10), 2,
               model_layers=32,
               description="8B layer: 8 rows, L~U[1024,8192], 32q/8kv, f16, shuffled pages"),
        Config("llama8b_q8_0", 32, ("uniform", 4096, 32768), 32, 8, 128, Q8_0,
               ("spare", 0.10), 3, model_layers=32,
               description="8B layer: 32 rows, L~U[4096,32768], 32q/8kv, q8_0, shuffled pages"),
        Config("skewed", 64, ("skewed", 40960, 16, 512), 32, 8, 128, F16, ("spare", 0.10), 4,
               model_layers=32,
               description="64 rows: one at 40960, 63 at L~U[16,512], 32q/8kv, f16, "
                           "append fused before attention"),
        # the 8B shape with bfloat16 KV (tinyllm's BF16 KV caching)
        Config("llama8b_bf16", 8, ("uniform", 1024, 8192), 32, 8, 128, BF16, ("spare", 0.10), 5,
               model_layers=32,
               description="8B layer: 8 rows, L~U[1024,8192], 32q/8kv, bf16, shuffled pages"),
        # and with fp32 KV (tinyllm's F32 KV caching)
        Config("llama8b_f32", 8, ("uniform", 1024, 8192), 32, 8, 128, F32, ("spare", 0.10), 6,
               model_layers=32,
               description="8B layer: 8 rows, L~U[1024,8192], 32q/8kv, f32, shuffled pages"),
    ]
}
CONFIG_ORDER = ["tiny", "qwen3_0p6b_layer", "llama8b_f16", "llama8b_q8_0", "skewed"]


def pages_for(length: int) -> int:
    return (max(int(length), 0) + PAGE - 1) // PAGE


def page_bytes_all_heads(cfg: Config) -> int:
    """Bytes of one page across all KV heads, K and V."""
    if cfg.dtype == Q8_0:
        per_token_head = cfg.head_dim + cfg.head_dim // 32 * 2
    else:
        per_token_head = cfg.head_dim * (4 if cfg.dtype == F32 else 2)
    return 2 * cfg.n_kv_heads * PAGE * per_token_head


@dataclass
class Workload:
    cfg: Config
    seq_lens: np.ndarray        # int32 [rows], attended tokens incl. the appended one
    num_pages: int              # pages per layer in the pool
    block_table: np.ndarray     # int32 [rows][bt_stride], -1 past each row's pages
    q: np.ndarray               # fp32 [rows][n_q][D]
    k_new: np.ndarray           # fp32 [rows][n_kv][D]
    v_new: np.ndarray           # fp32 [rows][n_kv][D]
    scale: float = field(default=0.0)

    @property
    def bt_stride(self) -> int:
        return self.block_table.shape[1]

    @property
    def rows(self) -> int:
        return self.seq_lens.shape[0]


def _draw_lengths(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    kind = cfg.lengths[0]
    if kind == "fixed":
        return np.array(cfg.lengths[1], np.int32)
    if kind == "uniform":
        _, lo, hi = cfg.lengths
        return rng.integers(lo, hi + 1, size=cfg.rows, dtype=np.int64).astype(np.int32)
    if kind == "skewed":
        _, long_len, lo, hi = cfg.lengths
        lens = rng.integers(lo, hi + 1, size=cfg.rows, dtype=np.int64).astype(np.int32)
        lens[int(rng.integers(0, cfg.rows))] = long_len
        return lens
    raise ValueError(kind)


def _pool_pages(cfg: Config, lens: np.ndarray) -> int:
    need = int(sum(pages_for(L) for L in lens))
    kind = cfg.pool[0]
    if kind == "fixed":
        return int(cfg.pool[1])
    if kind == "budget":
        _, budget, layers = cfg.pool
        return int(budget // (layers * page_bytes_all_heads(cfg)))
    if kind == "spare":
        return need + int(np.ceil(cfg.pool[1] * need))
    raise ValueError(kind)


def draw(cfg: Config | str, seed: int | None = None, lengths=None) -> Workload:
    """Draw one decode-step workload (lengths, pool size, block table, q, new K/V).

    A pool given as a byte budget may be too small for the lengths drawn; the
    lengths are then redrawn from the same stream until the rows fit."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    for _ in range(1000):
        lens = np.array(lengths, np.int32) if lengths is not None else _draw_lengths(cfg, rng)
        num_pages = _pool_pages(cfg, lens)
        if sum(pages_for(L) for L in lens) <= num_pages:
            break
        if lengths is not None:
            raise ValueError("given lengths do not fit the pool")
    else:
        raise RuntimeError("could not draw lengths that fit the pool")
    npg = [pages_for(L) for L in lens]
    stride = max(max(npg), 1)
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(lens), stride), -1, np.int32)
    at = 0
    for i, n in enumerate(npg):
        bt[i, :n] = perm[at:at + n]
        at += n
    q = rng.standard_normal((len(lens), cfg.n_q_heads, cfg.head_dim), dtype=np.float32)
    k_new = rng.standard_normal((len(lens), cfg.n_kv_heads, cfg.head_dim), dtype=np.float32)
    v_new = rng.standard_normal((len(lens), cfg.n_kv_heads, cfg.head_dim), dtype=np.float32)
    return Workload(cfg, lens, num_pages, bt, q, k_new, v_new,
                    scale=float(1.0 / np.sqrt(cfg.head_dim)))


CONTEXT_BLOCK_PAGES = 1024


def context_values(wl: Workload, layer: int = 0):
    """N(0,1) fp32 context K and V for the pool of one layer: [pages][n_kv][16][D].

    Drawn in blocks of CONTEXT_BLOCK_PAGES pages, each from a stream seeded by
    (config seed, layer, K or V, block), so every layer's pool differs and any
    block can be redrawn on its own (see context_value_blocks)."""
    ks, vs = [], []
    for _, k, v in context_value_blocks(wl, layer):
        ks.append(k)
        vs.append(v)
    return np.concatenate(ks), np.concatenate(vs)


def context_value_blocks(wl: Workload, layer: int = 0):
    """Yield (first_page, K, V) blocks of the values context_values returns."""
    cfg = wl.cfg
    for lo in range(0, wl.num_pages, CONTEXT_BLOCK_PAGES):
        hi = min(lo + CONTEXT_BLOCK_PAGES, wl.num_pages)
        shape = (hi - lo, cfg.n_kv_heads, PAGE, cfg.head_dim)
        kv = []
        for which in (1, 2):
            rng = np.random.default_rng([cfg.seed, layer, which, lo // CONTEXT_BLOCK_PAGES])
            kv.append(rng.standard_normal(shape, dtype=np.float32))
        yield lo, kv[0], kv[1]


def used_slots(wl: Workload, include_appended: bool = True) -> np.ndarray:
    """bool [num_pages][16]: pool slots that hold one of the rows' tokens.

    With include_appended=False the slot of each row's last token (the one the
    step appends) counts as unused."""
    mask = np.zeros((wl.num_pages, PAGE), bool)
    for i, L in enumerate(wl.seq_lens):
        n = int(L) if include_appended else int(L) - 1
        if n <= 0:
            continue
        t = np.arange(n)
        mask[wl.block_table[i, t // PAGE], t % PAGE] = True
    return mask


def mq_inputs(wl: Workload, q_len: int, seed: int = 0):
    """Queries and new K/V of a step with q_len new tokens per row (the
    verification of q_len - 1 drafted tokens, or a prefill chunk of q_len):
    q fp32 [rows][q_len][n_q][D], k_new and v_new fp32 [rows][q_len][n_kv][D],
    N(0, 1), from a stream seeded by (config seed, q_len, seed)."""
    cfg = wl.cfg
    rng = np.random.default_rng([cfg.seed, 1000 + q_len, seed])
    q = rng.standard_normal((wl.rows, q_len, cfg.n_q_heads, cfg.head_dim), dtype=np.float32)
    k_new = rng.standard_normal((wl.rows, q_len, cfg.n_kv_heads, cfg.head_dim), dtype=np.float32)
    v_new = rng.standard_normal((wl.rows, q_len, cfg.n_kv_heads, cfg.head_dim), dtype=np.float32)
    return q, k_new, v_new

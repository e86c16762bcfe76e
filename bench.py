#!/usr/bin/env python3
"""Benchmark one decode step of paged-KV attention on GB300.

A step is one pass of the whole hot path over one batch for one layer's pool:
pkv_decode_step, which stores each row's new token (kv_append's encoding) and
runs split-KV paged decode attention with its in-kernel merge over lengths
that include the token -- one kernel launch.  Default workload: the largest
single-GPU one, the 8B layer shape with q8_0 KV (32 rows, L ~ U[4096, 32768],
32 q / 8 KV heads, head_dim 128); the 8B f16 layer (8 rows, L ~ U[1024, 8192])
is timed the same way in the same run and reported under "also".  Steps rotate
over several layer pools whose total size is more than 4x the L2 cache, so
every step reads KV from HBM.

Metric (bytes counted per step: K and V of every attended token, q, out):
  value      KV GB/s, device-resident inputs, CUDA events on the stream
  roofline   the decode kernel's algorithmic GB/s over its mean launch-to-launch
             time in the timed region (the only kernel there), against the
             measured HBM copy bandwidth
  e2e        the same metric through the C ABI with the step's inputs copied
             from pinned host memory and the output copied back, every step
  cpu_baseline  the FP64 CPU oracle on a bounded sample of the same batch

`--impl reference` times the oracle alone on the host cores (the same metric).
Under torchrun each rank runs its own replica of the batch (no collective on
the data path); times are the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 126 * 2**20
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="llama8b_q8_0",
                   help="the workload of the reported value (default: the largest, 8B q8_0)")
    p.add_argument("--also", default="llama8b_f16",
                   help="comma-separated workloads timed the same way after the main one and\n"
                        "reported under \"also\" (\"\" for none)")
    p.add_argument("--lead-seconds", type=float, default=0.25,
                   help="untimed steps run straight into the timed ones (clock samples under\n"
                        "load; the start event fires on a busy stream)")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=0, help="layer pools to rotate (0: auto)")
    p.add_argument("--chunks", type=int, default=0, help="work chunks (0: one per resident CTA)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU baseline budget")
    p.add_argument("--window", type=int, default=0,
                   help="sliding window of every layer (0: none); bytes count attended tokens")
    p.add_argument("--no-graph", action="store_true",
                   help="skip the CUDA-graph replay timing (shorter runs under a profiler)")
    p.add_argument("--q-len", type=int, default=1,
                   help="new tokens (queries) per row: > 1 times the several-query step")
    p.add_argument("--kernel", choices=["step", "append", "split_combine", "plan", "alloc"],
                   default="step",
                   help="step: the decode step (the benchmark); the others run --steps calls of\n"
                        "one other entry point on the workload and print its mean call time\n"
                        "(for profiling those kernels alone; not the benchmark metric);\n"
                        "alloc: the host page allocator's work for one decode step of 256\n"
                        "sequences (reserve 1, batch tables, commit 1)")
    return p.parse_args()


# ------------------------------------------------------------ distributed ----
def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x across ranks (x itself at world size 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ sizes ----
def read_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bytes_per_value(dtype: int) -> float:
    """Stored bytes per K or V value: q8_0 34 per 32, f32 4, f16 and bf16 2."""
    return 34.0 / 32.0 if dtype == 1 else 4.0 if dtype == 3 else 2.0


def row_tokens(L: int, window=0, q_len=1) -> int:
    """Tokens a row of L tokens needs in one call: all L, or with a window W the
    union of its q_len queries' windows, the last min(L, W + q_len - 1)."""
    return min(L, window + q_len - 1) if window > 0 else L


def attended_tokens(wl, window=0, q_len=1) -> int:
    """Tokens read once by one decode call, summed over rows (see row_tokens)."""
    return int(sum(row_tokens(int(L), window, q_len) for L in wl.seq_lens))


def step_bytes(wl, window=0, q_len=1) -> int:
    """Algorithmic bytes of one decode call: K and V of every needed token read
    once (bytes_per_value per element), q and out (fp32, q_len queries per row)."""
    cfg = wl.cfg
    per_elem = bytes_per_value(cfg.dtype)
    kv = attended_tokens(wl, window, q_len) * cfg.n_kv_heads * cfg.head_dim * 2 * per_elem
    qo = 2 * wl.rows * q_len * cfg.n_q_heads * cfg.head_dim * 4
    return int(kv + qo)


KERNEL_SOURCES = {  # the files each decode kernel is compiled from (besides headers of the ABI)
    "paged_decode_kernel": ("decode.cu", "decode_common.cuh", "pkv_device.cuh"),
    "paged_decode_mq_kernel": ("decode_mq.cu", "decode_common.cuh", "pkv_device.cuh"),
    "paged_decode_mqt_kernel": ("decode_mq.cu", "decode_common.cuh", "pkv_device.cuh"),
    "paged_decode_mqtc_kernel": ("decode_mqtc.cu", "decode_common.cuh", "pkv_device.cuh"),
}


_TOKEN = re.compile(r'"(?:\\.|[^"\\\n])*"|/\*.*?\*/|//[^\n]*', re.S)


def code_only(text: str) -> str:
    """A C++/CUDA source without its comments and with its whitespace collapsed
    (string literals kept as they are): what decides the compiled kernel."""
    stripped = _TOKEN.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return " ".join(stripped.split())


def code_hash(paths) -> str:
    """Hash of the code of these files (comments and layout ignored)."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def kernel_source_hash(kernel: str) -> str:
    """Identifies the code a decode kernel is compiled from: a profile taken on
    it stays valid through edits of comments, not of code."""
    src = os.path.join(ROOT, "paged_kv_decode_09_gb300", "csrc")
    return code_hash(os.path.join(src, name) for name in KERNEL_SOURCES[kernel])


def profile_traffic(workload: str, kernel: str = "paged_decode_kernel", q_len: int = 1):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if it was taken on the current kernel source (else None)."""
    suffix = f"_q{q_len}" if q_len > 1 else ""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}{suffix}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_sha256_16:\s*([0-9a-f]{16})", text)
    if not m or m.group(2) != kernel_source_hash(kernel):
        return None
    return int(m.group(1))


# ------------------------------------------------------------- our kernels ----
def fill_pool(api, pool, layers, seed):
    """Fill every slot of every layer with N(0,1) values stored by the
    library's own kv_append (one pseudo-row per slot)."""
    import torch
    g = torch.Generator(device=pool.device).manual_seed(seed)
    per = 2048
    for layer in range(layers):
        for p0 in range(0, pool.num_pages, per):
            p1 = min(p0 + per, pool.num_pages)
            rows = (p1 - p0) * 16
            r = torch.arange(rows, device=pool.device, dtype=torch.int32)
            bt = (p0 + r // 16).to(torch.int32).reshape(rows, 1).contiguous()
            sl = (r % 16 + 1).to(torch.int32).contiguous()
            k = torch.randn(rows, pool.n_kv, 128, device=pool.device, generator=g)
            v = torch.randn(rows, pool.n_kv, 128, device=pool.device, generator=g)
            api.kv_append(pool, layer, k, v, bt, sl)
    torch.cuda.synchronize()


class StepSetup:
    """One workload's pool, inputs and decode-step call, ready to time."""

    def __init__(self, args, name, rank, dev):
        import numpy as np
        import torch

        from paged_kv_decode_09_gb300 import api
        from paged_kv_decode_09_gb300 import workloads as W

        self.torch, self.api, self.W = torch, api, W
        wl = W.draw(name)
        cfg = wl.cfg
        self.wl, self.cfg = wl, cfg
        layer_bytes = 2 * api.KVPool.bytes(1, wl.num_pages, cfg.n_kv_heads, cfg.dtype, 0) + \
            2 * api.KVPool.bytes(1, wl.num_pages, cfg.n_kv_heads, cfg.dtype, 1)
        self.layer_bytes = layer_bytes
        layers = args.layers or max(2, min(cfg.model_layers, -(-4 * L2_BYTES // layer_bytes)))
        self.layers = layers
        pool = api.KVPool(layers, wl.num_pages, cfg.n_kv_heads, cfg.dtype, device=dev)
        fill_pool(api, pool, layers, seed=1234 + rank)
        for layer in range(layers):
            pool.set_window(layer, args.window)
        self.pool = pool

        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        QL = args.q_len
        self.QL = QL
        if QL > 1:  # verification / chunk step: q_len new tokens per row
            hq_np, hk_np, hv_np = W.mq_inputs(wl, QL)
            q, k_new, v_new = t(hq_np), t(hk_np), t(hv_np)
            ws = api.WorkspaceMQ(pool, cfg.n_q_heads, wl.rows, QL, args.chunks)
            cols = QL * cfg.group  # (query, head) columns; the kernel's pass width follows them
            if cfg.dtype == W.F32 or cols <= (4 if cfg.dtype == W.BF16 else 8):
                width = min(cols, 8)
                kname = "paged_decode_mq_kernel"  # the warps of a CTA read different pages
            elif cfg.dtype == W.F16 or (cfg.dtype == W.BF16 and cols > 8):
                width = 32  # blocks of 8 pages on the tensor cores, passes of 32
                kname = "paged_decode_mqtc_kernel"
            else:  # teams of 2 or 4 warps share every page
                if cfg.dtype == W.BF16:
                    width = 8 if cols <= 8 else 16
                else:  # q8_0: two or four warps of 8 columns
                    width = 16 if cols <= 16 else 32
                kname = "paged_decode_mqt_kernel"
            passes = -(-QL // max(1, width // cfg.group))
        else:
            q, k_new, v_new = t(wl.q), t(wl.k_new), t(wl.v_new)
            ws = api.Workspace(pool, cfg.n_q_heads, wl.rows, args.chunks)
            passes = 1
            kname = "paged_decode_kernel"
        self.passes, self.kname, self.ws = passes, kname, ws
        bt, sl = t(wl.block_table), t(wl.seq_lens)
        out = torch.empty_like(q)
        self.q, self.k_new, self.v_new, self.bt, self.sl, self.out = q, k_new, v_new, bt, sl, out
        self.L = L = api.lib()
        self.stream = torch.cuda.current_stream(dev)
        self.sp = ctypes.c_void_p(self.stream.cuda_stream)
        P = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
        self.a_q, self.a_k, self.a_v, self.a_bt, self.a_sl, self.a_out, self.a_ws = map(
            P, (q, k_new, v_new, bt, sl, out, ws.tensor))
        self.scale = ctypes.c_float(wl.scale)
        self.nbytes = step_bytes(wl, args.window, QL)
        self.tokens = attended_tokens(wl, args.window, QL)

    def chk(self, st, what):
        if st:
            raise self.api.PkvError(st, what, self.L.pkv_last_error_message().decode())

    def call(self, layer, pq, pk, pv, pbt, psl, pout, on):
        """One decode step through the C ABI (the step's inputs at these pointers)."""
        L, wl, cfg, ws = self.L, self.wl, self.cfg, self.ws
        H, R, NQ, S, CH = self.pool.handle, wl.rows, cfg.n_q_heads, wl.bt_stride, ws.num_chunks
        if self.QL > 1:
            self.chk(L.pkv_decode_step_mq(H, layer, pq, pk, pv, pbt, S, psl, R, self.QL, NQ,
                                          self.scale, pout, self.a_ws, ws.nbytes, CH, on),
                     "pkv_decode_step_mq")
        else:
            self.chk(L.pkv_decode_step(H, layer, pq, pk, pv, pbt, S, psl, R, NQ, self.scale, pout,
                                       self.a_ws, ws.nbytes, CH, on), "pkv_decode_step")

    def step(self, layer, on=None):
        self.call(layer, self.a_q, self.a_k, self.a_v, self.a_bt, self.a_sl, self.a_out,
                  self.sp if on is None else on)

    def time_steps(self, K, warmup, world, local, lead_s):
        """Mean time of K back-to-back steps (max over ranks), with the clocks
        sampled meanwhile.

        Untimed lead steps run first, for lead_s seconds, straight into the
        timed ones: the clock sampler sees the GPU under this load, and the
        start event fires on a busy stream, so the timed region holds the K
        steps and not the latency of the first launch.  The two events are
        the only ones in the region: an event between launches would add its
        own gap and break the programmatic dependent launch."""
        torch = self.torch
        for w in range(warmup):
            self.step(w % self.layers)
        torch.cuda.synchronize()
        assert self.pool.read_status() == 0, "device status word set during warm-up"
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(local)
        barrier(world)
        torch.cuda.synchronize()
        clocks.start()
        n = 0
        t_end = time.perf_counter() + lead_s
        while n < 3 or time.perf_counter() < t_end:
            self.step(n % self.layers)
            n += 1
        e0.record(self.stream)
        for s in range(K):
            self.step((n + s) % self.layers)
        e1.record(self.stream)
        torch.cuda.synchronize()
        clock_info = clocks.stop()
        barrier(world)
        total_ms = max_over_ranks(e0.elapsed_time(e1), world)
        assert self.pool.read_status() == 0, "device status word set during the timed steps"
        return total_ms, clock_info, n

    def roofline(self, launch_ms, peak, peak_src, window):
        W = self.W
        achieved = self.nbytes / (launch_ms / 1e3) / 1e9
        return {
            "bound": "hbm", "kernel": f"{self.kname}<{W.DTYPE_NAMES[self.cfg.dtype]}>, G={self.cfg.group}",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (copy bandwidth)",
            # DRAM bytes of one launch (one pass: a step of the several-query
            # kernel is `launches_per_step` of them)
            "traffic": None if window else profile_traffic(self.cfg.name, self.kname, self.QL),
            "mean_launch_us": round(launch_ms * 1e3, 3),
            "timing": "events around the K back-to-back launches of the timed region, "
                      "after untimed lead steps on the same stream",
        }

    def config(self, args, world):
        wl, cfg, W, ws = self.wl, self.cfg, self.W, self.ws
        QL, passes = self.QL, self.passes
        return {
            "workload": cfg.name, "description": cfg.description, "rows": wl.rows,
            "n_q_heads": cfg.n_q_heads, "n_kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim,
            "kv_dtype": W.DTYPE_NAMES[cfg.dtype], "tokens_attended": self.tokens,
            "pages_per_layer": wl.num_pages, "layers_rotated": self.layers,
            "l2": f"inputs larger than L2: {self.layers} layer pools of "
                  f"{self.layer_bytes / 2**20:.0f} MiB rotated (> 4x the 126 MiB L2)",
            "chunks": ws.num_chunks, "bytes_per_step": self.nbytes,
            "parallelism": f"replicas x{world}",
            **({"window": args.window} if args.window else {}),
            **({"q_len": QL, "launches_per_step": passes} if QL > 1 else {}),
            "workspace_bytes": ws.nbytes,
            # traffic beyond the algorithmic bytes and not counted in them: the
            # block-table entries of the attended pages (once per launch; a
            # window that does not start on a page boundary touches one more
            # page), and at most every workspace byte written once and read once
            "uncounted_bytes": {"block_table": 4 * passes * int(sum(
                                    W.pages_for(row_tokens(int(L), args.window, QL))
                                    + (1 if args.window and int(L) else 0)
                                    for L in wl.seq_lens)),
                                "workspace_max": 2 * ws.nbytes},
        }


def run_ours(args, rank, world, local):
    import torch

    from paged_kv_decode_09_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, peak_src = read_peak()
    st = StepSetup(args, args.workload, rank, dev)
    wl, cfg = st.wl, st.cfg
    K = args.steps
    total_ms, clock_info, lead = st.time_steps(K, args.warmup, world, local, args.lead_seconds)
    # the only kernel in the timed region: a step is `passes` back-to-back
    # launches of it; the roofline takes the step (all passes) as the unit
    launch_ms = total_ms / K
    graph = None if args.no_graph else graph_timing(torch, dev, st.step, st.layers)
    e2e = e2e_timing(st, K, args.warmup, world, dev)

    nbytes = st.nbytes
    step_s = total_ms / 1e3 / K
    value = world * nbytes / step_s / 1e9
    result = {
        "metric": "paged decode-attn KV GB/s & % of GB300 HBM peak; rows*tokens/s at 1 GPU",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": W.DTYPE_NAMES[cfg.dtype] + " KV, f32 compute",
        "data": "synthetic: seeded lengths/block tables/q; KV N(0,1) stored by kv_append",
        "config": {**st.config(args, world), "lead_steps": lead},
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "rows_tokens_per_s": round(world * st.tokens / step_s, 1),
        "rows_per_s": round(world * wl.rows / step_s, 1),
        "roofline": st.roofline(launch_ms, peak, peak_src, args.window),
        "e2e": e2e,
        "gpu_launches": K * st.passes,
        "graph": graph,
        "clocks": clock_info,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, st.pool, args.cpu_seconds, args.window,
                                              args.q_len, st.q.cpu().numpy())
    # The other workloads of the 70% bar (the 8B f16 layer beside the 8B q8_0
    # headline), each timed the same way and reported with its own roofline.
    also = {}
    for name in [x for x in args.also.split(",") if x and x != args.workload]:
        del st
        torch.cuda.empty_cache()
        st = StepSetup(args, name, rank, dev)
        t_ms, clk, n_lead = st.time_steps(K, args.warmup, world, local, args.lead_seconds)
        g = None if args.no_graph else graph_timing(torch, dev, st.step, st.layers)
        s_ = t_ms / 1e3 / K
        v_ = world * st.nbytes / s_ / 1e9
        also[name] = {
            "value": round(v_, 2), "unit": "GB/s", "steps": K, "ms_per_step": round(t_ms / K, 6),
            "dtype": W.DTYPE_NAMES[st.cfg.dtype] + " KV, f32 compute",
            "config": {**st.config(args, world), "lead_steps": n_lead},
            "frac_of_hbm_peak": round(v_ / world / peak, 4),
            "rows_tokens_per_s": round(world * st.tokens / s_, 1),
            "roofline": st.roofline(t_ms / K, peak, peak_src, args.window),
            "gpu_launches": K * st.passes, "graph": g, "clocks": clk,
        }
        result["gpu_launches"] += K * st.passes
    if also:
        result["also"] = also
    return result


def e2e_timing(st, K, warmup, world, dev):
    """The same metric end to end through the C ABI: every step copies its
    inputs from pinned host memory and its output back.  As a serving loop
    would, the inputs sit in one packed buffer (one copy per step each way) and
    are double-buffered: the copy of step s + 1's inputs (on a copy stream)
    overlaps step s's kernel, the copy of step s's output (on another)
    overlaps step s + 1's."""
    torch = st.torch
    parts = (st.q, st.k_new, st.v_new, st.bt, st.sl)
    offs, size = [], 0
    for x in parts:
        offs.append(size)
        size += -(-x.numel() * x.element_size() // 256) * 256  # 256-byte aligned parts
    hpack = torch.empty(size, dtype=torch.uint8).pin_memory()
    for x, o in zip(parts, offs):
        hpack[o:o + x.numel() * x.element_size()].copy_(x.cpu().contiguous().view(-1).view(torch.uint8))
    dpack = [torch.empty(size, dtype=torch.uint8, device=dev) for _ in range(2)]
    douts = [torch.empty_like(st.out) for _ in range(2)]
    hout = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in parts)
    d2h = st.out.numel() * st.out.element_size()
    ptrs = [[ctypes.c_void_p(d.data_ptr() + o) for o in offs] for d in dpack]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # The copies and the stream edges go straight to the CUDA driver (the
    # per-step Python cost of torch's wrappers would otherwise bound the loop).
    cu = ctypes.CDLL("libcuda.so.1")
    cu.cuMemcpyHtoDAsync_v2.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    cu.cuMemcpyDtoHAsync_v2.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p]
    cu.cuEventRecord.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    cu.cuStreamWaitEvent.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    cu.cuEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint]

    def cu_ok(r, what):
        if r != 0:
            raise RuntimeError(f"{what}: CUDA driver error {r}")

    def new_event():
        e_ = ctypes.c_void_p()
        cu_ok(cu.cuEventCreate(ctypes.byref(e_), 2), "cuEventCreate")  # no timing
        return e_

    ev_in, ev_done, ev_out = ([new_event() for _ in range(2)] for _ in range(3))
    stream = st.stream
    c_st, c_h2d, c_d2h = (ctypes.c_void_p(x.cuda_stream) for x in (stream, s_h2d, s_d2h))
    hsrc = ctypes.c_void_p(hpack.data_ptr())
    dsts = [d.data_ptr() for d in dpack]
    oh = [ctypes.c_void_p(x.data_ptr()) for x in hout]
    po_ = [ctypes.c_void_p(x.data_ptr()) for x in douts]
    od = [x.data_ptr() for x in douts]

    def e2e_step(s_, layer):
        b = s_ % 2
        if s_ >= 2:
            cu.cuStreamWaitEvent(c_h2d, ev_done[b], 0)  # step s - 2 has read this buffer
        cu_ok(cu.cuMemcpyHtoDAsync_v2(dsts[b], hsrc, size, c_h2d), "H2D")
        cu.cuEventRecord(ev_in[b], c_h2d)
        cu.cuStreamWaitEvent(c_st, ev_in[b], 0)
        if s_ >= 2:
            cu.cuStreamWaitEvent(c_st, ev_out[b], 0)  # step s - 2's output left this buffer
        pq, pk, pv, pbt, psl = ptrs[b]
        st.call(layer, pq, pk, pv, pbt, psl, po_[b], st.sp)
        cu.cuEventRecord(ev_done[b], c_st)
        cu.cuStreamWaitEvent(c_d2h, ev_done[b], 0)
        cu_ok(cu.cuMemcpyDtoHAsync_v2(oh[b], od[b], d2h, c_d2h), "D2H")
        cu.cuEventRecord(ev_out[b], c_d2h)

    Ke = min(K, 2000)
    for w in range(warmup):
        e2e_step(w, w % st.layers)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    h0 = time.perf_counter()
    for s_ in range(Ke):
        e2e_step(s_, s_ % st.layers)
    host_us = (time.perf_counter() - h0) * 1e6 / Ke  # issue time per step on the host
    stream.wait_stream(s_d2h)  # the last output is on the host
    f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world)
    assert st.pool.read_status() == 0, "device status word set during the end-to-end steps"
    torch.testing.assert_close(hout[(Ke - 1) % 2], douts[(Ke - 1) % 2].cpu(), rtol=0, atol=0)
    return {"value": round(world * st.nbytes / (e2e_ms / 1e3 / Ke) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
            "ms_per_step": round(e2e_ms / Ke, 6),
            "copies": "one packed pinned H2D and one D2H per step, double-buffered on two "
                      "copy streams overlapping the kernels",
            "host_issue_us_per_step": round(host_us, 2)}


def graph_timing(torch, dev, step, layers, calls=20, replays=50):
    """Steps captured as a CUDA graph of `calls` calls (rotating the layer
    pools as the timed loop does), replayed `replays` times with events
    around each replay: per-call median, p10 and p90 in microseconds."""
    import numpy as np
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.graph(g, stream=cap):
            on = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
            for c in range(calls):
                step(c % layers, on)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(replays)]
        for e0, e1 in ev:
            e0.record()
            g.replay()
            e1.record()
        torch.cuda.synchronize()
        per_call = np.array([e0.elapsed_time(e1) * 1e3 / calls for e0, e1 in ev])
        return {"calls_per_graph": calls, "replays": replays,
                "median_us_per_call": round(float(np.median(per_call)), 3),
                "p10_us_per_call": round(float(np.percentile(per_call, 10)), 3),
                "p90_us_per_call": round(float(np.percentile(per_call, 90)), 3)}
    except Exception as exc:  # reported, not fatal: the event-timed loop is the measurement
        return {"error": f"{type(exc).__name__}: {str(exc)[:160]}"}


def run_alloc(args):
    """Host page allocator: per decode step, reserve one token for each of 256
    sequences, write the batch's block tables and lengths, commit the token."""
    from paged_kv_decode_09_gb300 import api
    rows, stride = 256, 2048
    a = api.PageAllocator(rows * stride, rows, stride)
    seqs = []
    for s in range(rows):
        seqs.append(a.open())
        a.reserve(seqs[-1], 4096)
        a.commit(seqs[-1], 4096)
    import numpy as np
    ids = np.arange(rows, dtype=np.int32)
    bt = np.empty((rows, stride), np.int32)
    sl = np.empty(rows, np.int32)
    L = api.lib()

    def step():
        L.pkv_alloc_reserve_many(a.handle, ids.ctypes.data, rows, 1)
        L.pkv_alloc_batch(a.handle, ids.ctypes.data, rows, 1, bt.ctypes.data, stride,
                          sl.ctypes.data)
        L.pkv_alloc_commit_many(a.handle, ids.ctypes.data, rows, 1)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    return {"kernel": "alloc", "rows": rows, "bt_stride": stride, "calls": args.steps,
            "mean_step_us": round(dt * 1e6, 2),
            "note": "host allocator work per decode step through ctypes; not the benchmark metric"}


def run_kernel(args, local):
    """--steps calls of one entry point other than the decode step, timed with
    events on the stream: kv_append (new K/V of every row), paged_decode_split
    followed by paged_decode_combine, or paged_decode_plan."""
    import numpy as np
    import torch

    from paged_kv_decode_09_gb300 import api
    from paged_kv_decode_09_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.draw(args.workload)
    cfg = wl.cfg
    layers = 2
    pool = api.KVPool(layers, wl.num_pages, cfg.n_kv_heads, cfg.dtype, device=dev)
    if args.kernel == "split_combine":
        fill_pool(api, pool, layers, seed=1234)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    q, k_new, v_new = t(wl.q), t(wl.k_new), t(wl.v_new)
    bt, sl = t(wl.block_table), t(wl.seq_lens)
    out = torch.empty_like(q)
    ws = api.Workspace(pool, cfg.n_q_heads, wl.rows, args.chunks)

    def call(i):
        if args.kernel == "append":
            api.kv_append(pool, i % layers, k_new, v_new, bt, sl)
        elif args.kernel == "split_combine":
            api.paged_decode_split(pool, i % layers, q, bt, sl, wl.scale, out, ws)
            api.paged_decode_combine(sl, cfg.n_q_heads, cfg.n_kv_heads, wl.bt_stride,
                                     ws.num_chunks, ws.tensor, out, kv_dtype=cfg.dtype)
        else:
            api.paged_decode_plan(sl, cfg.n_kv_heads, wl.bt_stride, ws.num_chunks,
                                  kv_dtype=cfg.dtype)

    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        call(i)
    e1.record()
    torch.cuda.synchronize()
    assert pool.read_status() == 0
    return {"kernel": args.kernel, "workload": cfg.name, "calls": args.steps,
            "mean_call_us": round(e0.elapsed_time(e1) * 1e3 / max(1, args.steps), 3),
            "note": "per-entry-point timing for profiling; not the benchmark metric"}


def cpu_baseline(wl, pool, budget_s, window=0, q_len=1, q=None):
    """The FP64 oracle, as it stands, on a bounded sample of the batch of layer
    0: on all the host's cores (the reported value) and on one core."""
    import numpy as np
    import torch

    import oracle as O
    cfg = wl.cfg
    if cfg.dtype == 3:  # f32 values
        kd, vd = pool.k_data[0].cpu().numpy(), pool.v_data[0].cpu().numpy()
        ks = vs = None
    elif cfg.dtype != 1:  # 16-bit patterns (f16, bf16)
        kd = pool.k_data[0].cpu().view(torch.int16).numpy().view(np.uint16)
        vd = pool.v_data[0].cpu().view(torch.int16).numpy().view(np.uint16)
        ks = vs = None
    else:  # q8_0 codes: the pool stores them offset-binary (code + 128)
        kd = (pool.k_data[0].cpu().numpy().view(np.uint8) ^ np.uint8(0x80)).view(np.int8)
        vd = (pool.v_data[0].cpu().numpy().view(np.uint8) ^ np.uint8(0x80)).view(np.int8)
        ks = pool.k_scales[0].cpu().view(torch.int16).numpy().view(np.uint16)
        vs = pool.v_scales[0].cpu().view(torch.int16).numpy().view(np.uint16)
    per_elem = bytes_per_value(cfg.dtype)

    def sample(budget):
        # shortest rows first; the batch is cycled until the budget is spent,
        # stopping on a whole pass once half of it is
        order = np.argsort(wl.seq_lens)
        done, secs, rows = 0, 0.0, 0
        for n in range(1 << 30):
            if n >= len(order) and n % len(order) == 0 and secs > 0.5 * budget:
                break
            i = order[n % len(order)]
            t0 = time.perf_counter()
            if q_len > 1:
                O.decode_attention_mq(cfg.dtype, q[i:i + 1], kd, vd, ks, vs,
                                      wl.block_table[i:i + 1], wl.seq_lens[i:i + 1], wl.num_pages,
                                      cfg.n_kv_heads, wl.scale, window=window)
            else:
                O.decode_attention(cfg.dtype, wl.q[i:i + 1], kd, vd, ks, vs,
                                   wl.block_table[i:i + 1], wl.seq_lens[i:i + 1], wl.num_pages,
                                   cfg.n_kv_heads, wl.scale, window=window)
            secs += time.perf_counter() - t0
            rows += 1
            done += row_tokens(int(wl.seq_lens[i]), window, q_len)
            if secs > budget:
                break
        nbytes = done * cfg.n_kv_heads * cfg.head_dim * 2 * per_elem + \
            2 * rows * q_len * cfg.n_q_heads * 128 * 4
        what = (f"{rows} of {wl.rows} rows" if rows < wl.rows
                else f"{rows / wl.rows:g} passes over the {wl.rows} rows")
        return nbytes / secs / 1e9, done / secs, f"{what} ({done} attended tokens), {secs:.1f} s"

    cores = O.num_threads()
    value, tps, text = sample(0.7 * budget_s)
    O.set_num_threads(1)
    try:
        value1, tps1, text1 = sample(0.3 * budget_s)
    finally:
        O.set_num_threads(cores)
    return {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{text} of one layer, attention only",
            "rows_tokens_per_s": round(tps, 1),
            "single_core": {"value": round(value1, 4), "unit": "GB/s", "cores": 1,
                            "sample": f"{text1} of one layer, attention only",
                            "rows_tokens_per_s": round(tps1, 1)},
            "cpu": cpu_model()}


def cpu_model() -> str:
    """The host CPU's model name (or architecture) as the system reports it."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# ------------------------------------------------------------- reference ----
def encoded_pool(O, W, wl, layer=0):
    """The oracle's encoding of one layer's context values, (k_data, v_data,
    k_scales, v_scales), built block by block so that the fp32 values of only
    one block are held at a time."""
    import numpy as np
    kd = vd = ks = vs = None
    for lo, k, v in W.context_value_blocks(wl, layer):
        kb, ksb = O.encode_pool(wl.cfg.dtype, k)
        vb, vsb = O.encode_pool(wl.cfg.dtype, v)
        if kd is None:
            kd = np.empty((wl.num_pages,) + kb.shape[1:], kb.dtype)
            vd = np.empty_like(kd)
            if ksb is not None:
                ks = np.empty((wl.num_pages,) + ksb.shape[1:], ksb.dtype)
                vs = np.empty_like(ks)
        hi = lo + kb.shape[0]
        kd[lo:hi], vd[lo:hi] = kb, vb
        if ksb is not None:
            ks[lo:hi], vs[lo:hi] = ksb, vsb
    return kd, vd, ks, vs


def run_reference(args):
    """The FP64 oracle on the host cores, each step one row of the batch."""
    import numpy as np

    import oracle as O
    from paged_kv_decode_09_gb300 import workloads as W
    wl = W.draw(args.workload)
    cfg = wl.cfg
    kd, vd, ks, vs = encoded_pool(O, W, wl)
    order = np.argsort(wl.seq_lens)
    G = cfg.group
    # A step is one row, or (when K rows would overrun the time budget) every
    # G-th query head of one row, i.e. one query head per KV head: 1/G of the
    # row's work, with the same per-head computation.
    heads = slice(None)
    QL = args.q_len
    q_mq = W.mq_inputs(wl, QL)[0] if QL > 1 else None

    def one(i):
        if q_mq is not None:
            O.decode_attention_mq(cfg.dtype, q_mq[i:i + 1, :, heads], kd, vd, ks, vs,
                                  wl.block_table[i:i + 1], wl.seq_lens[i:i + 1], wl.num_pages,
                                  cfg.n_kv_heads, wl.scale, window=args.window)
            return
        q = wl.q[i:i + 1, heads]
        O.decode_attention(cfg.dtype, q, kd, vd, ks, vs, wl.block_table[i:i + 1],
                           wl.seq_lens[i:i + 1], wl.num_pages, cfg.n_kv_heads, wl.scale,
                           window=args.window)

    per_elem = bytes_per_value(cfg.dtype)

    def tokens_of(i):
        return row_tokens(int(wl.seq_lens[i]), args.window, QL)

    def row_bytes(i, frac):
        return frac * (tokens_of(i) * cfg.n_kv_heads * cfg.head_dim * 2 * per_elem
                       + 2 * QL * cfg.n_q_heads * 128 * 4)

    mid = order[len(order) // 2]
    t0 = time.perf_counter()
    one(mid)
    t_row = time.perf_counter() - t0
    frac, sample = 1.0, "one row of the batch per step, cycling shortest first"
    if (args.steps + args.warmup) * t_row > 150.0 and G > 1:
        heads, frac = slice(None, None, G), 1.0 / G
        sample = (f"every {G}th query head (one per KV head) of one row per step, cycling "
                  f"shortest first: 1/{G} of a row's work")
    for w in range(args.warmup):
        one(order[w % wl.rows])
    nbytes, tokens, secs = 0.0, 0, 0.0
    for s in range(args.steps):
        i = order[s % wl.rows]
        t0 = time.perf_counter()
        one(i)
        secs += time.perf_counter() - t0
        nbytes += row_bytes(i, frac)
        tokens += frac * tokens_of(i)
    value = nbytes / secs / 1e9
    return {
        "impl": "reference",
        "metric": "paged decode-attn KV GB/s & % of GB300 HBM peak; rows*tokens/s at 1 GPU",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic: same seeded workload, pool encoded by the oracle",
        "config": {"workload": cfg.name, "description": cfg.description, "sample": sample,
                   **({"window": args.window} if args.window else {}),
                   **({"q_len": QL} if QL > 1 else {})},
        "rows_tokens_per_s": round(tokens / secs, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": O.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.impl == "reference":
        # host-only: rank 0 alone times the oracle, the other ranks exit at once
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.kernel == "alloc":
        print(json.dumps(run_alloc(args)), flush=True)
        return
    if args.kernel != "step":
        print(json.dumps(run_kernel(args, int(os.environ.get("LOCAL_RANK", "0")))), flush=True)
        return
    rank, world, local = dist_init(args)
    result = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()

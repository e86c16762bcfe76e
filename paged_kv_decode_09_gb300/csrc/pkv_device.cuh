// pkv_device.cuh — device helpers shared by the kernels of libpkv.so:
// inline-PTX wrappers for mbarriers and 1-D bulk async copies (global ->
// shared), a bounded barrier wait, and the per-CTA plan (row page offsets and
// the chunk a unit belongs to).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pkv.h"

namespace pkv {

constexpr int kPage = PKV_PAGE_TOKENS;  // tokens per page
constexpr int kD = PKV_HEAD_DIM;        // head_dim handled by the kernels
constexpr int kQBlock = PKV_Q8_BLOCK;   // q8_0 block along head_dim
constexpr unsigned kFull = 0xffffffffu;

// A wait on a shared-memory barrier gives up after this long (the whole
// decode of a batch takes well under a millisecond).
constexpr unsigned long long kWaitLimitNs = PKV_DEFAULT_WAIT_NS;  // ~1.07 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete.  Returns
// false, without waiting further, once *abort is set or after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// 1-D bulk async copy global -> shared, completing `bytes` of transaction on
// `bar`, with an L2 eviction-priority hint.  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 3-D tiled bulk tensor copy global -> shared through a tensor map (the
// map's swizzle applies), completing its bytes on `bar`, with an L2 hint.
// `tmap` is the generic address of a CUtensorMap kernel parameter; x must be
// a multiple of 16 bytes' worth of elements and dst aligned to the swizzle
// atom (1024 bytes for the 128-byte swizzle).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Fetch a tensor map (the generic address of a kernel parameter) into the
// cache the tensor copies read it from, ahead of the first copy.
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 4-D tiled bulk tensor copy global -> shared (as tma_load_3d, one more
// coordinate).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            int w, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}

// Four 8x8 16-bit matrices from shared memory; lanes 8j..8j+7 give the row
// addresses of matrix j, and lane t receives row t/4, elements 2(t%4) and
// 2(t%4)+1 of each (the transposed matrix with .trans).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// D = A B + D on the tensor cores for one warp: A 16x16 f16 (row), B 16x8
// f16 (column), D 16x8 f32.  Lane t = 4 gid + tig holds A rows gid and
// gid + 8 at columns 2tig, 2tig+1 (a0, a1) and 2tig+8, 2tig+9 (a2, a3), B
// rows 2tig, 2tig+1 (b0) and 2tig+8, 2tig+9 (b1) of column gid, and D rows
// gid (d[0], d[1]) and gid + 8 (d[2], d[3]) at columns 2tig, 2tig+1.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A B + D with tf32 operands (fp32 bit patterns, the low 13 fraction bits
// ignored): A 16x8 (row), B 8x8 (column), D 16x8 f32.  Lane t = 4 gid + tig
// holds A rows gid / gid + 8 at column tig (a0 / a1) and tig + 4 (a2 / a3),
// B rows tig (b0) and tig + 4 (b1) of column gid, and D as for mma_16816.
__device__ __forceinline__ void mma_1688_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 rounded to tf32 (10 fraction bits), to nearest with ties away.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// The KV stream is read once per call: mark it first to leave L2.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their memory operations are visible (returns at once
// when the grid was launched without the attribute), and allow the next
// dependent grid of the stream to be scheduled.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The kernels' test hook (kv_pool_set_test_stall): with stall_ns > 0, each
// warp waits up to stall_ns on `bar`, a barrier that nothing completes, as
// it would on a copy that never lands.  The wait runs out and the warp gives
// up: it sets the CTA's abort flag and PKV_DEV_TIMEOUT, and the kernel then
// queues its first copies, reads nothing, drains them and returns, as after
// a real timeout.  Called early in the kernel, where few registers are live.
// Returns true if the warp gave up.  Warp-uniform.
__device__ __forceinline__ bool test_stall(uint32_t bar, unsigned long long stall_ns,
                                           volatile int* ctl, int32_t* status) {
  if (stall_ns == 0) return false;
  bool ok = mbar_wait_bounded(bar, 0, ctl, stall_ns);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0 && !ctl[0]) {
    ctl[0] = 1;
    if (status) atomicOr(reinterpret_cast<unsigned int*>(status), PKV_DEV_TIMEOUT);
  }
  return !ok;
}

// Named barrier over `count` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Atomic add at GPU scope with acquire-release order: the writes ordered
// before it in the caller (including other threads' writes ordered by a
// barrier) are visible to whoever acquires the value it writes, and the
// caller sees every write released before the value it reads.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Load with acquire order at GPU scope: the caller sees every write released
// before the value it reads.
__device__ __forceinline__ int load_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Store with release order at GPU scope: the writes ordered before it in the
// caller (including other threads' writes ordered by a barrier) are visible
// to whoever acquires the value it stores.
__device__ __forceinline__ void store_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait (bounded) until *p is non-zero, reading it with acquire order; false
// after kWaitLimitNs or once *abort is set.
__device__ __forceinline__ bool wait_flag(const int* p, const volatile int* abort) {
  if (load_acquire(p)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (load_acquire(p)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void record_status(int32_t* status, uint32_t bits) {
  if (status) atomicOr(reinterpret_cast<unsigned int*>(status), bits);
}

// ---------------------------------------------------------------- plan ----
// First attended token of a row of L tokens under a sliding window of W
// tokens (W = 0: no window): the row attends to [window_start, L).
__device__ __forceinline__ int window_start(int L, int window) {
  return window > 0 && L > window ? L - window : 0;
}

// The per-CTA plan: validated lengths and the exclusive prefix sum of the
// pages each row reads, in shared memory.  lens[i] is seq_lens[i] clamped to
// [0, 16 * bt_stride] (a clamp records PKV_DEV_BAD_LENGTH); a row reads the
// pages holding tokens [window_start, L), block-table entries
// window_start / 16 onwards; row_start has num_rows + 1 entries.  Rows
// shorter than min_len (the queries of a several-query step) read nothing
// and record PKV_DEV_BAD_LENGTH.  Warp 0 scans; every thread of the CTA must
// call it.
__device__ __forceinline__ void plan_rows(const int32_t* __restrict__ seq_lens, int num_rows,
                                          int bt_stride, int window, int32_t* status, int* lens,
                                          int* row_start, int min_len = 1) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    if (lane == 0) row_start[0] = 0;
    for (int base = 0; base < num_rows; base += 32) {
      const int r = base + lane;
      int L = 0;
      if (r < num_rows) {
        L = seq_lens[r];
        const int cap = bt_stride * kPage;
        if (L < 0 || L > cap) {
          record_status(status, PKV_DEV_BAD_LENGTH);
          L = L < 0 ? 0 : cap;
        }
        lens[r] = L;
      }
      if (L > 0 && L < min_len) {  // fewer tokens than the step's queries: nothing read
        record_status(status, PKV_DEV_BAD_LENGTH);
        L = 0;
        lens[r] = 0;
      }
      int v = L > 0 ? (L + kPage - 1) / kPage - window_start(L, window) / kPage : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += u;
      }
      if (r < num_rows) row_start[r + 1] = carry + v;
      carry += __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();
}

// floor(x / y) for 0 <= x and 0 < y, for the work-split search.  Integer
// division is a long dependent sequence on the GPU, and the search runs a
// chain of them before a CTA can queue its first copy; for operands below
// 2^21 the quotient is estimated in fp32 (x times an approximate reciprocal
// of y: the estimate is within one of the quotient) and corrected by the
// sign of the remainder.  Larger operands take the plain division.  (Measured
// per CTA on the 8B f16 batch: the search 2059 -> 1830 cycles; elsewhere the
// plain 32-bit division was as fast or faster, so it is kept there.)
__device__ __forceinline__ int udiv(int x, int y) {
  if ((x | y) < (1 << 21)) {
    const int q = __float2int_rz(__fdividef(__int2float_rn(x), __int2float_rn(y)));
    const int r = x - q * y;
    return q + (r >= y ? 1 : 0) - (r < 0 ? 1 : 0);
  }
  return x / y;
}

// Chunk holding unit x (0 <= x < T) when T units are split into C chunks
// [floor(kT/C), floor((k+1)T/C)): the largest k with floor(kT/C) <= x, which
// is ceil((x + 1) C / T) - 1.  In 32-bit arithmetic when T (C + 1) < 2^31
// (a 64-bit division is a long software routine on the GPU).
__device__ __forceinline__ int chunk_of(long long x, long long T, int C) {
  if (T * (C + 1) < (1ll << 31)) {
    const int xi = static_cast<int>(x), Ti = static_cast<int>(T);
    return ((xi + 1) * C + Ti - 1) / Ti - 1;
  }
  return static_cast<int>(((x + 1) * C + T - 1) / T - 1);
}

// Row holding unit x: the largest i with n_kv * row_start[i] <= x (rows with
// no pages are skipped automatically).  Requires x < n_kv * row_start[rows].
__device__ __forceinline__ int row_of(const int* row_start, int num_rows, int n_kv,
                                      long long x) {
  int lo = 0, hi = num_rows;  // n_kv*row_start[lo] <= x < n_kv*row_start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(n_kv) * row_start[mid] <= x)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- split ----
// The work split of T (row, KV head, page) units into at most C chunks.
// Uniform: chunk k covers [floor(k T / C'), floor((k + 1) T / C')), C' =
// min(C, T).  Aligned to the (row, KV head) segments, for a cap of t units a
// chunk: a row of npg >= t pages gives each of its n_kv segments cps =
// ceil(npg / t) chunks, chunk q of a segment covering its pages
// [floor(q npg / cps), floor((q + 1) npg / cps)); a shorter row gives
// ceil(n_kv / m) chunks of m = floor(t / npg) whole segments (the last one
// fewer).  A segment split over several chunks then always ends where a chunk
// ends, so no chunk stops in the middle of its units to hand a partial state
// on.  t is the smallest cap from ceil(T / C) to floor(1.1 T / C) for which the
// rows need at most C chunks; the aligned split is taken when the call allows
// it, that range holds more than one cap and one of them fits, else the
// uniform one.
struct Split {
  int aligned;  // 1: aligned with cap t; 0: uniform
  int t;
  int used;     // chunks holding units: C' (uniform) or the rows' total (aligned)
  int pad;
};

// Choose the split for the rows planned by plan_rows (row_start), write it
// to *sp and, when aligned, the exclusive prefix sum of the rows' chunk
// counts to pc[0 .. num_rows].  Every thread of the CTA (at least 128) must
// call it; it ends with __syncthreads.
//
// The counts are monotone in the cap, so the cap is the first of
// lo0, lo0 + 1, .. hi0 whose count fits.  The CTA tests eight caps at a time:
// sixteen lanes a cap, each over every sixteenth row, a shuffle sum in the
// half warp, the eight counts in shared memory.
__device__ __forceinline__ void plan_split(const int* row_start, int num_rows, int n_kv, int C,
                                           bool allow_aligned, Split* sp, int* pc) {
  __shared__ int counts[8];
  const long long T = static_cast<long long>(n_kv) * row_start[num_rows];
  int aligned = 0, t = 0;
  // 32-bit arithmetic throughout; batches of 2^31 units or more take the
  // uniform split.
  if (allow_aligned && T > 0 && T < (1ll << 31) && C > 0) {
    const int T32 = static_cast<int>(T);
    const int Cs = C < (1 << 29) ? C : (1 << 29);  // counts saturate at Cs + 1
    const int q0 = udiv(T32, Cs);
    const int lo0 = q0 + (T32 - q0 * Cs != 0);  // ceil(T / C)
    const int hi0 = T32 < (1 << 27) ? udiv(11 * T32, 10 * Cs) : static_cast<int>((11ll * T32) / (10ll * Cs));
    // only when the cap may exceed ceil(T / C) (about 10 units a chunk or more)
    const int cand = threadIdx.x >> 4, sub = threadIdx.x & 15;  // 8 caps x 16 lanes
    for (int base = lo0; hi0 > lo0 && base <= hi0; base += 8) {
      if (threadIdx.x < 128) {
        const int cap = base + cand;
        int c = 0;
        for (int r = sub; r < num_rows; r += 16) {
          const int npg = row_start[r + 1] - row_start[r];
          int x = 0;
          if (npg > 0) {
            if (npg >= cap) {
              x = n_kv * udiv(npg + cap - 1, cap);
            } else {
              const int m = udiv(cap, npg);
              x = udiv(n_kv + m - 1, m);
            }
          }
          c = min(c + x, Cs + 1);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) c = min(c + __shfl_xor_sync(kFull, c, o), Cs + 1);
        if (sub == 0) counts[cand] = c;
      }
      __syncthreads();
      int found = 0;
#pragma unroll
      for (int u = 7; u >= 0; --u)
        if (base + u <= hi0 && counts[u] <= Cs) found = base + u;
      __syncthreads();  // counts[] is rewritten by the next round
      if (found) {
        aligned = 1;
        t = found;
        break;
      }
    }
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int used;
    if (aligned) {
      int carry = 0;
      if (lane == 0) pc[0] = 0;
      for (int base = 0; base < num_rows; base += 32) {
        const int r = base + lane;
        const int npg = r < num_rows ? row_start[r + 1] - row_start[r] : 0;
        int v = 0;
        if (npg > 0) {
          if (npg >= t) {
            v = n_kv * udiv(npg + t - 1, t);
          } else {
            const int m = udiv(t, npg);
            v = udiv(n_kv + m - 1, m);
          }
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(kFull, v, o);
          if (lane >= o) v += u;
        }
        if (r < num_rows) pc[r + 1] = carry + v;
        carry += __shfl_sync(kFull, v, 31);
      }
      used = carry;
    } else {
      used = static_cast<int>(T < C ? T : C);
    }
    if (lane == 0) {
      sp->aligned = aligned;
      sp->t = t;
      sp->used = used;
    }
  }
  __syncthreads();
}

// Units [b, e) of chunk k (empty, b = e = T, for k >= sp.used).
__device__ __forceinline__ void chunk_range(const Split& sp, int k, const int* row_start,
                                            const int* pc, int num_rows, int n_kv,
                                            long long& b, long long& e) {
  const long long T = static_cast<long long>(n_kv) * row_start[num_rows];
  if (k >= sp.used) {
    b = e = T;
    return;
  }
  if (!sp.aligned) {
    if (T * (sp.used + 1) < (1ll << 31)) {  // 32-bit arithmetic when it cannot overflow
      const int Ti = static_cast<int>(T);
      b = k * Ti / sp.used;
      e = (k + 1) * Ti / sp.used;
    } else {
      b = static_cast<long long>(k) * T / sp.used;
      e = static_cast<long long>(k + 1) * T / sp.used;
    }
    return;
  }
  int lo = 0, hi = num_rows;  // pc[lo] <= k < pc[hi]: the row is the largest such lo
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pc[mid] <= k)
      lo = mid;
    else
      hi = mid;
  }
  const int l = k - pc[lo], npg = row_start[lo + 1] - row_start[lo];
  const long long base = static_cast<long long>(n_kv) * row_start[lo];
  if (npg >= sp.t) {
    const int cps = (npg + sp.t - 1) / sp.t, h = l / cps, q = l - h * cps;
    const long long seg = base + static_cast<long long>(h) * npg;
    if (npg < 46340) {  // (q + 1) * npg < 2^31
      b = seg + q * npg / cps;
      e = seg + (q + 1) * npg / cps;
    } else {
      b = seg + static_cast<long long>(q) * npg / cps;
      e = seg + static_cast<long long>(q + 1) * npg / cps;
    }
  } else {
    const int m = sp.t / npg;
    const int h1 = (l + 1) * m < n_kv ? (l + 1) * m : n_kv;
    b = base + static_cast<long long>(l) * m * npg;
    e = base + static_cast<long long>(h1) * npg;
  }
}

// First and last chunk meeting segment (row i, KV head h) of npg > 0 pages.
__device__ __forceinline__ void segment_chunks(const Split& sp, int i, int h, const int* row_start,
                                               const int* pc, int num_rows, int n_kv, int& k0,
                                               int& k1) {
  const int npg = row_start[i + 1] - row_start[i];
  if (!sp.aligned) {
    const long long T = static_cast<long long>(n_kv) * row_start[num_rows];
    const long long s0 = static_cast<long long>(n_kv) * row_start[i] + static_cast<long long>(h) * npg;
    k0 = chunk_of(s0, T, sp.used);
    k1 = chunk_of(s0 + npg - 1, T, sp.used);
  } else if (npg >= sp.t) {
    const int cps = (npg + sp.t - 1) / sp.t;
    k0 = pc[i] + h * cps;
    k1 = k0 + cps - 1;
  } else {
    k0 = k1 = pc[i] + h / (sp.t / npg);
  }
}

}  // namespace pkv

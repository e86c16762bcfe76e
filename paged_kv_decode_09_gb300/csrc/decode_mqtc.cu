// decode_mqtc.cu — several queries per row on the fifth-generation tensor
// cores (tcgen05, accumulators in tensor memory), f16 and bf16 KV: the
// verification step of speculative decoding and small chunks of chunked
// prefill (Leone, "What ships": chunked prefill, exact speculative
// verification; LeatEngine, "Capabilities": chunked prefill, speculative
// decoding).
//
// The operation is that of decode_mq.cu: query j of a row of L tokens whose
// last q_len are new sits at P = L - q_len + j and attends causally to
// [max(0, P + 1 - W), P + 1); the (query, query head) pairs of a KV head are
// a pass's columns, here up to 32 of them.  What differs is how a page's
// products run: a block of 8 pages of one (row, KV head) is one matrix
// product per step, issued by one thread.  q and P are split into parts in
// the KV format, whose products accumulate: f16 takes two (the rounding and
// the rounding of the remainder, 11 significant bits each), bf16 three (8
// bits each), so a product keeps about 22 or 24 significant bits (as in the
// other kernels):
//   scores  S[128 tokens][32] = K[128 tokens][128 dims] (sum of the parts of
//           Q)^T: K straight from the staged tiles (A, K-major, 128-byte
//           swizzle); the parts of Q^T (the 32 columns' queries times scale *
//           log2 e; f16 normalised per column by a power of two) 32 rows each
//           in shared memory, one product per part into the same columns;
//   softmax one thread per (token, 16 columns), reading its row of S from
//           tensor memory: base 2, masks per column (causal, window, length),
//           the running maximum raised only when a block exceeds it by more
//           than 8 (a vote of the softmax warps), P scaled by 2^7 and split
//           into its parts (f16: the leading 11 bits and the rounding of the
//           rest; bf16: 8, 8 and the rounding of the rest), written as
//           [P1 | P2 (| P3)] [128 tokens][32 a part] to shared memory, a
//           token's 16 columns in two 16-byte stores per part;
//   values  O^T[128 dims][32 a part] += V^T [P1 | P2 (| P3)]: V read in place
//           from the staged tiles and P both as MN-major operands; the parts'
//           columns of O^T, added at the end, stay in tensor memory for the
//           whole piece.
//
// The warps have one job each, and the blocks flow through them as a
// pipeline.  Warps 8 and 10 fetch block-table entries, store the new tokens
// of the first pass (K, V) one block ahead of their copies, and queue one
// tensor copy per tile of K and of V into rings of 32 KiB slots (8 pages;
// three for K, two for V).  A tile lands as [2 token groups][2 halves][8
// tokens][64 dims], so the 8-token groups of a slot's 8 tiles sit a uniform 2
// KiB apart for either half: the operand layout the products read.  Warp 9
// (one elected lane) issues the products, the scores of block b + 2 before
// the values of block b.  Warps 0..7 run the softmax of block b meanwhile.
// A K slot is free again once its scores are computed, well before the
// block's values, so K copies run ahead of the softmax; V copies, needed
// last, follow their own ring.  S is double-buffered in tensor memory and P
// in shared memory; Q^T, one buffer, is replaced once a piece's last scores
// are read.  Shared-memory barriers carry every hand-over:
//   kfull[s], vfull[s]  copies of K or V slot s landed (transaction bytes)
//   kempty[s]  the scores of K slot s computed  (product commit)
//   vempty[s]  the values of V slot s computed  (product commit)
//   sfull[x]  scores in S buffer x             (product commit)
//   sfree[x]  S buffer x read                  (softmax warps, 8 arrivals)
//   pready[x] P buffer x written               (softmax warps, 8 arrivals)
//   pvdone[x] the values product from P x done (product commit)
//   qready    Q^T of the next piece written    (softmax warps, 8 arrivals)
// Every wait is bounded; the warp that gives up sets the CTA's abort flag,
// which ends every other wait, and the CTA drains its copies and products
// before it releases the tensor memory.
//
// One CTA per SM.  The work split is the uniform split of the (row, KV head,
// page) units with a price per piece (kPiecePenalty), so that a chunk that
// crosses into another segment reads fewer pages.  A segment split over
// chunks leaves a partial state per piece in the workspace (slots of 32
// columns); the piece that takes the segment's last arrival ticket (taken as
// its last block starts) merges them once the others have published theirs
// (a release add to the segment's count of pieces written), staging two
// pieces' accumulators at a time in shared memory by bulk copies.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kSwWarps = 8;                          // softmax warps 0..7
constexpr int kSwThreads = kSwWarps * 32;            // 256
constexpr int kKWarp = 8, kMmaWarp = 9, kVWarp = 10;  // warp 11 only fills the warpgroup
constexpr int kTcThreads = 384;
constexpr int kSwBar = 1;                            // named barrier of the softmax warps
constexpr int kBlockPages = 8;                       // pages of a block: the products' M = 128 tokens
constexpr int kVStages = 2;                          // slots of the V ring
constexpr uint32_t kSlotBytes = kBlockPages * 4096;  // a ring slot: 8 tiles of K or V, 32 KiB
constexpr uint32_t kTmemO = 64;                      // S0: 0..31, S1: 32..63, O^T from 64
constexpr float kPUp = 128.0f;                       // P is stored times 2^7 (as kPShift)
constexpr float kNoMax = -1e30f;                     // a column's m before its first score
// The work split's price of a piece, in units (pages): a chunk that a
// segment starts in pays it.  One more piece (its end, partial state and
// merge, and the next piece's start) costs about as long as 50 pages of
// blocks; on the 8B f16 layer at 32 columns 48, 52 and 56 measured 38.7,
// 38.9 and 38.4 us (40 and 64, earlier: 40.6 and 39.3 us).
constexpr int kPiecePenalty = 56;

// The KV formats: f16 parts of q and P keep 11 significant bits each, so
// two of them hold the ~22 bits the other kernels keep; bf16 parts keep 8,
// so three (~24 bits).  bf16's larger Q^T and P leave room for 2 K slots.
template <int DT>
struct TcFmt;
template <>
struct TcFmt<PKV_KV_F16> {
  static constexpr int kParts = 2;
  static constexpr int kKStages = 3;
  static constexpr uint32_t kFormat = 0;     // operand type in the instruction descriptor
  static constexpr uint32_t kTmemCols = 128;
};
template <>
struct TcFmt<PKV_KV_BF16> {
  static constexpr int kParts = 3;
  static constexpr int kKStages = 2;
  static constexpr uint32_t kFormat = 1;
  static constexpr uint32_t kTmemCols = 256;
};

// Shared memory, from a 1024-byte aligned base.
template <int DT>
struct TcSmem {
  using F = TcFmt<DT>;
  static constexpr uint32_t kAlign = 1024;
  static constexpr uint32_t kQRows = 32 * F::kParts;           // Q^T rows: 32 columns a part
  static constexpr uint32_t kQHalf = kQRows * 128;             // one 64-dim half of Q^T
  static constexpr uint32_t kPCols = 32 * F::kParts;           // P columns: 32 a part
  static constexpr uint32_t kPBuf = (kPCols + 63) / 64 * 16384;  // 64-column planes [128][128 B]
  static constexpr uint32_t kV = F::kKStages * kSlotBytes;     // K ring from 0, then the V ring
  static constexpr uint32_t kQ = kV + kVStages * kSlotBytes;   // Q^T: [2 halves][kQRows][128 B]
  static constexpr uint32_t kP = kQ + 2 * kQHalf;              // P x2: [planes][128 tokens][128 B]
  static constexpr uint32_t kRed = kP + 2 * kPBuf;         // float [2][4][32] block maxima, [4][32] sums
  static constexpr uint32_t kQexp = kRed + 3 * 4 * 32 * 4; // float [2][32]: 2^e of each column's q
  static constexpr uint32_t kBar = kQexp + 2 * 32 * 4;     // 21 barriers, 8 bytes each
  static constexpr uint32_t kCtl = kBar + 22 * 8;          // int [4]: [0] abort, [1] last arrival
  static constexpr uint32_t kTmem = kCtl + 16;             // uint32: tensor-memory base
  static constexpr uint32_t kRows = kTmem + 16;             // int row_start[rows + 1], lens[rows]
  static size_t bytes(int rows) { return kAlign + kRows + (2 * static_cast<size_t>(rows) + 1) * 4; }
};
// barrier indices
constexpr int kBKfull = 0, kBKempty = 3, kBVfull = 6, kBVempty = 8, kBSfull = 10, kBSfree = 12,
              kBPready = 14, kBPvdone = 16, kBQready = 18, kBStall = 19, kBMerge = 20, kNumBars = 21;

// --------------------------------------------------------- tcgen05 PTX ----
// Shared-memory matrix descriptor: 128-byte swizzle, start address and the
// two byte offsets in units of 16 bytes.  K-major operands (rows of 64
// elements, 8 rows per 1024-byte atom): sbo = 1024, lbo unused.  The MN-major
// V^T operand: lbo = bytes between the 64-element halves of M, sbo = bytes
// between groups of 8 rows along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16 with f32 accumulation; A and B both f16
// (format 0) or both bf16 (format 1).
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, bool a_mn_major, bool b_mn_major,
                                                uint32_t format) {
  return (1u << 4) | (format << 7) | (format << 10) | (a_mn_major ? (1u << 15) : 0u) |
         (b_mn_major ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every product this thread has issued is complete.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 16 consecutive 32-bit columns of the warp's 32 lanes (lane = thread).
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int u = 0; u < 16; ++u) v[u] = __uint_as_float(r[u]);
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 2^x by the hardware approximation (about 22 correct bits; 2^-inf = 0,
// results below 2^-126 flushed to 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier of `count` threads that also ORs `pred` over them.
__device__ __forceinline__ bool barrier_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Tensor copy of the 5-D box at {0, 0, 0, 0, v} (a whole tile) into shared
// memory, completing on `bar`, with an L2 eviction-priority hint.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* tmap, int v, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %2, %2, %2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(0), "r"(v), "r"(bar), "l"(policy)
      : "memory");
}

// The maximum (kMax) or sum over the warp's 32 lanes of each of a lane's 16
// values, by a butterfly that halves the values a lane keeps at each step
// (8, 4, 2, 1 exchanges, then one more): 16 shuffles.  Lane l returns value
// (l >> 1) & 15's result; v is overwritten.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int half = 8 >> s, bit = 16 >> s;
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(kFull, send, bit);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  const float r = __shfl_xor_sync(kFull, v[0], 1);
  return kMax ? fmaxf(v[0], r) : v[0] + r;
}

// Atomic add at GPU scope with release order, no value returned: the writes
// ordered before it (including other threads' writes ordered by a CTA-scope
// barrier) are visible to whoever acquires the sum.
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A pair of fp32 values as the kParts parts of the format, each packed as a
// pair: f16: the rounding and the rounding of the remainder; bf16: the
// leading 8 bits, the next 8, and the rounding of the rest (x0 in the low
// half of each word).
template <int DT>
__device__ __forceinline__ void split_parts(float x0, float x1, uint32_t (&w)[TcFmt<DT>::kParts]) {
  if constexpr (DT == PKV_KV_F16) {
    w[0] = split_f16x2(x0, x1, false);
    w[1] = split_f16x2(x0, x1, true);
  } else {
    const float a0 = __uint_as_float(__float_as_uint(x0) & 0xFFFF0000u);
    const float a1 = __uint_as_float(__float_as_uint(x1) & 0xFFFF0000u);
    const float r0 = x0 - a0, r1 = x1 - a1;  // exact
    const float b0 = __uint_as_float(__float_as_uint(r0) & 0xFFFF0000u);
    const float b1 = __uint_as_float(__float_as_uint(r1) & 0xFFFF0000u);
    const __nv_bfloat162 pa = __floats2bfloat162_rn(a0, a1), pb = __floats2bfloat162_rn(b0, b1);
    const __nv_bfloat162 pc = __floats2bfloat162_rn(r0 - b0, r1 - b1);
    w[0] = *reinterpret_cast<const uint32_t*>(&pa);
    w[1] = *reinterpret_cast<const uint32_t*>(&pb);
    w[2] = *reinterpret_cast<const uint32_t*>(&pc);
  }
}

// A pair of probabilities (times 2^7, at most 2^15) as the parts of the
// format: f16: the leading 11 bits (exact in f16 from 2^-14 up) and the
// rounding of the rest, one packed conversion each; bf16 as split_parts.
template <int DT>
__device__ __forceinline__ void split_p(float p0, float p1, uint32_t (&w)[TcFmt<DT>::kParts]) {
  if constexpr (DT == PKV_KV_F16) {
    const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
    const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
    const __half2 hh = __floats2half2_rn(h0, h1), ll = __floats2half2_rn(p0 - h0, p1 - h1);
    w[0] = *reinterpret_cast<const uint32_t*>(&hh);
    w[1] = *reinterpret_cast<const uint32_t*>(&ll);
  } else {
    split_parts<DT>(p0, p1, w);
  }
}

// True in one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Whether the phase of `bar` with the given parity has completed (does not
// suspend the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// A wait of one lane of the warp, polling without suspending (each hand-over
// of the pipeline is on its critical path), its outcome given to every lane
// (warp-uniform: the tensor-memory loads that follow are warp-collective).
// Gives up, as mbar_wait_bounded does, once *abort is set or after
// kWaitLimitNs.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          int lane) {
  int ok = 1;
  if (lane == 0 && !mbar_test_wait(bar, parity)) {
    const unsigned long long t0 = global_ns();
    ok = 0;
    while (!ok) {
#pragma unroll 1
      for (int i = 0; i < 64 && !ok; ++i) ok = mbar_test_wait(bar, parity) ? 1 : 0;
      if (!ok && (*abort || global_ns() - t0 > kWaitLimitNs)) break;
    }
  }
  return __shfl_sync(kFull, ok, 0) != 0;
}

// A block: the units [x, x + n) of one (row, KV head) segment, n <= 8.
struct Blk {
  int i, h, n, L, pfirst;  // row, KV head, pages, row length, first page's index in the row
  long long x, seg_end;
};

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_mqtc_kernel(const __grid_constant__ DecodeArgs a,
                             const __grid_constant__ TileMaps maps) {
  static_assert(DT == PKV_KV_F16 || DT == PKV_KV_BF16,
                "the tensor-core several-query kernel takes 16-bit KV");
  using F = TcFmt<DT>;
  using SM = TcSmem<DT>;
  constexpr int kKStages = F::kKStages;
  constexpr int kParts = F::kParts;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((SM::kAlign - (smem_addr(smem_raw) & (SM::kAlign - 1))) &
                              (SM::kAlign - 1));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + SM::kCtl);
  int* row_start = reinterpret_cast<int*>(smem + SM::kRows);
  int* lens = row_start + a.num_rows + 1;
  const uint32_t bars = smem_addr(smem + SM::kBar);
  auto bar = [&](int b, int x) { return bars + 8u * static_cast<uint32_t>(b + x); };
  const uint32_t sQ = smem_addr(smem + SM::kQ), sP = smem_addr(smem + SM::kP);
  const int G = a.n_q / a.n_kv;
  const int nc = a.nq * G;  // columns of this pass, <= 32
  const int plan_window = a.window > 0 ? a.window + a.q_len - 1 : 0;

  if (tid == 0) {
    prefetch_tensormap(&maps.kp);  // kernel parameters, not written by an earlier kernel
    prefetch_tensormap(&maps.vp);
    ctl[0] = 0;
    ctl[1] = 0;
    for (int b = 0; b < kNumBars; ++b) {
      const bool sw = b >= kBSfree && b < kBSfree + 2;
      const bool sw2 = b >= kBPready && b < kBPready + 2;
      const bool sw3 = b == kBQready;
      mbar_init(bars + 8u * b, (sw || sw2 || sw3) ? kSwWarps : 1);
    }
    fence_mbar_init();
  }
  // Q^T and P start zeroed: Q^T rows of columns beyond nc stay zero
  for (int e = tid; e < static_cast<int>((SM::kRed - SM::kQ) / 16); e += kTcThreads)
    reinterpret_cast<uint4*>(smem + SM::kQ)[e] = make_uint4(0u, 0u, 0u, 0u);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(smem + SM::kTmem)),
                 "r"(F::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, plan_window, blockIdx.x == 0 ? a.status : nullptr,
            lens, row_start, a.q_len);  // ends with __syncthreads
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM::kTmem);
  const bool stalled = test_stall(bar(kBStall, 0), a.test_stall_ns, ctl, a.status);
  // ---- the work split: the uniform split of the (row, KV head, page) units
  // over virtual units, in which every segment is preceded by kPiecePenalty
  // units that no chunk reads.  A chunk that a segment starts in gets that
  // many fewer units: the cost of one more piece (its end, partial state
  // and merge, and the next piece's start).  Segment s = (row i, head h),
  // real units [r_s, r_s + npg), sits at virtual [r_s + P (s + 1), ...).
  const long long T = static_cast<long long>(a.n_kv) * row_start[a.num_rows];
  const long long Tv = T + static_cast<long long>(kPiecePenalty) * a.n_kv * a.num_rows;
  // chunks of at least one virtual unit: a chunk inside a segment then holds
  // at least one of its units (chunks past C are empty)
  const int C = static_cast<int>(min(static_cast<long long>(a.vchunks), Tv));
  auto vrow = [&](int r) {  // virtual start of row r (its first penalty)
    return static_cast<long long>(a.n_kv) * (row_start[r] + static_cast<long long>(kPiecePenalty) * r);
  };
  auto vreal = [&](long long vb) -> long long {  // the first unit at virtual position >= vb
    if (vb >= Tv) return T;
    int lo = 0, hi = a.num_rows;  // vrow(lo) <= vb < vrow(hi)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (vrow(mid) <= vb)
        lo = mid;
      else
        hi = mid;
    }
    const int npg = row_start[lo + 1] - row_start[lo];
    const long long base = static_cast<long long>(a.n_kv) * row_start[lo];
    if (npg == 0) return base;
    const long long r = vb - vrow(lo);
    const long long h = r / (npg + kPiecePenalty);
    const long long off = r - h * (npg + kPiecePenalty) - kPiecePenalty;
    return base + h * npg + (off > 0 ? off : 0);
  };
  // first and last chunk of segment (i, h) of npg > 0 pages
  auto seg_chunks = [&](int i, int h, int& k0, int& k1) {
    const int npg = row_start[i + 1] - row_start[i];
    const long long v0 = static_cast<long long>(a.n_kv) * row_start[i] + static_cast<long long>(h) * npg +
                         static_cast<long long>(kPiecePenalty) * (static_cast<long long>(i) * a.n_kv + h + 1);
    k0 = chunk_of(v0, Tv, C);
    k1 = chunk_of(v0 + npg - 1, Tv, C);
  };
  const int k = blockIdx.x;
  const long long c_begin = k < C ? vreal(static_cast<long long>(k) * Tv / C) : T;
  const long long c_end = k < C ? vreal(static_cast<long long>(k + 1) * Tv / C) : T;

  if (blockIdx.x == 0) {  // rows without tokens (or shorter than q_len): zeros
    for (int i = 0; i < a.num_rows; ++i)
      if (row_start[i + 1] == row_start[i])
        for (int jj = 0; jj < a.nq; ++jj)
          for (int e = tid; e < a.n_q * kD; e += kTcThreads)
            a.out[((static_cast<long long>(i) * a.q_len + a.q0 + jj) * a.n_q) * kD + e] = 0.f;
  }

  // The block starting at unit x (x < c_end): up to 8 units of x's segment.
  auto block_at = [&](long long x, Blk& bk) {
    const int i = row_of(row_start, a.num_rows, a.n_kv, x);
    const int npg = row_start[i + 1] - row_start[i];
    const long long row_base = static_cast<long long>(a.n_kv) * row_start[i];
    bk.i = i;
    bk.h = static_cast<int>(x - row_base) / npg;
    const long long seg_start = row_base + static_cast<long long>(bk.h) * npg;
    bk.seg_end = seg_start + npg;
    const long long e = min(min(bk.seg_end, c_end), x + kBlockPages);
    bk.n = static_cast<int>(e - x);
    bk.x = x;
    bk.L = lens[i];
    bk.pfirst = window_start(bk.L, plan_window) / kPage + static_cast<int>(x - seg_start);
  };

  const int zero = 0;
  if (warp == kKWarp || warp == kVWarp) {
    // ------------------------------------------------------------ copies ----
    // K (warp 8) or V (warp 10): slot b % 2 of the ring for block b, once the
    // product that read the slot's previous block is done.
    const bool is_v = warp == kVWarp;
    const CUtensorMap* map = is_v ? &maps.vp : &maps.kp;
    const uint32_t ring = smem_addr(smem) + (is_v ? SM::kV : 0u);
    const int bfull = is_v ? kBVfull : kBKfull, bempty = is_v ? kBVempty : kBKempty;
    const int ns = is_v ? kVStages : kKStages;
    const float* src_new = is_v ? a.v_new : a.k_new;
    uint8_t* data = is_v ? a.v_data : a.k_data;
    const uint64_t policy = policy_evict_first();
    // lane q < n: the block-table entry of the block's page q, read one
    // block ahead (while the slot of the block before is awaited)
    auto entry = [&](const Blk& bk) {
      return lane < bk.n
                 ? __ldg(a.block_table + static_cast<long long>(bk.i) * a.bt_stride + bk.pfirst + lane)
                 : 0;
    };
    // The new tokens (first pass) in block bk's pages, in the kv_append
    // encoding, before the block's copies: 4 dims per lane, the loads of 8
    // tokens issued before their stores.
    auto append_block = [&](const Blk& bk, int pg) {
      const int first_new = bk.L - a.q_len;
      const int lo = max(first_new, bk.pfirst * kPage);
      const int hi = min(bk.L, (bk.pfirst + bk.n) * kPage);
      const bool ok_pg = lane < bk.n && pg >= 0 && pg < a.num_pages;
      for (int p0 = lo; p0 < hi; p0 += 8) {
        float4 v4[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const long long src_row = static_cast<long long>(bk.i) * a.q_len + (p0 + e - first_new);
          if (p0 + e < hi)
            v4[e] = __ldg(reinterpret_cast<const float4*>(src_new + (src_row * a.n_kv + bk.h) * kD +
                                                           lane * 4));
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int pos = p0 + e;
          if (pos < hi) {
            const int q = pos / kPage - bk.pfirst;
            const int pgq = __shfl_sync(kFull, pg, q);
            if (__shfl_sync(kFull, ok_pg ? 1 : 0, q)) {
              uint2 w;  // 4 dims in the format (round to nearest even)
              if constexpr (DT == PKV_KV_F16) {
                const __half2 h01 = __floats2half2_rn(v4[e].x, v4[e].y);
                const __half2 h23 = __floats2half2_rn(v4[e].z, v4[e].w);
                w.x = *reinterpret_cast<const uint32_t*>(&h01);
                w.y = *reinterpret_cast<const uint32_t*>(&h23);
              } else {
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(v4[e].x, v4[e].y);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(v4[e].z, v4[e].w);
                w.x = *reinterpret_cast<const uint32_t*>(&h01);
                w.y = *reinterpret_cast<const uint32_t*>(&h23);
              }
              const size_t tile = static_cast<size_t>(pgq) * a.n_kv + bk.h;
              *reinterpret_cast<uint2*>(data + tile * (kPage * kD * 2) + (pos % kPage) * (kD * 2) +
                                        lane * 8) = w;
            }
          }
        }
      }
      // the tiles are read next by the async proxy (tensor copies)
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
    };
    int b = 0;
    bool failed = stalled;
    Blk bk;
    int pg = 0;
    if (c_begin < c_end) {
      block_at(c_begin, bk);
      pg = entry(bk);
      if (src_new != nullptr && !failed) append_block(bk, pg);
    }
    for (long long x = c_begin; x < c_end && !failed; ++b) {
      const long long xn = x + bk.n;
      Blk bn;
      int pgn = 0;
      if (xn < c_end) {
        block_at(xn, bn);
        pgn = entry(bn);
      }
      const int st = b % ns;
      if (b >= ns && !warp_wait(bar(bempty, st), ((b / ns) - 1) & 1, ctl, lane)) {
        failed = true;
        break;
      }
      const bool ok_pg = lane < bk.n && pg >= 0 && pg < a.num_pages;
      if (lane < bk.n && !ok_pg) {
        if (!is_v) record_status(a.status, PKV_DEV_BAD_PAGE);
        pg = 0;
      }
      const uint32_t dst0 = ring + st * kSlotBytes;
      if (lane == 0) mbar_arrive_expect_tx(bar(bfull, st), static_cast<uint32_t>(bk.n) * 4096u);
      __syncwarp();
      if (lane < bk.n)  // page q of the block at 4 KiB * q: one copy of the whole tile
        tma_load_5d(dst0 + lane * 4096, map, pg * a.n_kv + bk.h, bar(bfull, st), policy);
      // the next block's new tokens, while its slot is still in use
      if (src_new != nullptr && xn < c_end) append_block(bn, pgn);
      x = xn;
      bk = bn;
      pg = pgn;
    }
    // drain: the copies of the last slots land before the CTA exits
    for (int bb = max(0, b - ns); bb < b; ++bb)
      if (lane == 0) mbar_wait_bounded(bar(bfull, bb % ns), (bb / ns) & 1, &zero);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- products ----
    // The whole warp runs this loop (its waits are warp-uniform); one elected
    // lane issues the products and their commits.
    const bool leader = elect_one();
    const uint32_t id_s = tc_idesc(128, 32, false, false, F::kFormat);
    const uint32_t id_pv = tc_idesc(128, SM::kPCols, true, true, F::kFormat);
    int b = 0, p = 0;
    // the values products still to issue, oldest first: up to two blocks
    // (the scores run two blocks ahead of the values)
    int pv_cnt = 0, pv_b[2] = {0, 0}, pv_n[2] = {0, 0};
    bool pv_first[2] = {false, false};
    int last_bar = -1;  // barrier of the last commit, and its parity
    uint32_t last_par = 0;
    bool failed = stalled;
    auto fail = [&]() {
      if (!failed && lane == 0 && !ctl[0]) {
        ctl[0] = 1;
        record_status(a.status, PKV_DEV_TIMEOUT);
      }
      failed = true;
    };
    auto issue_pv = [&]() {  // the oldest pending values product
      const int vb = pv_b[0], vn = pv_n[0];
      const bool vfirst = pv_first[0];
      pv_b[0] = pv_b[1];
      pv_n[0] = pv_n[1];
      pv_first[0] = pv_first[1];
      --pv_cnt;
      if (!warp_wait(bar(kBPready, vb & 1), (vb >> 1) & 1, ctl, lane) ||
          !warp_wait(bar(kBVfull, vb % kVStages), (vb / kVStages) & 1, ctl, lane)) {
        fail();
        return;
      }
      tc_fence_after();
      // 16 tokens (page kk, 4 KiB kk into the slot) a step: V^T rows (dims)
      // in halves 1 KiB apart, 8-token groups 2 KiB apart; P rows 16 kk ..
      // (N-major)
      const uint64_t ad0 = sw128_desc(smem_addr(smem) + SM::kV + (vb % kVStages) * kSlotBytes,
                                      1024, 2048);
      const uint64_t bd0 = sw128_desc(sP + (vb & 1) * SM::kPBuf, 16384, 1024);
      if (leader) {
        for (int kk = 0; kk < vn; ++kk)
          tc_mma(tmem + kTmemO, ad0 + kk * (4096 >> 4), bd0 + kk * (2048 >> 4), id_pv,
                 (!vfirst || kk > 0) ? 1 : 0);
        tc_commit(bar(kBVempty, vb % kVStages));
        tc_commit(bar(kBPvdone, vb & 1));
      }
      __syncwarp();
      last_bar = kBPvdone + (vb & 1);
      last_par = (vb >> 1) & 1;
    };
    for (long long x = c_begin; x < c_end && !failed; ++p) {
      Blk pb;
      block_at(x, pb);
      const long long b_piece = min(pb.seg_end, c_end);
      // a new piece: its Q^T is written once the softmax warps have read the
      // scores of the last block before it, which may wait for the values
      // products still pending here
      while (!failed && pv_cnt > 0) issue_pv();
      if (failed) break;
      if (!warp_wait(bar(kBQready, 0), p & 1, ctl, lane)) {
        fail();
        break;
      }
      const uint64_t qd0 = sw128_desc(sQ, 16, 1024);
      bool first = true;
      for (long long xb = x; xb < b_piece; ++b) {
        const int n = static_cast<int>(min(b_piece - xb, static_cast<long long>(kBlockPages)));
        const int st = b % kKStages;
        if (!warp_wait(bar(kBKfull, st), (b / kKStages) & 1, ctl, lane) ||
            (b >= 2 && !warp_wait(bar(kBSfree, b & 1), ((b - 2) >> 1) & 1, ctl, lane))) {
          fail();
          break;
        }
        tc_fence_after();
        // 16 dims a step: K half kk / 4 (1 KiB further), 32 bytes in, its
        // 8-token groups 2 KiB apart; the parts of Q^T, each 32 rows, accumulate
        // into the same columns
        const uint64_t kd0 = sw128_desc(smem_addr(smem) + st * kSlotBytes, 16, 2048);
        if (leader) {
          const uint32_t tS = tmem + (b & 1) * 32;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            const uint32_t qoff16 = ((kk >> 2) * SM::kQHalf + (kk & 3) * 32) >> 4;
#pragma unroll
            for (int q = 0; q < kParts; ++q)  // part q of Q^T: rows 32 q .. (4096 bytes a part)
              tc_mma(tS, kd0 + off, qd0 + qoff16 + q * (4096 >> 4), id_s, (kk > 0 || q > 0) ? 1 : 0);
          }
          tc_commit(bar(kBKempty, st));
          tc_commit(bar(kBSfull, b & 1));
        }
        __syncwarp();
        last_bar = kBSfull + (b & 1);
        last_par = (b >> 1) & 1;
        if (pv_cnt == 2) {
          issue_pv();
          if (failed) break;
        }
        if (pv_cnt == 0) {
          pv_b[0] = b;
          pv_n[0] = n;
          pv_first[0] = first;
        } else {
          pv_b[1] = b;
          pv_n[1] = n;
          pv_first[1] = first;
        }
        ++pv_cnt;
        first = false;
        xb += n;
      }
      x = b_piece;
    }
    while (!failed && pv_cnt > 0) issue_pv();
    // drain: every product issued completes before the tensor memory goes
    if (lane == 0 && last_bar >= 0) mbar_wait_bounded(bars + 8u * last_bar, last_par, &zero);
    __syncwarp();
  } else if (warp == kVWarp + 1) {
    // fills the warpgroup; nothing to do
  } else {
    // ----------------------------------------------------------- softmax ----
    const int qw = warp & 3, hc = warp >> 2;  // tensor-memory lane quarter, column half
    const int t = 32 * qw + lane;             // this thread's token row of a block (and dim of O)
    const uint32_t lane_off = static_cast<uint32_t>(32 * qw) << 16;
    float* red = reinterpret_cast<float*>(smem + SM::kRed);
    float* qexp_s = reinterpret_cast<float*>(smem + SM::kQexp);
    bool failed = stalled;
    auto fail = [&]() {
      if (!failed && !ctl[0]) {
        ctl[0] = 1;
        record_status(a.status, PKV_DEV_TIMEOUT);
      }
      failed = true;
    };
    // Q^T of the piece at unit x, and its columns' scales into qexp buffer
    // qb: thread tid takes column tid / 8, dims 16 (tid % 8) ..
    auto write_q = [&](long long x, int qb) {
      Blk pb;
      block_at(x, pb);
      const int c = tid >> 3, d0 = (tid & 7) * 16;
      float v[16];
      const bool in = c < nc;
      const float* qv = in ? a.q + ((static_cast<long long>(pb.i) * a.q_len + a.q0 + c / G) * a.n_q +
                                    pb.h * G + c % G) * kD + d0
                           : nullptr;
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in) x4 = __ldg(reinterpret_cast<const float4*>(qv + e));
        v[e] = x4.x * a.qscale;
        v[e + 1] = x4.y * a.qscale;
        v[e + 2] = x4.z * a.qscale;
        v[e + 3] = x4.w * a.qscale;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[e]));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));  // the column's 8 threads
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
      int e2 = 0;
      if (DT == PKV_KV_F16 && amax > 0.f && amax <= 3.0e38f) {
        int ex;
        frexpf(amax, &ex);
        e2 = ex - 14;  // largest |q| in [2^13, 2^14): both f16 parts normal
      }
      if (in && DT == PKV_KV_F16) {
        // rows c (hi) and 32 + c (lo); dims d0 .. d0 + 15 = two 16-byte chunks
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int row = part * 32 + c;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = split_f16x2(ldexpf(v[8 * ch + 2 * e], -e2), ldexpf(v[8 * ch + 2 * e + 1], -e2),
                                 part == 1);
            const int d = d0 + 8 * ch;
            const uint32_t off = (d >> 6) * SM::kQHalf + row * 128 +
                                 ((((d & 63) >> 3) ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + SM::kQ + off) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        if ((tid & 7) == 0) qexp_s[qb * 32 + c] = ldexpf(1.0f, e2);
      } else if (in) {
        // bf16: part q in row 32 q + c (no scaling: bf16 has fp32's range)
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t w[kParts][4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t pw[kParts];
            split_parts<DT>(v[8 * ch + 2 * e], v[8 * ch + 2 * e + 1], pw);
#pragma unroll
            for (int q = 0; q < kParts; ++q) w[q][e] = pw[q];
          }
          const int d = d0 + 8 * ch;
#pragma unroll
          for (int q = 0; q < kParts; ++q) {
            const int row = q * 32 + c;
            const uint32_t off = (d >> 6) * SM::kQHalf + row * 128 +
                                 ((((d & 63) >> 3) ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + SM::kQ + off) =
                make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
          }
        }
        if ((tid & 7) == 0) qexp_s[qb * 32 + c] = ldexpf(1.0f, e2);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q^T for the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBQready, 0));
    };
    // the query of the thread's column 16 hc + u: qbase + 4 bits u of qoff
    const int qbase = (16 * hc) / G;
    uint64_t qoff = 0;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      qoff |= static_cast<uint64_t>((16 * hc + u) / G - qbase) << (4 * u);

    int b = 0, p = 0, rb = 0;
    int nmerge = 0;  // merge rounds staged so far (parity of the merge barrier)
    if (tid < 64) qexp_s[tid] = 0.f;  // columns beyond nc keep 0
    named_barrier(kSwBar, kSwThreads);
    // Q^T of piece p + 1 replaces p's once the scores of p's last block are
    // read (all of p's score products are then done), after that block's
    // probabilities: the product thread, two blocks ahead, waits for it.
    if (c_begin < c_end && !failed) write_q(c_begin, 0);
    named_barrier(kSwBar, kSwThreads);  // qexp of piece 0
    for (long long x = c_begin; x < c_end; ++p) {
      Blk pb;
      block_at(x, pb);
      const long long b_piece = min(pb.seg_end, c_end);
      const int i = pb.i, h = pb.h, L = pb.L;
      const long long j = static_cast<long long>(i) * a.n_kv + h;
      int k0, k1;
      seg_chunks(i, h, k0, k1);
      const int P0 = L - a.q_len + a.q0;  // position of the pass's first query
      // tokens every used column attends: [all_lo, P0]
      const int all_lo = window_start(P0 + (nc - 1) / G + 1, a.window);
      const float4* qexp4 = reinterpret_cast<const float4*>(qexp_s + (p & 1) * 32 + 16 * hc);
      // per column: m = the running maximum minus 7 (so that 2^(s - m) is P
      // times 2^7), l = the sum of the thread's 2^(s - m).  Before a column's
      // first score m is -1e30, a finite stand-in for -inf: s - m is then -inf
      // for a masked score and above the raise threshold for any other.
      float m[16], l[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        m[u] = kNoMax;
        l[u] = 0.f;
      }
      bool first = true;
      long long xb = x;
      const bool whole = (k0 == k1);
      // the piece's arrival ticket (thread 0), taken when its last block
      // starts: the round trip overlaps the block
      int ticket = 0;
      for (; xb < b_piece; ++b) {
        const int n = static_cast<int>(min(b_piece - xb, static_cast<long long>(kBlockPages)));
        const int pfirst = pb.pfirst + static_cast<int>(xb - x);
        if (tid == 0 && !whole && xb + n >= b_piece) ticket = atomicAdd(mq_counter(a.flags, j, 0), 1);
        // ---- scores of block b from S buffer b & 1: d = s - m, masked to -inf
        const int t0 = pfirst * kPage;
        const bool fast = t0 >= all_lo && t0 + n * kPage <= P0 + 1;  // every token, every column
        const bool in_blk = t < n * kPage;  // rows of pages past n: stale stage data
        const int pos = t0 + t;
        // score of column u, from S and the column's scale (masked to -inf)
        auto score = [&](int u, float sv, float qe) {
          bool ok = in_blk;
          if (!fast) {
            const int P = P0 + qbase + static_cast<int>((qoff >> (4 * u)) & 15);
            ok = ok && pos < L && 16 * hc + u < nc && pos <= P && pos >= window_start(P + 1, a.window);
          }
          return ok ? sv * qe : -INFINITY;
        };
        float sc[16];  // the scores (-inf when masked)
        if (!failed && !warp_wait(bar(kBSfull, b & 1), (b >> 1) & 1, ctl, lane)) fail();
        const uint32_t tS = tmem + lane_off + (b & 1) * 32 + 16 * hc;
        bool up = false;
        if (!failed) {
          tc_fence_after();
          float sv[16];
          tc_ld16(tS, sv);
          tc_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBSfree, b & 1));  // S buffer b & 1 read
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 q4 = qexp4[e];
            const float qe[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int u = 4 * e + k;
              sc[u] = score(u, sv[u], qe[k]);
              up = up || sc[u] - m[u] > 15.0f;  // -inf when masked (m is finite)
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) sc[u] = -INFINITY;
        }
        // ---- the running maximum: raised (by a vote of the softmax warps)
        // only when the block exceeds it by more than 8
        const bool vote = barrier_or(kSwBar, kSwThreads, up || failed);
        if (vote) {
          if (barrier_or(kSwBar, kSwThreads, failed)) {
            failed = true;
            break;
          }
          float* rr = red + rb * 128;
          {
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = sc[u];
            const float mx = warp_reduce16<true>(v, lane);  // column (lane >> 1) & 15
            if ((lane & 1) == 0) rr[qw * 32 + 16 * hc + ((lane >> 1) & 15)] = mx;
          }
          named_barrier(kSwBar, kSwThreads);
          rb ^= 1;  // the next raise writes the other buffer (a vote lies between)
          float my_al = 1.0f;  // lane u % 16 keeps alpha of column 16 hc + u % 16
          bool any_scale = false;
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int c = 16 * hc + u;
            const float b4 = fmaxf(fmaxf(rr[c], rr[32 + c]), fmaxf(rr[64 + c], rr[96 + c]));
            const float mn = b4 > m[u] + 15.0f ? b4 - 7.0f : m[u];
            // 0 from the stand-in; not needed in a piece's first block (l is 0
            // and the block's values product overwrites O^T)
            const float al = (first || mn == m[u]) ? 1.0f : ex2_approx(m[u] - mn);
            if ((lane & 15) == u) my_al = al;
            any_scale = any_scale || al != 1.0f;
            l[u] *= al;
            m[u] = mn;
          }
          // O^T columns of the warp's 16 columns (hi and lo parts), times
          // alpha, once the values product of block b - 1 is done (not in a
          // piece's first block: its values product overwrites O^T)
          if (!first && any_scale) {
            if (!warp_wait(bar(kBPvdone, (b - 1) & 1), ((b - 1) >> 1) & 1, ctl, lane)) {
              fail();
            } else {
              tc_fence_after();
#pragma unroll
              for (int part = 0; part < kParts; ++part) {
                const uint32_t tO = tmem + lane_off + kTmemO + 32 * part + 16 * hc;
                float ov[16];
                tc_ld16(tO, ov);
                tc_wait_ld();
#pragma unroll
                for (int u = 0; u < 16; ++u) ov[u] *= __shfl_sync(kFull, my_al, u);
                tc_st16(tO, ov);
                tc_wait_st();
              }
            }
          }
        }
        // ---- probabilities into P buffer b & 1 once the values product of
        // block b - 2 has read it: row t (token) of [128 tokens][64], columns
        // 0..31 Phi (pu's leading 11 bits, exact in f16 from 2^-14 up), 32..63
        // Plo (the f16 rounding of the rest), 128-byte swizzle
        if (!failed && b >= 2 && !warp_wait(bar(kBPvdone, b & 1), ((b - 2) >> 1) & 1, ctl, lane))
          fail();
        if (!failed) {
          uint8_t* prow = smem + SM::kP + (b & 1) * SM::kPBuf + t * 128;
#pragma unroll
          for (int e = 0; e < 2; ++e) {  // columns 16 hc + 8 e .. + 7
            uint32_t w[kParts][4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int u = 8 * e + 2 * k;
              // P times 2^7 (2^-inf = 0 for masked scores; m is finite)
              const float p0 = ex2_approx(sc[u] - m[u]), p1 = ex2_approx(sc[u + 1] - m[u + 1]);
              l[u] += p0;
              l[u + 1] += p1;
              uint32_t pw[kParts];
              split_p<DT>(p0, p1, pw);
#pragma unroll
              for (int q = 0; q < kParts; ++q) w[q][k] = pw[q];
            }
            // part q: columns 32 q + 16 hc + 8 e ..: 16-byte chunk ch of the
            // row, in plane ch / 8 (parts 0 and 1 in plane 0)
            const int ch = 2 * hc + e;
            *reinterpret_cast<uint4*>(prow + ((ch ^ (t & 7)) << 4)) =
                make_uint4(w[0][0], w[0][1], w[0][2], w[0][3]);
            *reinterpret_cast<uint4*>(prow + (((ch + 4) ^ (t & 7)) << 4)) =
                make_uint4(w[1][0], w[1][1], w[1][2], w[1][3]);
            if constexpr (kParts == 3)
              *reinterpret_cast<uint4*>(prow + 16384 + ((ch ^ (t & 7)) << 4)) =
                  make_uint4(w[2][0], w[2][1], w[2][2], w[2][3]);
          }
          // V rows of slots past the row's length in a page the block reads:
          // the pool may hold anything there (NaN * 0 is NaN).  Zeroed once
          // the block's V copies have landed.
          const int q = t / kPage, slot = t % kPage;
          const bool zero_v = hc == 0 && q < n && pos >= L;
          if (__any_sync(kFull, zero_v)) {
            if (!warp_wait(bar(kBVfull, b % kVStages), (b / kVStages) & 1, ctl, lane)) {
              fail();
            } else if (zero_v) {
#pragma unroll
              for (int hv = 0; hv < 2; ++hv) {
                uint4* row = reinterpret_cast<uint4*>(smem + SM::kV + (b % kVStages) * kSlotBytes +
                                                      q * 4096 + (slot >> 3) * 2048 + hv * 1024 +
                                                      (slot & 7) * 128);
#pragma unroll
                for (int e = 0; e < 8; ++e) row[e] = make_uint4(0u, 0u, 0u, 0u);
              }
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P, zeroed V rows
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBPready, b & 1));
          // the next piece's Q^T once this piece's last scores are read: it
          // overlaps the wait for this block's values product at the piece end
          if (xb + n >= b_piece && b_piece < c_end) write_q(b_piece, (p + 1) & 1);
        }
        first = false;
        xb += n;
      }
      // ---- piece end: the values product of the piece's last block done
      if (!failed && !warp_wait(bar(kBPvdone, (b - 1) & 1), ((b - 1) >> 1) & 1, ctl, lane)) fail();
      if (barrier_or(kSwBar, kSwThreads, failed)) {
        failed = true;
        break;
      }
      tc_fence_after();
      float o[16];  // O^T (its parts' columns added) and the sums carry P's factor 2^7: removed here
      if constexpr (kParts == 2) {
        float olo[16];
        tc_ld16(tmem + lane_off + kTmemO + 16 * hc, o);
        tc_ld16(tmem + lane_off + kTmemO + 32 + 16 * hc, olo);
        tc_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) o[u] = (o[u] + olo[u]) * (1.0f / kPUp);
      } else {
        tc_ld16(tmem + lane_off + kTmemO + 16 * hc, o);
#pragma unroll
        for (int q = 1; q < kParts; ++q) {
          float oq[16];
          tc_ld16(tmem + lane_off + kTmemO + 32 * q + 16 * hc, oq);
          tc_wait_ld();
#pragma unroll
          for (int u = 0; u < 16; ++u) o[u] += oq[u];
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) o[u] *= 1.0f / kPUp;
      }
      tc_fence_before();  // O^T read before the next piece's first values product
      float* rs = red + 256;
      {
        const float ls = warp_reduce16<false>(l, lane);  // column (lane >> 1) & 15
        if ((lane & 1) == 0) rs[qw * 32 + 16 * hc + ((lane >> 1) & 15)] = ls;
      }
      named_barrier(kSwBar, kSwThreads);
      float Ls[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = 16 * hc + u;
        Ls[u] = ((rs[c] + rs[32 + c]) + (rs[64 + c] + rs[96 + c])) * (1.0f / kPUp);
      }
      auto out_col = [&](int c) {
        return a.out + ((static_cast<long long>(i) * a.q_len + a.q0 + c / G) * a.n_q + h * G +
                        c % G) * kD;
      };
      const int d = t;  // O^T lane = dim
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = 16 * hc + u;
        if (c >= nc) continue;
        if (whole) {
          out_col(c)[d] = o[u] / Ls[u];
        } else {
          const long long slot = (k + j) * kMqCols + c;
          a.part_acc[slot * kD + d] = o[u];
          if (qw == 0 && lane == 0) {
            // the running maximum (-inf: no token of the column in the piece)
            a.part_ml[slot * 2] = Ls[u] > 0.f ? m[u] + static_cast<float>(kPShift) : -INFINITY;
            a.part_ml[slot * 2 + 1] = Ls[u];
          }
        }
      }
      if (!whole) {
        // The last-ticketed piece merges the segment; every other piece
        // publishes its partial state by a release add to the segment's
        // count of pieces written, which the merging piece acquires.
        if (tid == 0) ctl[1] = ticket == k1 - k0;
        asm volatile("fence.proxy.async.global;" ::: "memory");  // the partial, for bulk copies
        named_barrier(kSwBar, kSwThreads);  // the CTA's partial written; ctl[1]
        const bool last = ctl[1] != 0;
        if (tid == 0) {
          if (!last) {
            red_release_add(mq_counter(a.flags, j, 1), 1);
          } else {  // bounded wait (acquire) for the other k1 - k0 pieces
            const int* cnt = mq_counter(a.flags, j, 1);
            if (load_acquire(cnt) < k1 - k0) {
              const unsigned long long t0w = global_ns();
              while (load_acquire(cnt) < k1 - k0) {
                if (ctl[0] || global_ns() - t0w > kWaitLimitNs) {
                  fail();
                  break;
                }
              }
            }
          }
        }
        if (barrier_or(kSwBar, kSwThreads, failed)) {
          failed = true;
          break;
        }
        if (last) {
          // Merge the pieces (thread 0's acquire, passed on by the barrier),
          // two per round: their accumulators [32 columns][128] (16 KiB a
          // piece) staged in the P buffers by bulk copies, their (m, l) read
          // directly.  Thread tid: column tid / 8, dims 16 (tid % 8) ..
          const int c = tid >> 3, dd = (tid & 7) * 16;
          float Mx = -INFINITY, Lx = 0.f, Ax[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) Ax[e] = 0.f;
          const uint64_t keep = policy_evict_first();
          for (int kb = k0; kb <= k1; kb += 2) {
            const int np = min(2, k1 - kb + 1);
            if (tid == 0) {
              asm volatile("fence.proxy.async.global;" ::: "memory");  // after the acquire
              mbar_arrive_expect_tx(bar(kBMerge, 0), static_cast<uint32_t>(np) * 16384u);
              for (int u = 0; u < np; ++u)
                bulk_g2s(sP + u * 16384,
                         a.part_acc + (static_cast<long long>(kb + u) + j) * kMqCols * kD, 16384u,
                         bar(kBMerge, 0), keep);
            }
            float mk[2], lk[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              mk[u] = -INFINITY;
              lk[u] = 0.f;
              if (u < np && c < nc) {
                const long long slot = (static_cast<long long>(kb + u) + j) * kMqCols + c;
                mk[u] = __ldcg(a.part_ml + slot * 2);
                lk[u] = __ldcg(a.part_ml + slot * 2 + 1);
              }
            }
            if (!warp_wait(bar(kBMerge, 0), nmerge & 1, ctl, lane)) fail();
            ++nmerge;
            if (!failed && c < nc) {
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                if (mk[u] == -INFINITY) continue;  // no token of this query in the piece (or none)
                const float4* src =
                    reinterpret_cast<const float4*>(smem + SM::kP + u * 16384 + (c * kD + dd) * 4);
                const float mn = fmaxf(Mx, mk[u]);
                const float f0 = exp2f(Mx - mn), f1 = exp2f(mk[u] - mn);
                Lx = Lx * f0 + lk[u] * f1;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float4 x4 = src[e];
                  Ax[4 * e] = Ax[4 * e] * f0 + x4.x * f1;
                  Ax[4 * e + 1] = Ax[4 * e + 1] * f0 + x4.y * f1;
                  Ax[4 * e + 2] = Ax[4 * e + 2] * f0 + x4.z * f1;
                  Ax[4 * e + 3] = Ax[4 * e + 3] * f0 + x4.w * f1;
                }
                Mx = mn;
              }
            }
            named_barrier(kSwBar, kSwThreads);  // the staged pieces read
          }
          if (c < nc) {
            float* oc = out_col(c) + dd;
            const float inv = 1.0f / Lx;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              reinterpret_cast<float4*>(oc)[e] =
                  make_float4(Ax[4 * e] * inv, Ax[4 * e + 1] * inv, Ax[4 * e + 2] * inv,
                              Ax[4 * e + 3] * inv);
          }
          if (tid == 0) {  // ready for the next call
            *mq_counter(a.flags, j, 0) = 0;
            *mq_counter(a.flags, j, 1) = 0;
          }
        }
      }
      named_barrier(kSwBar, kSwThreads);  // red and the merge flag are free for the next piece
      x = b_piece;
    }
    tc_fence_before();
  }

  // ---- teardown: every role has drained its copies and products
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(F::kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------ launchers ----
template <int DT>
static cudaError_t mqtc_prepare(size_t smem) {
  static std::atomic<size_t> granted[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && granted[dev].load(std::memory_order_relaxed) >= smem)
    return cudaSuccess;
  e = cudaFuncSetAttribute(paged_decode_mqtc_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e == cudaSuccess && dev >= 0 && dev < 64) {
    size_t cur = granted[dev].load();
    while (cur < smem && !granted[dev].compare_exchange_weak(cur, smem)) {
    }
  }
  return e;
}

template <int DT>
static cudaError_t launch_mqtc_t(const DecodeArgs& a, const TileMaps& maps, int chunks,
                                 cudaStream_t st) {
  const size_t smem = TcSmem<DT>::bytes(a.num_rows);
  cudaError_t e = mqtc_prepare<DT>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(chunks);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = PKV_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // One chunk per SM: the segment-aligned split needs more chunks than that
  // for any batch of a few long rows, and trying it costs the kernel's start.
  DecodeArgs au = a;
  au.aligned_split = 0;
  e = cudaLaunchKernelEx(&cfg, paged_decode_mqtc_kernel<DT>, au, maps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_paged_decode_mqtc(int dtype, const DecodeArgs& a, const TileMaps& maps,
                                     int chunks, cudaStream_t st) {
  if (dtype == PKV_KV_F16) return launch_mqtc_t<PKV_KV_F16>(a, maps, chunks, st);
  if (dtype == PKV_KV_BF16) return launch_mqtc_t<PKV_KV_BF16>(a, maps, chunks, st);
  return cudaErrorInvalidValue;
}

// Rows whose plan tables fit beside the rings in the device's opt-in shared
// memory (queried once per device).
template <int DT>
static int mqtc_max_rows_t() {
  static std::atomic<int> cached[64];  // 0: not queried yet; else rows + 1
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c - 1;
  }
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  const long long fixed = TcSmem<DT>::kAlign + TcSmem<DT>::kRows + 4;  // 2 rows + 1 ints of plan
  const int rows = optin > fixed ? static_cast<int>((optin - fixed) / 8) : 0;
  if (dev >= 0 && dev < 64) cached[dev].store(rows + 1, std::memory_order_relaxed);
  return rows;
}

int paged_decode_mqtc_max_rows(int dtype) {
  if (dtype == PKV_KV_F16) return mqtc_max_rows_t<PKV_KV_F16>();
  if (dtype == PKV_KV_BF16) return mqtc_max_rows_t<PKV_KV_BF16>();
  return 0;
}

template <int DT>
static cudaError_t mqtc_occupancy_t(int rows, int* blocks) {
  const size_t smem = TcSmem<DT>::bytes(rows);
  cudaError_t e = mqtc_prepare<DT>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, paged_decode_mqtc_kernel<DT>,
                                                       kTcThreads, smem);
}

cudaError_t paged_decode_mqtc_blocks_per_sm(int dtype, int rows, int* blocks) {
  if (dtype == PKV_KV_F16) return mqtc_occupancy_t<PKV_KV_F16>(rows, blocks);
  if (dtype == PKV_KV_BF16) return mqtc_occupancy_t<PKV_KV_BF16>(rows, blocks);
  return cudaErrorInvalidValue;
}

}  // namespace pkv

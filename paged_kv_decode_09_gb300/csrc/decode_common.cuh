// decode_common.cuh — pieces shared by the decode kernels (decode.cu: one
// query per row; decode_mq.cu: several): build-time knobs, the shared-memory
// tile geometry and its swizzled addressing, the conversions of stored values
// into MMA operands, and the merge of partial states.
#pragma once

#include <cmath>
#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// Build-time knobs (defaults are the tuned values): shared-memory stages per
// warp and the CTAs per SM the register allocation must allow, for each
// dtype (q8_0 is bound by instruction issue: more warps hide more latency),
// programmatic dependent launch of the decode kernel (1 on), and the partial
// states a merge loads per round trip.
#ifndef PKV_F16_RING
#define PKV_F16_RING 2
#endif
#ifndef PKV_Q8_RING
#define PKV_Q8_RING 2
#endif
#ifndef PKV_F16_CTAS_PER_SM
#define PKV_F16_CTAS_PER_SM 3
#endif
#ifndef PKV_Q8_CTAS_PER_SM
#define PKV_Q8_CTAS_PER_SM 4
#endif
#ifndef PKV_PDL
#define PKV_PDL 1
#endif
#ifndef PKV_F32_CTAS_PER_SM
#define PKV_F32_CTAS_PER_SM 2  // 16 KiB stages, one per warp: the shared memory of 2 CTAs
#endif
#ifndef PKV_MERGE_BATCH
#define PKV_MERGE_BATCH 8  // 4 for q8_0, whose 4 CTAs per SM leave 128 registers a thread
#endif

constexpr int kWarps = 4;  // warps per CTA; the final piece merge gives each thread one dim
constexpr int kThreads = kWarps * 32;
static_assert(kThreads == kD, "the final piece merge maps one thread to one dim");

// Shared-memory stage of one unit: the K tile then the V tile of one
// (page, KV head), each [16 tokens][128 dims] under the 128-byte swizzle
// (f16: two 2 KiB halves of 64 dims); q8_0 block scales in a separate area.
template <int DT>
struct Tiles;
template <>
struct Tiles<PKV_KV_F16> {
  static constexpr uint32_t kData = kPage * kD * 2;  // 4096 bytes of one K or V tile
  static constexpr uint32_t kScale = 0;
  static constexpr uint32_t kCodes = 2 * kData;  // K and V tiles of a stage
  static constexpr uint32_t kScales = 0;
  static constexpr uint32_t kTx = kCodes;  // bytes a stage's barrier waits for
  static constexpr int kRing = PKV_F16_RING;  // stages per warp
};
template <>
struct Tiles<PKV_KV_BF16> : Tiles<PKV_KV_F16> {};  // same geometry: 16-bit values
template <>
struct Tiles<PKV_KV_F32> {
  static constexpr uint32_t kData = kPage * kD * 4;  // 8 KiB of one K or V tile: four 2 KiB boxes
  static constexpr uint32_t kScale = 0;
  static constexpr uint32_t kCodes = 2 * kData;
  static constexpr uint32_t kScales = 0;
  static constexpr uint32_t kTx = kCodes;
  static constexpr int kRing = 1;  // one 16 KiB stage per warp
};
template <>
struct Tiles<PKV_KV_Q8_0> {
  static constexpr uint32_t kData = kPage * kD;                   // 2048 codes
  static constexpr uint32_t kScale = kPage * (kD / kQBlock) * 2;  // 128 bytes of f16 scales
  static constexpr uint32_t kCodes = 2 * kData;
  static constexpr uint32_t kScales = 2 * kScale;  // K scales then V scales
  static constexpr uint32_t kTx = kCodes + kScales;
  static constexpr int kRing = PKV_Q8_RING;  // stages per warp
};

// Copy tile z (one (page, KV head) of K or V) into a stage: one tensor copy
// for every format.  The 16-bit and f32 tiles go through 4-D maps whose box
// lists the dims of a 128-byte row, the 16 tokens, then the row's place in
// the 256-byte (512-byte) token, so the copy lands as 2 (4) swizzled boxes
// of [16 tokens][128 bytes]; q8_0 tiles are one such box.  One copy per tile
// instead of 2 (16-bit) or 4 (f32): fewer copies to queue at the start of a
// step, when every warp of the GPU queues its first stages at once.
template <int DT>
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const void* tmap, int z, uint32_t bar,
                                              uint64_t policy) {
  if constexpr (DT == PKV_KV_Q8_0)
    tma_load_3d(dst, tmap, 0, 0, z, bar, policy);
  else
    tma_load_4d(dst, tmap, 0, 0, 0, z, bar, policy);
}

// ------------------------------------------------------------ operands ----
// Byte offset of the 16-byte chunk c (8 f16 / bf16, 4 f32 or 16 int8 values)
// of token row t in a swizzled tile: 128-byte rows, chunk index xor (row mod
// 8); 16-bit tiles keep dims 64..127 in a second 2 KiB box, f32 tiles hold
// four 2 KiB boxes of 32 dims.
template <int DT>
__device__ __forceinline__ uint32_t tile_offset(int t, int c) {
  if constexpr (DT != PKV_KV_Q8_0)
    return (c >> 3) * 2048 + t * 128 + (((c & 7) ^ (t & 7)) << 4);
  else
    return t * 128 + ((c ^ (t & 7)) << 4);
}

// Two 8-bit codes of a stored word `u` (offset-binary: code + 128 in each
// byte) as an exact f16 pair: the bytes chosen by `sel` go into the low
// mantissa byte of 1024 (0x64xx = 1024 + code + 128), then 1152 is
// subtracted in f16.
template <uint32_t kSel>
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t u) {
  const uint32_t biased = __byte_perm(u, 0x64646464u, kSel);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&biased),
                            __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&r);
}
constexpr uint32_t kSelB01 = 0x4140, kSelB23 = 0x4342, kSelB02 = 0x4240, kSelB13 = 0x4341;

// Per half, the larger magnitude of two f16 pairs; the sign bit of the result
// is the xor of the inputs' signs (clear it with 0x7fff7fff at the end of a
// chain).  A NaN half yields the other operand's half.
__device__ __forceinline__ uint32_t abs_max_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The tf32 part of x (`lo` false: its rounding; true: the rounding of the
// remainder), as an fp32 bit pattern.
__device__ __forceinline__ uint32_t tf32_part(float x, bool lo) {
  const uint32_t h = to_tf32(x);
  return lo ? to_tf32(x - __uint_as_float(h)) : h;
}

// The f16 part (`lo` false: the rounding of x; true: the rounding of the
// remainder) of a pair, low half x0.
__device__ __forceinline__ uint32_t split_f16x2(float x0, float x1, bool lo) {
  __half2 h = __floats2half2_rn(x0, x1);
  if (lo) {
    const float2 f = __half22float2(h);
    h = __floats2half2_rn(x0 - f.x, x1 - f.y);
  }
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 2^x on the special-function unit, for the page softmax.  Subnormal results
// flush to 0: a probability below 2^-126 of the running maximum is lost in
// the fp32 sums anyway.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// P-operand scaling shared by the kernels (see the single-query kernel's notes).
// The P operand is scaled by a power of two so that its f16 parts stay
// normal: f16 KV by 2^7 (p <= 2^8, so P <= 2^15); q8_0, where P carries the V
// block scale, by 2^(7 - vx) with 2^vx above every V scale of the piece so
// far (raised, with the accumulators rescaled, when a page exceeds it).  O
// holds the scaled sums; o_scale() undoes it.
constexpr int kPShift = 7;
constexpr int kNoScale = -64;  // vx before the piece's first page
__device__ __forceinline__ float pow2i(int e) {  // 2^e for -126 <= e <= 127
  return __int_as_float((127 + e) << 23);
}
// ---------------------------------------------------------------- merge ----
// The merge's flags below the end of the workspace (DecodeArgs::flags).
__device__ __forceinline__ int* seg_counter(int32_t* flags, long long j) { return flags - 1 - 2 * j; }
__device__ __forceinline__ int* slot_ready(int32_t* flags, long long s) { return flags - 2 - 2 * s; }
__device__ __forceinline__ int* mq_counter(int32_t* flags, long long j, int w) {
  return flags - 1 - (static_cast<long long>(kMqCounters) * j + w);
}

// Merge the base-2 partial states of segment j held in slots k + j for the
// chunks k0..k1 that meet it; one thread per dim d, all G heads:
//   M = max_k m2_k,  out = sum_k 2^(m2_k - M) acc_k / sum_k 2^(m2_k - M) l_k,
// evaluated batch by batch with a running maximum (the sums are rescaled when
// it grows).  Loads go through L2 (other CTAs wrote the slots in this
// launch); a batch of pieces costs one round trip.
template <int G, int kBatch = PKV_MERGE_BATCH>  // kBatch: pieces loaded per round trip
__device__ __forceinline__ void merge_segment(const float* part_ml, const float* part_acc,
                                              long long j, int k0, int k1, float* o, int d) {
  float M[G], Ls[G], A[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = -INFINITY;
    Ls[g] = 0.f;
    A[g] = 0.f;
  }
  for (int kk = k0; kk <= k1; kk += kBatch) {
    float m[kBatch][G], l[kBatch][G], x[kBatch][G];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const bool in = kk + u <= k1;
      const long long slot = kk + u + j;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2) : -INFINITY;
        l[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2 + 1) : 0.f;
        x[u][g] = in ? __ldcg(part_acc + (slot * G + g) * kD + d) : 0.f;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float bm = M[g];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) bm = fmaxf(bm, m[u][g]);
      const float sc = exp2f(M[g] - bm);  // 0 on the first batch (M = -inf)
      Ls[g] *= sc;
      A[g] *= sc;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float w = exp2f(m[u][g] - bm);
        Ls[g] = fmaf(w, l[u][g], Ls[g]);
        A[g] = fmaf(w, x[u][g], A[g]);
      }
      M[g] = bm;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) o[g * kD + d] = A[g] / Ls[g];
}

// Chunks actually used for T units when C are launched: min(C, T), so that
// no chunk is empty.
__device__ __forceinline__ int used_chunks(long long T, int C) {
  return static_cast<int>(T < C ? T : C);
}

// The same merge as merge_segment, done by one warp (lane l: dims 4l..4l+3).
template <int G>
__device__ __forceinline__ void merge_segment_warp(const float* part_ml, const float* part_acc,
                                                   long long j, int k0, int k1, float* o, int lane) {
  constexpr int kBatch = 2;
  float M[G], Ls[G];
  float4 A[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = -INFINITY;
    Ls[g] = 0.f;
    A[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int kk = k0; kk <= k1; kk += kBatch) {
    float m[kBatch][G], l[kBatch][G];
    float4 x[kBatch][G];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const bool in = kk + u <= k1;
      const long long slot = kk + u + j;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2) : -INFINITY;
        l[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2 + 1) : 0.f;
        x[u][g] = in ? __ldcg(reinterpret_cast<const float4*>(part_acc + (slot * G + g) * kD) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float bm = M[g];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) bm = fmaxf(bm, m[u][g]);
      const float sc = exp2f(M[g] - bm);
      Ls[g] *= sc;
      A[g].x *= sc;
      A[g].y *= sc;
      A[g].z *= sc;
      A[g].w *= sc;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float w = exp2f(m[u][g] - bm);
        Ls[g] = fmaf(w, l[u][g], Ls[g]);
        A[g].x = fmaf(w, x[u][g].x, A[g].x);
        A[g].y = fmaf(w, x[u][g].y, A[g].y);
        A[g].z = fmaf(w, x[u][g].z, A[g].z);
        A[g].w = fmaf(w, x[u][g].w, A[g].w);
      }
      M[g] = bm;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
    *reinterpret_cast<float4*>(o + g * kD + lane * 4) =
        make_float4(A[g].x / Ls[g], A[g].y / Ls[g], A[g].z / Ls[g], A[g].w / Ls[g]);
}

// The merge of segment j by the CTA that finishes its last piece: the CTA's
// own piece state, in registers (thread d holds M, Ls, A of dim d for the G
// heads), and the partial states of the segment's other pieces (slots
// kk + j for kk in [k0, k1], kk != k).  The four warps load the other pieces
// together, kPpw pieces a warp per L2 round trip (4 kPpw a trip for the CTA),
// lane l taking dims 4l .. 4l + 3; each warp folds its pieces into one state,
// leaves it in the shared merge buffer, and after a CTA barrier thread d
// combines its own state with the four warps' and writes the output.  Every
// thread of the CTA calls it; the merge buffer must be free.
template <int G, int kPpw>
__device__ __forceinline__ void merge_segment_cta(const float* part_ml, const float* part_acc,
                                                  long long j, int k0, int k1, int k,
                                                  const float (&M)[G], const float (&Ls)[G],
                                                  const float (&A)[G], float* mrg_acc,
                                                  float* mrg_ml, float* o) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_other = k1 - k0;
  float wm[G], wl[G];
  float4 wa[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    wm[g] = -INFINITY;
    wl[g] = 0.f;
    wa[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int base = 0; base < n_other; base += 4 * kPpw) {
    float m[kPpw][G], l[kPpw][G];
    float4 x[kPpw][G];
#pragma unroll
    for (int u = 0; u < kPpw; ++u) {
      const int p = base + warp + 4 * u;
      const bool in = p < n_other;
      const int kk = k0 + p + (k0 + p >= k ? 1 : 0);  // the p-th piece other than k
      const long long slot = kk + j;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2) : -INFINITY;
        l[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2 + 1) : 0.f;
        x[u][g] = in ? __ldcg(reinterpret_cast<const float4*>(part_acc + (slot * G + g) * kD) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float bm = wm[g];
#pragma unroll
      for (int u = 0; u < kPpw; ++u) bm = fmaxf(bm, m[u][g]);
      if (bm == -INFINITY) continue;  // no piece for this warp yet
      const float sc = exp2f(wm[g] - bm);  // 0 while wm is -inf
      wl[g] *= sc;
      wa[g].x *= sc;
      wa[g].y *= sc;
      wa[g].z *= sc;
      wa[g].w *= sc;
#pragma unroll
      for (int u = 0; u < kPpw; ++u) {
        const float f = exp2f(m[u][g] - bm);  // 0 for a missing piece
        wl[g] = fmaf(f, l[u][g], wl[g]);
        wa[g].x = fmaf(f, x[u][g].x, wa[g].x);
        wa[g].y = fmaf(f, x[u][g].y, wa[g].y);
        wa[g].z = fmaf(f, x[u][g].z, wa[g].z);
        wa[g].w = fmaf(f, x[u][g].w, wa[g].w);
      }
      wm[g] = bm;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      mrg_ml[(warp * G + g) * 2] = wm[g];
      mrg_ml[(warp * G + g) * 2 + 1] = wl[g];
    }
    *reinterpret_cast<float4*>(mrg_acc + (warp * G + g) * kD + lane * 4) = wa[g];
  }
  named_barrier(1, kThreads);
  const int d = threadIdx.x;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float Mx = M[g];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) Mx = fmaxf(Mx, mrg_ml[(w * G + g) * 2]);
    const float f0 = exp2f(M[g] - Mx);
    float L = f0 * Ls[g], Ax = f0 * A[g];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = exp2f(mrg_ml[(w * G + g) * 2] - Mx);  // 0 for a warp without pieces
      L = fmaf(f, mrg_ml[(w * G + g) * 2 + 1], L);
      Ax = fmaf(f, mrg_acc[(w * G + g) * kD + d], Ax);
    }
    o[g * kD + d] = Ax / L;
  }
}

// merge_segment_cta for pieces that publish their partials through ready
// flags (slot_ready): before a warp loads a piece's partial, one of its lanes
// waits for that piece's flag (acquire, bounded; the piece's CTA has already
// arrived, so it is running and publishes without waiting on anything) and
// clears it for the next call.  Returns false, without writing the output,
// if a wait gave up (then *abort is set and PKV_DEV_TIMEOUT recorded).
template <int G, int kPpw>
__device__ __forceinline__ bool merge_segment_cta_ready(const float* part_ml, const float* part_acc,
                                                        int32_t* flags, long long j, int k0, int k1,
                                                        int k, const float (&M)[G],
                                                        const float (&Ls)[G], const float (&A)[G],
                                                        float* mrg_acc, float* mrg_ml, float* o,
                                                        volatile int* abort, int32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_other = k1 - k0;
  float wm[G], wl[G];
  float4 wa[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    wm[g] = -INFINITY;
    wl[g] = 0.f;
    wa[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  bool ok = true;
  for (int base = 0; base < n_other; base += 4 * kPpw) {
    // lane u < kPpw waits for the flag of the warp's piece u of this round
    if (lane < kPpw) {
      const int p = base + warp + 4 * lane;
      if (p < n_other) {
        int* f = slot_ready(flags, k0 + p + (k0 + p >= k ? 1 : 0) + j);
        if (wait_flag(f, abort))
          *f = 0;  // ready for the next call
        else
          ok = false;
      }
    }
    ok = __all_sync(kFull, ok);
    if (!ok) break;
    __syncwarp();  // the lanes' acquires, ordered for the warp
    float m[kPpw][G], l[kPpw][G];
    float4 x[kPpw][G];
#pragma unroll
    for (int u = 0; u < kPpw; ++u) {
      const int p = base + warp + 4 * u;
      const bool in = p < n_other;
      const long long slot = k0 + p + (k0 + p >= k ? 1 : 0) + j;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2) : -INFINITY;
        l[u][g] = in ? __ldcg(part_ml + (slot * G + g) * 2 + 1) : 0.f;
        x[u][g] = in ? __ldcg(reinterpret_cast<const float4*>(part_acc + (slot * G + g) * kD) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float bm = wm[g];
#pragma unroll
      for (int u = 0; u < kPpw; ++u) bm = fmaxf(bm, m[u][g]);
      if (bm == -INFINITY) continue;
      const float sc = exp2f(wm[g] - bm);
      wl[g] *= sc;
      wa[g].x *= sc;
      wa[g].y *= sc;
      wa[g].z *= sc;
      wa[g].w *= sc;
#pragma unroll
      for (int u = 0; u < kPpw; ++u) {
        const float f = exp2f(m[u][g] - bm);
        wl[g] = fmaf(f, l[u][g], wl[g]);
        wa[g].x = fmaf(f, x[u][g].x, wa[g].x);
        wa[g].y = fmaf(f, x[u][g].y, wa[g].y);
        wa[g].z = fmaf(f, x[u][g].z, wa[g].z);
        wa[g].w = fmaf(f, x[u][g].w, wa[g].w);
      }
      wm[g] = bm;
    }
  }
  if (!ok && lane == 0 && !abort[0]) {
    abort[0] = 1;
    record_status(status, PKV_DEV_TIMEOUT);
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      mrg_ml[(warp * G + g) * 2] = wm[g];
      mrg_ml[(warp * G + g) * 2 + 1] = wl[g];
    }
    *reinterpret_cast<float4*>(mrg_acc + (warp * G + g) * kD + lane * 4) = wa[g];
  }
  named_barrier(1, kThreads);
  if (abort[0]) return false;
  const int d = threadIdx.x;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float Mx = M[g];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) Mx = fmaxf(Mx, mrg_ml[(w * G + g) * 2]);
    const float f0 = exp2f(M[g] - Mx);
    float L = f0 * Ls[g], Ax = f0 * A[g];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = exp2f(mrg_ml[(w * G + g) * 2] - Mx);
      L = fmaf(f, mrg_ml[(w * G + g) * 2 + 1], L);
      Ax = fmaf(f, mrg_acc[(w * G + g) * kD + d], Ax);
    }
    o[g * kD + d] = Ax / L;
  }
  return true;
}

// Spin (bounded) until the shared merge buffer has been released for piece
// `piece`; false on timeout or abort.
__device__ __forceinline__ bool wait_merge_buffer(volatile int* ctl, int piece) {
  if (ctl[2] >= piece) return true;
  const unsigned long long t0 = global_ns();
  while (ctl[2] < piece) {
    if (ctl[0]) return false;
    if (global_ns() - t0 > kWaitLimitNs) return false;
    __nanosleep(32);
  }
  return true;
}

// ------------------------------------------------------------- append ----
// A warp stores one new K and V token of KV head h (row `src_row` of the
// fp32 [..][n_kv][128] inputs k_new, v_new) into slot `slot` of tile
// (page, h) just before it copies that tile: 4 dims per lane; q8_0 blocks
// of 32 dims span 8 lanes.  Same encoding as kv_append.
template <int DT>
__device__ __forceinline__ void append_token(const DecodeArgs& a, long long src_row, int h,
                                             int page, int slot, int lane) {
  using TL = Tiles<DT>;
  const size_t tile = static_cast<size_t>(page) * a.n_kv + h;
  const long long src = (src_row * a.n_kv + h) * kD + lane * 4;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const float4 x = __ldg(reinterpret_cast<const float4*>((which ? a.v_new : a.k_new) + src));
    uint8_t* data = which ? a.v_data : a.k_data;
    if constexpr (DT == PKV_KV_F16) {
      const __half2 lo = __floats2half2_rn(x.x, x.y), hi = __floats2half2_rn(x.z, x.w);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&lo);
      w.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(data + tile * TL::kData + slot * (kD * 2) + lane * 8) = w;
    } else if constexpr (DT == PKV_KV_F32) {
      *reinterpret_cast<float4*>(data + tile * TL::kData + slot * (kD * 4) + lane * 16) = x;
    } else if constexpr (DT == PKV_KV_BF16) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&lo);
      w.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(data + tile * TL::kData + slot * (kD * 2) + lane * 8) = w;
    } else {
      float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      const float dq = amax / 127.0f;
      const float v[4] = {x.x, x.y, x.z, x.w};
      uint32_t packed = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float c = dq != 0.0f ? fminf(fmaxf(roundf(v[e] / dq), -127.0f), 127.0f) : 0.0f;
        packed |= (static_cast<uint32_t>(static_cast<int>(c)) & 0xffu) << (8 * e);
      }
      // stored offset-binary: code + 128 in each byte
      *reinterpret_cast<uint32_t*>(data + tile * TL::kData + slot * kD + lane * 4) =
          packed ^ 0x80808080u;
      if ((lane & 7) == 0) {
        uint8_t* sc = which ? a.v_scales : a.k_scales;
        reinterpret_cast<__half*>(sc + tile * TL::kScale)[slot * (kD / kQBlock) + (lane >> 3)] =
            __float2half_rn(dq);
      }
    }
  }
  // The tile is read next by the async proxy (bulk copy): order these generic
  // writes before it.
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

}  // namespace pkv

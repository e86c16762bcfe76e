// decode_mq.cu — paged decode attention with several queries per row: the
// verification step of speculative decoding and small chunks of chunked
// prefill (Leone, "What ships": chunked prefill, exact speculative
// verification; LeatEngine, "Capabilities": chunked prefill, speculative
// decoding).
//
// A row of L tokens whose last q_len are new has one query per new token:
// query j sits at position P = L - q_len + j and attends causally to
// [max(0, P + 1 - W), P + 1) under a window W (all of [0, P + 1) without
// one).  The (query, query head) pairs of a KV head are the "columns" of a
// call, C = q_len * G of them; each page of a (row, KV head) is read once per
// pass for all the pass's columns, and a call takes as many passes as its
// kernel's pass width requires (below).  The new tokens are stored in the
// first pass, by the warp that copies their page, just before the copy.
//
// Two kernels:
//   paged_decode_mq_kernel: the single-query kernel's structure (decode.cu):
//     the four warps of a CTA stream different pages of its chunk, each for
//     all (up to 8) columns, and merge their states at piece ends.
//   paged_decode_mqt_kernel: a team of 2 or 4 warps streams every page of
//     its chunk together, each warp owning a share of the columns (up to 32
//     in all), so a page is copied once for all of them.
// The page's MMA layout is the same in both:
//   scores: S[16 tokens][cols] = K Q^T as in the single-query kernel, with
//     the columns split over NT score n-tiles of 4 (query, head) columns x
//     {hi, lo} parts; lane 4 gid + tig ends with the scores of columns tig
//     and 4 + tig.
//   values: O^T[128 dims][cols] += V^T P^T with one B operand per part of P
//     (two MMAs into the same accumulator), so the 8 columns of an n-tile are
//     8 (query, head) pairs and O stays 32 registers a lane.
// f32 pages run the same lanes on CUDA cores (as in the single-query kernel).
// A query whose causal range does not reach a page sees only masked scores
// there: its probabilities are 0 and its running state is left alone.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// Score n-tiles (4 columns each) per dtype: bf16 runs its scores as tf32
// k-steps of 8 dims, whose query operands take twice the registers.
template <int DT>
__host__ __device__ constexpr int mq_tiles() {
  return DT == PKV_KV_BF16 ? 1 : 2;
}

// The kernel a call takes, by its C = q_len * G columns:
//   f16 : C <= 8 paged_decode_mq_kernel; beyond, the tensor-core kernel
//         (decode_mqtc.cu, passes of 32 columns) for calls of up to
//         paged_decode_mqtc_max_rows(f16) rows (its plan tables share the CTA's
//         shared memory with its rings: 2055 rows with 227 KiB), else four
//         warps of 4 columns per page up to 16 columns, of 8 beyond (passes
//         of 32).  On the 8B f16 layer at 16 and 32 columns the tensor-core
//         kernel measured 38.1 and 38.4 us, the team kernels 54.2 and 68.2.
//   bf16: C <= 4 paged_decode_mq_kernel; C <= 8 two warps of 4 columns (four
//         would leave two idle); beyond, the tensor-core kernel (passes of
//         32, three bf16 parts of q and P) up to paged_decode_mqtc_max_rows()
//         rows, else four warps of 4 (passes of 16).
//   q8_0: C <= 8 paged_decode_mq_kernel; C <= 16 two warps of 8 columns;
//         beyond, four warps of 8 (passes of 32).  Every warp that reads a
//         page converts its int8 codes, so the fewer warps per page the
//         better: two passes of 8 columns cost more than one page read by two
//         warps, four warps of 4 columns more still.
//   f32 : paged_decode_mq_kernel, passes of 8 columns (CUDA cores).
enum MqKind { kMqSingle = 0, kMqPair1, kMqPair2, kMqTeam1, kMqTeam2, kMqTc };
static int mq_kind(int dtype, int group, int q_len) {
  const int cols = q_len * group;
  if (dtype == PKV_KV_F32) return kMqSingle;
  if (dtype == PKV_KV_Q8_0) return cols <= 8 ? kMqSingle : cols <= 16 ? kMqPair2 : kMqTeam2;
  if (dtype == PKV_KV_BF16) return cols <= 4 ? kMqSingle : cols <= 8 ? kMqPair1 : kMqTc;
  return cols <= 8 ? kMqSingle : kMqTc;
}
// The kernel of a call of `rows` rows: the tensor-core kernel's calls of
// more rows than its plan tables hold go to the team kernels.
static int mq_kind_rows(int dtype, int group, int q_len, int rows) {
  const int kind = mq_kind(dtype, group, q_len);
  if (kind != kMqTc || rows <= paged_decode_mqtc_max_rows(dtype)) return kind;
  return dtype == PKV_KV_BF16 || q_len * group <= 16 ? kMqTeam1 : kMqTeam2;
}
static int mq_kind_cols(int dtype, int kind) {
  switch (kind) {
    case kMqSingle: return dtype == PKV_KV_BF16 ? 4 : 8;
    case kMqPair1: return 8;
    case kMqPair2: case kMqTeam1: return 16;
    default: return 32;  // kMqTeam2, kMqTc
  }
}
// score n-tiles (4 columns each) of a warp, and warps per page, of a kind
__host__ __device__ constexpr int kind_nt(int kind) {
  return kind == kMqTeam2 || kind == kMqPair2 ? 2 : 1;
}
__host__ __device__ constexpr int kind_ts(int kind) {
  return kind == kMqPair1 || kind == kMqPair2 ? 2 : 4;
}

int mq_pass_queries(int dtype, int group, int q_len, int rows) {
  const int per = mq_kind_cols(dtype, mq_kind_rows(dtype, group, q_len, rows)) / group;
  return per > 0 ? per : 1;
}

constexpr int kWarpCols = 8;  // (query, head) columns of one warp's state: 2 score n-tiles
// f32 KV keeps a warp's scaled queries in shared memory, one column every
// kQStride floats (the 16-byte pad puts the columns' chunks in different banks).
constexpr int kQStride = kD + 4;

template <int DT>
struct MqSmem {
  static constexpr int kStages = kWarps * Tiles<DT>::kRing;
  static constexpr uint32_t kAlign = 1024;
  static constexpr uint32_t kScl = kStages * Tiles<DT>::kCodes;
  static constexpr uint32_t kBar = kScl + kStages * Tiles<DT>::kScales;
  static constexpr uint32_t kMrgAcc = kBar + ((kStages * 8 + 15) / 16) * 16;  // f32 [warps][8][D]
  static constexpr uint32_t kMrgMl = kMrgAcc + kWarps * kWarpCols * kD * 4;    // f32 [warps][8][2]
  static constexpr uint32_t kQ = kMrgMl + kWarps * kWarpCols * 2 * 4;  // f32 KV: [warps][8][kQStride] q
  static constexpr uint32_t kCtl =
      kQ + (DT == PKV_KV_F32 ? kWarps * kWarpCols * kQStride * 4 : 0);
  static constexpr uint32_t kStall = kCtl + 16;  // the test hook's barrier (nothing completes it)
  static constexpr uint32_t kSplit = kCtl + 32;  // the work split
  static constexpr uint32_t kRows = kSplit + 16;  // row_start, lens, chunks before each row
  static size_t bytes(int rows) { return kAlign + kRows + plan_ints(rows) * 4; }
  static_assert(Tiles<DT>::kCodes % 1024 == 0, "tile stages keep the swizzle atom alignment");
};

template <int DT>
__host__ __device__ constexpr int mq_steps() {  // k-steps over the 128 dims: f16 MMAs take 16 dims, tf32 MMAs 8
  return DT == PKV_KV_BF16 ? 16 : DT == PKV_KV_F32 ? 1 : 8;  // f32: CUDA cores, no fragments
}

template <int DT, int kTiles>
struct MqState {
  static constexpr int NT = kTiles;
  static constexpr int kSteps = mq_steps<DT>();
  uint32_t qb[NT][kSteps][2];  // score B operands of n-tile t: column gid -> (4t + gid/2, part gid%2)
  float qexp[NT];              // 2^e of the lane's score column 4t + tig
  float m[NT], l[NT];          // softmax state of the lane's score columns
  float o[8][4];               // O^T: dims x V-columns 2tig (o[.][0, 2]) and 2tig + 1 (o[.][1, 3])
  int vx;                      // q8_0: bound on the piece's V block scales (as decode.cu)
  float* qs;                   // f32 KV: the warp's scaled queries [8][kQStride] in shared memory
};

template <int DT>
__device__ __forceinline__ float mq_o_scale(int vx) {
  if constexpr (DT == PKV_KV_F16)
    return 1.0f / (1 << kPShift);
  else if constexpr (DT == PKV_KV_BF16 || DT == PKV_KV_F32)
    return 1.0f;
  else
    return pow2i(vx - kPShift);
}

// Dim of O row r, element e (0: c0/c1, 2: c2/c3) in lane 4 gid + tig (as decode.cu).
template <int DT>
__device__ __forceinline__ int mq_dim(int r, int e, int gid) {
  if constexpr (DT == PKV_KV_F32)  // dims 32j + 4gid + {0..3} (CUDA-core accumulation)
    return 32 * (r >> 1) + 4 * gid + 2 * (r & 1) + (e ? 1 : 0);
  else if constexpr (DT != PKV_KV_Q8_0)
    return 16 * r + gid + (e ? 8 : 0);
  else
    return 16 * r + 2 * gid + (e ? 1 : 0);
}

// One column's query (qv, nullptr for an unused column) into the score B
// operands of the lane (part `lo`), with the dims mapping of the single-query
// kernel, normalised by a power of two per column (f16, q8_0).
template <int DT>
__device__ __forceinline__ void mq_load_column(const float* qv, float qscale, bool lo, int tig,
                                               uint32_t (&qb)[mq_steps<DT>()][2], int& e2) {
  if constexpr (DT == PKV_KV_BF16) {
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      float2 x = make_float2(0.f, 0.f);
      if (qv) x = __ldg(reinterpret_cast<const float2*>(qv + 8 * ks + 2 * tig));
      qb[ks][0] = tf32_part(x.x * qscale, lo);
      qb[ks][1] = tf32_part(x.y * qscale, lo);
    }
    e2 = 0;
  } else {
    float v[32];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (qv) {
        if constexpr (DT == PKV_KV_F16) {
          const float2 a = __ldg(reinterpret_cast<const float2*>(qv + 16 * ks + 2 * tig));
          const float2 b = __ldg(reinterpret_cast<const float2*>(qv + 16 * ks + 8 + 2 * tig));
          x = make_float4(a.x, a.y, b.x, b.y);
        } else {
          x = __ldg(reinterpret_cast<const float4*>(qv + 16 * ks + 4 * tig));
        }
      }
      v[4 * ks] = x.x * qscale;
      v[4 * ks + 1] = x.y * qscale;
      v[4 * ks + 2] = x.z * qscale;
      v[4 * ks + 3] = x.w * qscale;
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));  // the column's 128 dims: over tig
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    e2 = 0;
    if (amax > 0.f && amax <= 3.0e38f) {
      int ex;
      frexpf(amax, &ex);
      e2 = ex - 14;
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qb[ks][0] = split_f16x2(ldexpf(v[4 * ks], -e2), ldexpf(v[4 * ks + 1], -e2), lo);
      qb[ks][1] = split_f16x2(ldexpf(v[4 * ks + 2], -e2), ldexpf(v[4 * ks + 3], -e2), lo);
    }
  }
}

// Per-unit work of a pass: columns c < nc are (query q0 + c / G, head c % G);
// pf is the page's first token; col_hi[t] / col_lo[t] bound the attended
// positions of the lane's score column 4t + tig (empty for unused columns).
template <int DT, int NT>
__device__ __forceinline__ void mq_process_unit(const uint8_t* st, const uint8_t* sc, int pf,
                                                const int (&col_lo)[2], const int (&col_hi)[2],
                                                int slot_lo, int slot_hi, int nc, int lane,
                                                MqState<DT, NT>& S) {
  using TL = Tiles<DT>;
  const int gid = lane >> 2, tig = lane & 3;
  const int ld_tok = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int ld_chunk = lane >> 4;
  const uint32_t kt = smem_addr(st), vt = kt + TL::kData;

  // ---- scores of the lane's columns 4t + tig, tokens gid and gid + 8
  float s[NT][2];
  if constexpr (DT == PKV_KV_F32) {
    // CUDA cores, fp32: dot products of the column's q (shared buffer) with K
    // rows gid and gid + 8, four partial sums each
    float4 acc[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int c = 0; c < 32; ++c) {  // 16-byte chunks of the 128 dims
      const float4 k0 = *reinterpret_cast<const float4*>(st + tile_offset<DT>(gid, c));
      const float4 k1 = *reinterpret_cast<const float4*>(st + tile_offset<DT>(gid + 8, c));
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float4 qv = *reinterpret_cast<const float4*>(S.qs + (4 * t + tig) * kQStride + 4 * c);
        acc[t][0] = make_float4(fmaf(qv.x, k0.x, acc[t][0].x), fmaf(qv.y, k0.y, acc[t][0].y),
                                fmaf(qv.z, k0.z, acc[t][0].z), fmaf(qv.w, k0.w, acc[t][0].w));
        acc[t][1] = make_float4(fmaf(qv.x, k1.x, acc[t][1].x), fmaf(qv.y, k1.y, acc[t][1].y),
                                fmaf(qv.z, k1.z, acc[t][1].z), fmaf(qv.w, k1.w, acc[t][1].w));
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      s[t][0] = (acc[t][0].x + acc[t][0].y) + (acc[t][0].z + acc[t][0].w);
      s[t][1] = (acc[t][1].x + acc[t][1].y) + (acc[t][1].z + acc[t][1].w);
    }
  } else if constexpr (DT == PKV_KV_BF16) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c2 = 0; c2 < 8; ++c2) {
      uint32_t w0, w1, w2, w3;
      ldsm_x4(kt + tile_offset<DT>(ld_tok, 2 * c2 + ld_chunk), w0, w1, w2, w3);
      mma_1688_tf32(c, w0 << 16, w1 << 16, w0 & 0xffff0000u, w1 & 0xffff0000u,
                    S.qb[0][2 * c2][0], S.qb[0][2 * c2][1]);
      mma_1688_tf32(c, w2 << 16, w3 << 16, w2 & 0xffff0000u, w3 & 0xffff0000u,
                    S.qb[0][2 * c2 + 1][0], S.qb[0][2 * c2 + 1][1]);
    }
    s[0][0] = c[0] + c[1];
    s[0][1] = c[2] + c[3];
  } else if constexpr (DT == PKV_KV_F16) {
    float c[NT][4] = {};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kt + tile_offset<DT>(ld_tok, 2 * ks + ld_chunk), a0, a1, a2, a3);
#pragma unroll
      for (int t = 0; t < NT; ++t) mma_16816(c[t], a0, a1, a2, a3, S.qb[t][ks][0], S.qb[t][ks][1]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      s[t][0] = c[t][0] + c[t][1];
      s[t][1] = c[t][2] + c[t][3];
    }
  } else {
    const uint2 k0 = *reinterpret_cast<const uint2*>(sc + gid * 8);
    const uint2 k1 = *reinterpret_cast<const uint2*>(sc + (gid + 8) * 8);
#pragma unroll
    for (int t = 0; t < NT; ++t) s[t][0] = s[t][1] = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t w0, w1, w2, w3;
      ldsm_x4(kt + tile_offset<DT>(ld_tok, 2 * b + ld_chunk), w0, w1, w2, w3);
      const uint32_t a0 = codes_to_f16x2<kSelB01>(w0), a1 = codes_to_f16x2<kSelB01>(w1);
      const uint32_t a2 = codes_to_f16x2<kSelB23>(w0), a3 = codes_to_f16x2<kSelB23>(w1);
      const uint32_t b0 = codes_to_f16x2<kSelB01>(w2), b1 = codes_to_f16x2<kSelB01>(w3);
      const uint32_t b2 = codes_to_f16x2<kSelB23>(w2), b3 = codes_to_f16x2<kSelB23>(w3);
      const uint32_t kp = __byte_perm(b < 2 ? k0.x : k0.y, b < 2 ? k1.x : k1.y,
                                      (b & 1) ? 0x7632 : 0x5410);
      const float2 ksc = __half22float2(*reinterpret_cast<const __half2*>(&kp));
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(c, a0, a1, a2, a3, S.qb[t][2 * b][0], S.qb[t][2 * b][1]);
        mma_16816(c, b0, b1, b2, b3, S.qb[t][2 * b + 1][0], S.qb[t][2 * b + 1][1]);
        s[t][0] = fmaf(ksc.x, c[0] + c[1], s[t][0]);
        s[t][1] = fmaf(ksc.y, c[2] + c[3], s[t][1]);
      }
    }
  }

  // ---- masks and online softmax, per score column
  float p[NT][2], alpha[NT];
  bool grow_any = false;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int c = 4 * t + tig;
    if (c < nc) {  // attended positions [col_lo, col_hi) of this column
      const int t0 = pf + gid, t1 = pf + gid + 8;
      s[t][0] = (t0 >= col_lo[t] && t0 < col_hi[t] && gid >= slot_lo && gid < slot_hi)
                    ? s[t][0] * S.qexp[t] : -INFINITY;
      s[t][1] = (t1 >= col_lo[t] && t1 < col_hi[t] && gid + 8 >= slot_lo && gid + 8 < slot_hi)
                    ? s[t][1] * S.qexp[t] : -INFINITY;
    } else {
      s[t][0] = s[t][1] = 0.f;  // an unused column: finite, never written
    }
    float mx = fmaxf(s[t][0], s[t][1]);
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
    const bool grow = mx > S.m[t] + 8.0f;  // never for a column with no token here
    alpha[t] = grow ? ex2_ftz(S.m[t] - mx) : 1.0f;
    if (grow) S.m[t] = mx;
    grow_any |= grow;
  }
  if (__any_sync(kFull, grow_any)) {
    // V-columns 2tig and 2tig + 1 take the alphas of those score columns
    // (held by lanes tig' = column % 4, score n-tile column / 4)
    float av[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = 2 * tig + e;
      float a0 = __shfl_sync(kFull, alpha[0], c & 3);
      if constexpr (NT == 2) {
        const float a1 = __shfl_sync(kFull, alpha[1], c & 3);
        a0 = c < 4 ? a0 : a1;
      }
      av[e] = a0;
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) S.l[t] *= alpha[t];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      S.o[r][0] *= av[0];
      S.o[r][1] *= av[1];
      S.o[r][2] *= av[0];
      S.o[r][3] *= av[1];
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const float mu = S.m[t] == -INFINITY ? 0.f : S.m[t];  // all -inf here: p = 0
    p[t][0] = ex2_ftz(s[t][0] - mu);
    p[t][1] = ex2_ftz(s[t][1] - mu);
    S.l[t] += p[t][0] + p[t][1];
  }

  if constexpr (DT == PKV_KV_F32) {
    // O += p_t V_t on CUDA cores: lane 4 gid + tig keeps V-columns 2tig + e
    // (e = 0, 1) at dims 32 j + 4 gid + {0..3}.  Column c's p_t sits in lane
    // 4 (t mod 8) + (c mod 4), score tile c / 4 (one shuffle per tile, then a
    // select).  Slots no column attends are skipped (their V may be NaN).
    const uint8_t* vs = st + TL::kData;
    const int c0 = 2 * tig, c1 = 2 * tig + 1;
    auto accumulate = [&](int t) {
      const int hi = t >> 3;
      float pe[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = e ? c1 : c0;
        const int src = 4 * (t & 7) + (c & 3);
        float v = __shfl_sync(kFull, hi ? p[0][1] : p[0][0], src);
        if constexpr (NT == 2) {
          const float v1 = __shfl_sync(kFull, hi ? p[1][1] : p[1][0], src);
          if (c >= 4) v = v1;
        } else {
          if (c >= 4) v = 0.f;  // 4 columns: V-columns 4..7 unused
        }
        pe[e] = c < nc ? v : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 x = *reinterpret_cast<const float4*>(vs + tile_offset<DT>(t, 8 * j + gid));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          S.o[2 * j][e] = fmaf(pe[e], x.x, S.o[2 * j][e]);
          S.o[2 * j][e + 2] = fmaf(pe[e], x.y, S.o[2 * j][e + 2]);
          S.o[2 * j + 1][e] = fmaf(pe[e], x.z, S.o[2 * j + 1][e]);
          S.o[2 * j + 1][e + 2] = fmaf(pe[e], x.w, S.o[2 * j + 1][e + 2]);
        }
      }
    };
    if (slot_lo == 0 && slot_hi == kPage) {
#pragma unroll
      for (int t = 0; t < kPage; ++t) accumulate(t);
    } else {
      for (int t = slot_lo; t < slot_hi; ++t) accumulate(t);
    }
    __syncwarp();
    return;
  }

  // ---- P^T operands: V-column gid = score column gid (n-tile gid / 4, lanes
  // tig' = gid % 4): tokens 2tig, 2tig+1 from lanes 8 tig + gid % 4 and
  // 8 tig + 4 + gid % 4, tokens + 8 from their second scores
  const int src = 8 * tig + (gid & 3);
  float pa = __shfl_sync(kFull, p[0][0], src), pb = __shfl_sync(kFull, p[0][0], src + 4);
  float pc = __shfl_sync(kFull, p[0][1], src), pd = __shfl_sync(kFull, p[0][1], src + 4);
  if constexpr (NT == 2) {
    const float qa = __shfl_sync(kFull, p[1][0], src), qb2 = __shfl_sync(kFull, p[1][0], src + 4);
    const float qc = __shfl_sync(kFull, p[1][1], src), qd = __shfl_sync(kFull, p[1][1], src + 4);
    if (gid >= 4) {
      pa = qa;
      pb = qb2;
      pc = qc;
      pd = qd;
    }
  } else {
    if (gid >= 4) pa = pb = pc = pd = 0.f;  // 4 columns: V-columns 4..7 unused
  }
  if (gid >= nc) pa = pb = pc = pd = 0.f;
  const int t0 = 2 * tig;

  // ---- values: each part of P is its own B operand into the same accumulator
  if constexpr (DT == PKV_KV_F16 || DT == PKV_KV_BF16) {
    // V values of slots no column attends may be anything (NaN * 0 is NaN):
    // masked in the registers, the stage is shared by readers.  Fragment
    // words hold tokens (2tig, 2tig + 1) [w0, w2] or (2tig + 8, 2tig + 9) [w1, w3].
    auto ok = [&](int t) { return t >= slot_lo && t < slot_hi; };
    const bool partial = slot_lo > 0 || slot_hi < kPage;  // warp-uniform
    const uint32_t vm_lo = (ok(t0) ? 0x0000ffffu : 0u) | (ok(t0 + 1) ? 0xffff0000u : 0u);
    const uint32_t vm_hi = (ok(t0 + 8) ? 0x0000ffffu : 0u) | (ok(t0 + 9) ? 0xffff0000u : 0u);
    if constexpr (DT == PKV_KV_F16) {
      constexpr float kUp = static_cast<float>(1 << kPShift);
      const uint32_t h0 = split_f16x2(pa * kUp, pb * kUp, false);
      const uint32_t h1 = split_f16x2(pc * kUp, pd * kUp, false);
      const uint32_t l0 = split_f16x2(pa * kUp, pb * kUp, true);
      const uint32_t l1 = split_f16x2(pc * kUp, pd * kUp, true);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t w0, w1, w2, w3;
        ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * mt + ld_chunk), w0, w1, w2, w3);
        if (partial) {
          w0 &= vm_lo;
          w1 &= vm_hi;
          w2 &= vm_lo;
          w3 &= vm_hi;
        }
        mma_16816(S.o[mt], w0, w2, w1, w3, h0, h1);
        mma_16816(S.o[mt], w0, w2, w1, w3, l0, l1);
      }
    } else {
      const uint32_t h0 = tf32_part(pa, false), h1 = tf32_part(pb, false);
      const uint32_t h8 = tf32_part(pc, false), h9 = tf32_part(pd, false);
      const uint32_t l0 = tf32_part(pa, true), l1 = tf32_part(pb, true);
      const uint32_t l8 = tf32_part(pc, true), l9 = tf32_part(pd, true);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t w0, w1, w2, w3;
        ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * mt + ld_chunk), w0, w1, w2, w3);
        if (partial) {
          w0 &= vm_lo;
          w1 &= vm_hi;
          w2 &= vm_lo;
          w3 &= vm_hi;
        }
        const uint32_t x0 = w0 << 16, x1 = w2 << 16, x2 = w0 & 0xffff0000u, x3 = w2 & 0xffff0000u;
        const uint32_t y0 = w1 << 16, y1 = w3 << 16, y2 = w1 & 0xffff0000u, y3 = w3 & 0xffff0000u;
        mma_1688_tf32(S.o[mt], x0, x1, x2, x3, h0, h1);
        mma_1688_tf32(S.o[mt], x0, x1, x2, x3, l0, l1);
        mma_1688_tf32(S.o[mt], y0, y1, y2, y3, h8, h9);
        mma_1688_tf32(S.o[mt], y0, y1, y2, y3, l8, l9);
      }
    }
  } else if constexpr (DT == PKV_KV_Q8_0) {
    uint4 va = *reinterpret_cast<const uint4*>(sc + TL::kScale + t0 * 8);
    uint4 vb = *reinterpret_cast<const uint4*>(sc + TL::kScale + (t0 + 8) * 8);
    if (slot_lo > 0 || slot_hi < kPage) {  // unattended slots: P = 0, scales may be NaN
      if (t0 < slot_lo || t0 >= slot_hi) va.x = va.y = 0u;
      if (t0 + 1 < slot_lo || t0 + 1 >= slot_hi) va.z = va.w = 0u;
      if (t0 + 8 < slot_lo || t0 + 8 >= slot_hi) vb.x = vb.y = 0u;
      if (t0 + 9 < slot_lo || t0 + 9 >= slot_hi) vb.z = vb.w = 0u;
    }
    uint32_t mb = abs_max_f16x2(abs_max_f16x2(va.x, va.y), abs_max_f16x2(va.z, va.w));
    mb = abs_max_f16x2(mb, abs_max_f16x2(abs_max_f16x2(vb.x, vb.y), abs_max_f16x2(vb.z, vb.w)));
    mb &= 0x7fff7fffu;
    uint32_t m16 = max(mb & 0xffffu, mb >> 16);
    m16 = max(m16, __shfl_xor_sync(kFull, m16, 1));
    m16 = max(m16, __shfl_xor_sync(kFull, m16, 2));
    const int vx = static_cast<int>(m16 >> 10) - 14;
    if (vx > S.vx) {  // warp-uniform
      const float r = pow2i(max(S.vx - vx, -126));
#pragma unroll
      for (int rr = 0; rr < 8; ++rr)
#pragma unroll
        for (int e = 0; e < 4; ++e) S.o[rr][e] *= r;
      S.vx = vx;
    }
    const float up = pow2i(kPShift - S.vx);
    const float2 pab = make_float2(pa * up, pb * up), pcd = make_float2(pc * up, pd * up);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t sel = (b & 1) ? 0x7632 : 0x5410;
      const uint32_t sa = __byte_perm(b < 2 ? va.x : va.y, b < 2 ? va.z : va.w, sel);
      const uint32_t sb = __byte_perm(b < 2 ? vb.x : vb.y, b < 2 ? vb.z : vb.w, sel);
      const float2 x01 = __fmul2_rn(pab, __half22float2(*reinterpret_cast<const __half2*>(&sa)));
      const float2 x23 = __fmul2_rn(pcd, __half22float2(*reinterpret_cast<const __half2*>(&sb)));
      const uint32_t h0 = split_f16x2(x01.x, x01.y, false), h1 = split_f16x2(x23.x, x23.y, false);
      const uint32_t l0 = split_f16x2(x01.x, x01.y, true), l1 = split_f16x2(x23.x, x23.y, true);
      uint32_t w0, w1, w2, w3;
      ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * b + ld_chunk), w0, w1, w2, w3);
      const uint32_t e0 = codes_to_f16x2<kSelB02>(w0), e1 = codes_to_f16x2<kSelB13>(w0);
      const uint32_t e2 = codes_to_f16x2<kSelB02>(w1), e3 = codes_to_f16x2<kSelB13>(w1);
      mma_16816(S.o[2 * b], e0, e1, e2, e3, h0, h1);
      mma_16816(S.o[2 * b], e0, e1, e2, e3, l0, l1);
      const uint32_t f0 = codes_to_f16x2<kSelB02>(w2), f1 = codes_to_f16x2<kSelB13>(w2);
      const uint32_t f2 = codes_to_f16x2<kSelB02>(w3), f3 = codes_to_f16x2<kSelB13>(w3);
      mma_16816(S.o[2 * b + 1], f0, f1, f2, f3, h0, h1);
      mma_16816(S.o[2 * b + 1], f0, f1, f2, f3, l0, l1);
    }
  }
  __syncwarp();
}

// Merge the pieces k0..k1 of segment j (slots k + j, kMqCols columns each)
// for the columns c0 .. c0 + kCols - 1 that are below nc; one warp, lane l:
// dims 4l..4l+3; column c goes to out_col(c).  The loads of kBatch pieces of
// all kCols columns are issued together (one L2 round trip per batch).
template <int kCols, int kBatch, class OutCol>
__device__ __forceinline__ void mq_merge_segment_warp(const float* part_ml, const float* part_acc,
                                                      long long j, int k0, int k1, int c0, int nc,
                                                      OutCol&& out_col, int lane) {
  float M[kCols], Ls[kCols];
  float4 A[kCols];
#pragma unroll
  for (int u = 0; u < kCols; ++u) {
    M[u] = -INFINITY;
    Ls[u] = 0.f;
    A[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int kk = k0; kk <= k1; kk += kBatch) {
    float m[kBatch][kCols], l[kBatch][kCols];
    float4 x[kBatch][kCols];
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
#pragma unroll
      for (int u = 0; u < kCols; ++u) {
        const bool in = kk + b <= k1 && c0 + u < nc;
        const long long slot = (kk + b + j) * kMqCols + c0 + u;
        m[b][u] = in ? __ldcg(part_ml + slot * 2) : -INFINITY;
        l[b][u] = in ? __ldcg(part_ml + slot * 2 + 1) : 0.f;
        x[b][u] = in ? __ldcg(reinterpret_cast<const float4*>(part_acc + slot * kD) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int u = 0; u < kCols; ++u) {
      float bm = M[u];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) bm = fmaxf(bm, m[b][u]);
      if (bm == -INFINITY) continue;  // no token of this query in any piece so far
      const float sc = exp2f(M[u] - bm);
      Ls[u] *= sc;
      A[u] = make_float4(A[u].x * sc, A[u].y * sc, A[u].z * sc, A[u].w * sc);
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const float w = exp2f(m[b][u] - bm);
        Ls[u] = fmaf(w, l[b][u], Ls[u]);
        A[u] = make_float4(fmaf(w, x[b][u].x, A[u].x), fmaf(w, x[b][u].y, A[u].y),
                           fmaf(w, x[b][u].z, A[u].z), fmaf(w, x[b][u].w, A[u].w));
      }
      M[u] = bm;
    }
  }
#pragma unroll
  for (int u = 0; u < kCols; ++u) {
    if (c0 + u >= nc) continue;
    const float inv = 1.0f / Ls[u];
    *reinterpret_cast<float4*>(out_col(c0 + u) + lane * 4) =
        make_float4(A[u].x * inv, A[u].y * inv, A[u].z * inv, A[u].w * inv);
  }
}

// --------------------------------------------------------------- kernel ----
template <int DT>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_mq_kernel(const __grid_constant__ DecodeArgs a,
                           const __grid_constant__ TileMaps maps) {
  using TL = Tiles<DT>;
  using SM = MqSmem<DT>;
  constexpr int R = TL::kRing;
  constexpr int NT = mq_tiles<DT>();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((SM::kAlign - (smem_addr(smem_raw) & (SM::kAlign - 1))) &
                              (SM::kAlign - 1));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  // [0] abort  [1] warps arrived at the current piece end  [2] merge-buffer generation
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + SM::kCtl);
  int* row_start = reinterpret_cast<int*>(smem + SM::kRows);
  int* lens = row_start + a.num_rows + 1;
  const uint32_t bar0 = smem_addr(smem + SM::kBar) + warp * R * 8;
  uint8_t* ring = smem + static_cast<size_t>(warp) * R * TL::kCodes;
  uint8_t* ring_sc = smem + SM::kScl + static_cast<size_t>(warp) * R * TL::kScales;
  const int G = a.n_q / a.n_kv;
  const int nc = a.nq * G;  // columns of this pass
  // the pages read cover the first query's window: [L - q_len + 1 - W, L)
  const int plan_window = a.window > 0 ? a.window + a.q_len - 1 : 0;

  if (threadIdx.x == 0) {
    // the tensor maps are kernel parameters, not written by an earlier kernel
    prefetch_tensormap(&maps.k);
    prefetch_tensormap(&maps.v);
    ctl[0] = 0;
    ctl[1] = 0;
    ctl[2] = 0;
    mbar_init(smem_addr(smem + SM::kStall), 1);
  }
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, plan_window,
            blockIdx.x == 0 ? a.status : nullptr, lens, row_start, a.q_len);
  const bool stalled = test_stall(smem_addr(smem + SM::kStall), a.test_stall_ns, ctl, a.status);
  int* pc = lens + a.num_rows;
  plan_split(row_start, a.num_rows, a.n_kv, gridDim.x, a.aligned_split,
             reinterpret_cast<Split*>(smem + SM::kSplit), pc);
  // read from shared memory where used (at each piece): no registers held across the loop
  const Split* sp = reinterpret_cast<const Split*>(smem + SM::kSplit);
  const int k = blockIdx.x;
  long long c_begin, c_end;
  chunk_range(*sp, k, row_start, pc, a.num_rows, a.n_kv, c_begin, c_end);

  // Rows without tokens (or shorter than q_len): zero outputs for this pass.
  if (k == 0) {
    for (int i = 0; i < a.num_rows; ++i)
      if (row_start[i + 1] == row_start[i])
        for (int jj = 0; jj < a.nq; ++jj)
          for (int e = threadIdx.x; e < a.n_q * kD; e += kThreads)
            a.out[((static_cast<long long>(i) * a.q_len + a.q0 + jj) * a.n_q) * kD + e] = 0.f;
  }

  const long long first = c_begin + warp;
  const int n_units = first < c_end ? static_cast<int>((c_end - first + kWarps - 1) / kWarps) : 0;

  // Unit descriptors, 32 at a time: page, KV head, row, page index in the row.
  auto fetch = [&](int base, int& pg, int& hh, int& row, int& pidx) {
    const int u = base + lane;
    pg = hh = row = pidx = 0;
    if (u < n_units) {
      const long long x = first + static_cast<long long>(u) * kWarps;
      const int i = row_of(row_start, a.num_rows, a.n_kv, x);
      const int npg = row_start[i + 1] - row_start[i];
      const int off = static_cast<int>(x - static_cast<long long>(a.n_kv) * row_start[i]);
      hh = off / npg;
      const int p = off - hh * npg;
      int pabs = window_start(lens[i], plan_window) / kPage + p;  // block-table entry
      int page = __ldg(a.block_table + static_cast<long long>(i) * a.bt_stride + pabs);
      if (page < 0 || page >= a.num_pages) {
        record_status(a.status, PKV_DEV_BAD_PAGE);
        page = 0;
        pabs = -1;  // take no append
      }
      pg = page;
      row = i;
      pidx = pabs;
    }
  };
  int c_pg, c_h, c_row, c_p, n_pg, n_h, n_row, n_p;
  int batch = 0;
  fetch(0, c_pg, c_h, c_row, c_p);
  int issued = 0;
  const uint64_t policy = policy_evict_first();

  auto issue = [&]() {
    const int u = issued;
    if (u >= batch + 32) {
      c_pg = n_pg;
      c_h = n_h;
      c_row = n_row;
      c_p = n_p;
      batch += 32;
      fetch(batch + 32, n_pg, n_h, n_row, n_p);
    }
    const int jj = u - batch;
    const int pg = __shfl_sync(kFull, c_pg, jj);
    const int hh = __shfl_sync(kFull, c_h, jj);
    const int pabs = __shfl_sync(kFull, c_p, jj);
    if (a.k_new != nullptr && pabs >= 0) {  // first pass: new tokens of this page first
      const int row = __shfl_sync(kFull, c_row, jj);
      const int L = lens[row], first_new = L - a.q_len;
      const int lo = max(first_new, pabs * kPage), hi = min(L, pabs * kPage + kPage);
      for (int pos = lo; pos < hi; ++pos)
        append_token<DT>(a, static_cast<long long>(row) * a.q_len + (pos - first_new), hh, pg,
                         pos % kPage, lane);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const int s = u % R;
      const uint32_t bar = bar0 + 8 * s;
      const uint32_t dst = smem_addr(ring + s * TL::kCodes);
      const int z = pg * a.n_kv + hh;
      mbar_arrive_expect_tx(bar, TL::kTx);
      tma_load_tile<DT>(dst, &maps.k, z, bar, policy);
      tma_load_tile<DT>(dst + TL::kData, &maps.v, z, bar, policy);
      if constexpr (DT == PKV_KV_Q8_0) {
        const uint32_t sdst = smem_addr(ring_sc + s * TL::kScales);
        const size_t unit = static_cast<size_t>(z);
        bulk_g2s(sdst, a.k_scales + unit * TL::kScale, TL::kScale, bar, policy);
        bulk_g2s(sdst + TL::kScale, a.v_scales + unit * TL::kScale, TL::kScale, bar, policy);
      }
    }
    ++issued;
  };
  while (issued < n_units && issued < R) issue();
  fetch(32, n_pg, n_h, n_row, n_p);  // the next batch, once the first copies are on their way

  float* mrg_acc = reinterpret_cast<float*>(smem + SM::kMrgAcc);
  float* mrg_ml = reinterpret_cast<float*>(smem + SM::kMrgMl);
  int consumed = 0;
  bool aborted = stalled;
  MqState<DT, NT> S;
  S.qs = reinterpret_cast<float*>(smem + SM::kQ) + warp * kWarpCols * kQStride;  // f32 KV only

  int piece = 0;
  for (long long x = c_begin; x < c_end; ++piece) {
    const int i = row_of(row_start, a.num_rows, a.n_kv, x);
    const int npg = row_start[i + 1] - row_start[i];
    const long long row_base = static_cast<long long>(a.n_kv) * row_start[i];
    const int h = static_cast<int>(x - row_base) / npg;  // x - row_base < n_kv * npg < 2^31
    const long long seg_start = row_base + static_cast<long long>(h) * npg;
    const long long seg_end = seg_start + npg;
    const long long b = min(seg_end, c_end);
    const int L = lens[i];
    const int p0 = window_start(L, plan_window) / kPage;
    const long long j = static_cast<long long>(i) * a.n_kv + h;
    int k0, k1;
    segment_chunks(*sp, i, h, row_start, pc, a.num_rows, a.n_kv, k0, k1);

    // the lane's score columns 4t + tig: attended positions [col_lo, col_hi)
    int col_lo[2] = {0, 0}, col_hi[2] = {0, 0};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int c = 4 * t + tig;
      if (c < nc) {
        const int P = L - a.q_len + a.q0 + c / G;
        col_hi[t] = P + 1;
        col_lo[t] = window_start(P + 1, a.window);
      }
    }
    // the warp's slots of interest in any page: union of the pass's columns
    const int pos_lo = window_start(L - a.q_len + a.q0 + 1, a.window);
    const int pos_hi = L - a.q_len + a.q0 + a.nq;  // last query of the pass + 1
    if constexpr (DT == PKV_KV_F32) {
      // the pass's columns times scale * log2 e into the warp's buffer (zeros
      // for unused columns): lane l writes dims 4l .. 4l + 3 of each
      __syncwarp();  // the previous piece's reads are done
#pragma unroll
      for (int c = 0; c < kWarpCols; ++c) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < nc)
          x = __ldg(reinterpret_cast<const float4*>(
                        a.q + ((static_cast<long long>(i) * a.q_len + a.q0 + c / G) * a.n_q + h * G +
                               c % G) * kD) + lane);
        *reinterpret_cast<float4*>(S.qs + c * kQStride + 4 * lane) =
            make_float4(x.x * a.qscale, x.y * a.qscale, x.z * a.qscale, x.w * a.qscale);
      }
      __syncwarp();
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        S.qexp[t] = 1.0f;
        S.m[t] = -INFINITY;
        S.l[t] = 0.f;
      }
    } else {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int cq = 4 * t + (gid >> 1);  // the column whose query this lane loads
        const float* qv = cq < nc
                              ? a.q + ((static_cast<long long>(i) * a.q_len + a.q0 + cq / G) * a.n_q +
                                       h * G + cq % G) * kD
                              : nullptr;
        int e2;
        mq_load_column<DT>(qv, a.qscale, (gid & 1) != 0, tig, S.qb[t], e2);
        S.qexp[t] = ldexpf(1.0f, __shfl_sync(kFull, e2, 8 * tig));  // lane 8 tig: column 4t + tig
        S.m[t] = -INFINITY;
        S.l[t] = 0.f;
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) S.o[r][e] = 0.f;
    S.vx = kNoScale;

    const int r0 = static_cast<int>((x - c_begin) % kWarps);
    for (long long pos = x + ((warp - r0 + kWarps) % kWarps); pos < b; pos += kWarps) {
      const int u = static_cast<int>((pos - first) / kWarps);
      const int s = u % R;
      bool ok = !aborted && mbar_wait_bounded(bar0 + 8 * s, (u / R) & 1, ctl);
      ok = __all_sync(kFull, ok);
      if (!ok) {
        if (!aborted && lane == 0 && !ctl[0]) {
          ctl[0] = 1;
          record_status(a.status, PKV_DEV_TIMEOUT);
        }
        aborted = true;
        continue;
      }
      consumed = u + 1;
      const int pf = (p0 + static_cast<int>(pos - seg_start)) * kPage;  // page's first token
      const int slot_lo = max(0, pos_lo - pf), slot_hi = min(kPage, pos_hi - pf);
      mq_process_unit<DT, NT>(ring + s * TL::kCodes, ring_sc + s * TL::kScales, pf, col_lo, col_hi,
                          slot_lo, slot_hi, nc, lane, S);
      if (issued < n_units) issue();
    }

    // ---- piece end (as the single-query kernel, kWarpCols columns)
    float l_tot[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float v = S.l[t];
      v += __shfl_xor_sync(kFull, v, 4);
      v += __shfl_xor_sync(kFull, v, 8);
      v += __shfl_xor_sync(kFull, v, 16);
      l_tot[t] = v;
    }
    const bool final_piece = (b == c_end);
    int okb = 1;
    if (lane == 0) okb = wait_merge_buffer(ctl, piece);
    okb = __shfl_sync(kFull, okb, 0);
    if (!okb && !aborted) {
      if (lane == 0 && !ctl[0]) {
        ctl[0] = 1;
        record_status(a.status, PKV_DEV_TIMEOUT);
      }
      aborted = true;
    }
    if (gid == 0) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int c = 4 * t + tig;
        mrg_ml[(warp * kWarpCols + c) * 2] = aborted ? -INFINITY : S.m[t];
        mrg_ml[(warp * kWarpCols + c) * 2 + 1] = l_tot[t];
      }
    }
    {
      const float osc = mq_o_scale<DT>(S.vx);
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 2 * tig + (e & 1);
          mrg_acc[(warp * kWarpCols + c) * kD + mq_dim<DT>(r, e & 2, gid)] = S.o[r][e] * osc;
        }
    }
    const bool whole = (k0 == k1);
    auto out_col = [&](int c) {
      return a.out + ((static_cast<long long>(i) * a.q_len + a.q0 + c / G) * a.n_q + h * G +
                      c % G) * kD;
    };
    // merge the 4 warps' states of column c (dim d): base-2 weights
    auto merge_dim = [&](int c, int d, float& M, float& Ls, float& A) {
      M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mrg_ml[(w * kWarpCols + c) * 2]);
      Ls = 0.f;
      A = 0.f;
      if (M == -INFINITY) return;  // no token of this query in the piece
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(mrg_ml[(w * kWarpCols + c) * 2] - M);
        Ls = fmaf(f, mrg_ml[(w * kWarpCols + c) * 2 + 1], Ls);
        A = fmaf(f, mrg_acc[(w * kWarpCols + c) * kD + d], A);
      }
    };
    auto write_piece_dim = [&](int c, int d, float M, float Ls, float A) {
      if (whole) {
        out_col(c)[d] = A / Ls;
      } else {
        const long long slot = (k + j) * kMqCols + c;
        a.part_acc[slot * kD + d] = A;
        if (d == 0) {
          a.part_ml[slot * 2] = M;
          a.part_ml[slot * 2 + 1] = Ls;
        }
      }
    };
    if (final_piece) {
      named_barrier(1, kThreads);
      const bool live = !ctl[0];
      const int d = threadIdx.x;
      if (live) {
        for (int c = 0; c < nc; ++c) {
          float M, Ls, A;
          merge_dim(c, d, M, Ls, A);
          write_piece_dim(c, d, M, Ls, A);
        }
      }
      const bool counted = live && !whole && a.flags != nullptr;
      named_barrier(1, kThreads);
      if (threadIdx.x == 0) {
        int seg_last = 0;
        // the CTA's partial (ordered by the barrier) is released by the
        // arrival; the last to arrive acquires every other piece's
        if (counted) seg_last = atomic_add_acq_rel(mq_counter(a.flags, j, 0), 1) == k1 - k0;
        ctl[1] = seg_last;
      }
      named_barrier(1, kThreads);
      if (ctl[1]) {  // the CTA merges the segment: warp w takes columns 2w, 2w + 1
        mq_merge_segment_warp<2, 4>(a.part_ml, a.part_acc, j, k0, k1, 2 * warp, nc, out_col,
                                    lane);
        if (threadIdx.x == 0) *mq_counter(a.flags, j, 0) = 0;
      }
    } else {
      __syncwarp();
      int lastw = 0;
      if (lane == 0) {
        __threadfence_block();
        lastw = atomicAdd(const_cast<int*>(&ctl[1]), 1) == kWarps - 1;
      }
      lastw = __shfl_sync(kFull, lastw, 0);
      if (lastw) {
        __threadfence_block();
        const bool live = !ctl[0];
        if (live) {
          for (int c = 0; c < nc; ++c)
            for (int d = lane; d < kD; d += 32) {
              float M, Ls, A;
              merge_dim(c, d, M, Ls, A);
              write_piece_dim(c, d, M, Ls, A);
            }
        }
        __syncwarp();
        if (lane == 0) {
          ctl[1] = 0;
          __threadfence_block();
          ctl[2] = piece + 1;
        }
        if (live && !whole && a.flags != nullptr) {
          __syncwarp();
          int seg_last = 0;
          // the warp's partial (ordered by __syncwarp) is released by the arrival
          if (lane == 0) seg_last = atomic_add_acq_rel(mq_counter(a.flags, j, 0), 1) == k1 - k0;
          seg_last = __shfl_sync(kFull, seg_last, 0);
          if (seg_last) {
            __syncwarp();  // lane 0's acquire, ordered for the warp
            mq_merge_segment_warp<kWarpCols, 1>(a.part_ml, a.part_acc, j, k0, k1, 0, nc, out_col,
                                              lane);
            if (lane == 0) *mq_counter(a.flags, j, 0) = 0;
          }
        }
      }
    }
    x = b;
  }

  if (aborted || ctl[0]) {
    const int zero = 0;
    for (int u = consumed > issued - R ? consumed : issued - R; u < issued; ++u)
      if (u >= 0) mbar_wait_bounded(bar0 + 8 * (u % R), (u / R) & 1, &zero);
  }
}

// -------------------------------------------------- shared-page kernel ----
// With more than 8 (query, head) columns in a pass (more than 4 for bf16) a
// team of TS warps (2 or 4) reads every page of its chunk together, warp w of
// the team taking columns [w CW, (w + 1) CW): a page is copied once for up to
// TS * CW columns.  A CTA holds 4 / TS teams, each with its own chunk (chunk
// b * teams + team of the a.vchunks) and its own ring of stages.  Unit v of
// a team's chunk is copied by its warp v mod TS into the team's stage v mod
// (stages), once all TS warps have read the unit that stage held before (an
// empty barrier of TS arrivals).  Each warp holds whole columns, so a piece
// end needs no merge inside the CTA: a warp writes its columns (to the output,
// or to its workspace slot) and the last piece of the segment to arrive for
// those columns merges them.
// CTAs per SM of the kernel with 8 columns a warp (4 columns a warp: 3).
#ifndef PKV_MQT2_CTAS
#define PKV_MQT2_CTAS 3
#endif
__host__ __device__ constexpr int team_ctas(int nt) { return nt == 1 ? 3 : PKV_MQT2_CTAS; }
// Stages of a CTA (its teams' rings together, each a multiple of the team's
// warps: unit v + stages has v's copier): as many as the shared memory of the
// CTAs an SM holds allows.
__host__ __device__ constexpr int team_stages(int nt) { return team_ctas(nt) == 3 ? 8 : 12; }

template <int DT, int kStages>
struct MqtSmem {
  static constexpr uint32_t kAlign = 1024;
  static constexpr uint32_t kScl = kStages * Tiles<DT>::kCodes;
  static constexpr uint32_t kFull = kScl + kStages * Tiles<DT>::kScales;
  static constexpr uint32_t kEmpty = kFull + kStages * 8;
  static constexpr uint32_t kCtl = kEmpty + kStages * 8;
  static constexpr uint32_t kStall = kCtl + 16;  // the test hook's barrier (nothing completes it)
  static constexpr uint32_t kSplit = kCtl + 32;  // the work split
  static constexpr uint32_t kRows = kSplit + 16;  // row_start, lens, chunks before each row
  static size_t bytes(int rows) { return kAlign + kRows + plan_ints(rows) * 4; }
};

template <int DT, int NT, int TS>
__global__ void __launch_bounds__(kThreads, team_ctas(NT))
    paged_decode_mqt_kernel(const __grid_constant__ DecodeArgs a,
                            const __grid_constant__ TileMaps maps) {
  using TL = Tiles<DT>;
  constexpr int RS = team_stages(NT);  // stages of the CTA
  using SM = MqtSmem<DT, RS>;
  constexpr int kTeams = kWarps / TS;
  constexpr int RT = RS / kTeams;      // stages of a team
  constexpr int CW = 4 * NT;           // columns of one warp
  static_assert(RT % TS == 0, "a unit and the unit RT later have the same copier");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((SM::kAlign - (smem_addr(smem_raw) & (SM::kAlign - 1))) &
                              (SM::kAlign - 1));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int team = warp / TS, wt = warp % TS;          // team, and warp within it
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + SM::kCtl);  // [0] abort
  int* row_start = reinterpret_cast<int*>(smem + SM::kRows);
  int* lens = row_start + a.num_rows + 1;
  const uint32_t full0 = smem_addr(smem + SM::kFull) + team * RT * 8;    // the team's barriers
  const uint32_t empty0 = smem_addr(smem + SM::kEmpty) + team * RT * 8;
  uint8_t* ring = smem + static_cast<size_t>(team) * RT * TL::kCodes;    // and stages
  uint8_t* ring_sc = smem + SM::kScl + static_cast<size_t>(team) * RT * TL::kScales;
  const int G = a.n_q / a.n_kv;
  const int nc = a.nq * G;                             // columns of this pass
  const int cbase = wt * CW;                           // this warp's first column
  const int ncw = min(max(nc - cbase, 0), CW);         // and how many it has
  const int plan_window = a.window > 0 ? a.window + a.q_len - 1 : 0;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&maps.k);  // kernel parameters, not written by an earlier kernel
    prefetch_tensormap(&maps.v);
    ctl[0] = 0;
    mbar_init(smem_addr(smem + SM::kStall), 1);
    const uint32_t f = smem_addr(smem + SM::kFull), e = smem_addr(smem + SM::kEmpty);
    for (int s = 0; s < RS; ++s) {
      mbar_init(f + 8 * s, 1);
      mbar_init(e + 8 * s, TS);
    }
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, plan_window,
            blockIdx.x == 0 ? a.status : nullptr, lens, row_start, a.q_len);
  const bool stalled = test_stall(smem_addr(smem + SM::kStall), a.test_stall_ns, ctl, a.status);
  int* pc = lens + a.num_rows;
  plan_split(row_start, a.num_rows, a.n_kv, a.vchunks, a.aligned_split,
             reinterpret_cast<Split*>(smem + SM::kSplit), pc);
  // read from shared memory where used (at each piece): no registers held across the loop
  const Split* sp = reinterpret_cast<const Split*>(smem + SM::kSplit);
  const int k = blockIdx.x * kTeams + team;
  long long c_begin, c_end;
  chunk_range(*sp, k, row_start, pc, a.num_rows, a.n_kv, c_begin, c_end);

  if (blockIdx.x == 0) {  // rows without tokens (or shorter than q_len): zeros
    for (int i = 0; i < a.num_rows; ++i)
      if (row_start[i + 1] == row_start[i])
        for (int jj = 0; jj < a.nq; ++jj)
          for (int e = threadIdx.x; e < a.n_q * kD; e += kThreads)
            a.out[((static_cast<long long>(i) * a.q_len + a.q0 + jj) * a.n_q) * kD + e] = 0.f;
  }

  const int n_units = static_cast<int>(c_end - c_begin);
  // this warp copies the units v = wt + TS u (u = 0, 1, ...) of its team's chunk
  const long long first = c_begin + wt;
  const int n_mine = first < c_end ? static_cast<int>((c_end - first + TS - 1) / TS) : 0;

  auto fetch = [&](int base, int& pg, int& hh, int& row, int& pidx) {
    const int u = base + lane;
    pg = hh = row = pidx = 0;
    if (u < n_mine) {
      const long long x = first + static_cast<long long>(u) * TS;
      const int i = row_of(row_start, a.num_rows, a.n_kv, x);
      const int npg = row_start[i + 1] - row_start[i];
      const int off = static_cast<int>(x - static_cast<long long>(a.n_kv) * row_start[i]);
      hh = off / npg;
      const int p = off - hh * npg;
      int pabs = window_start(lens[i], plan_window) / kPage + p;  // block-table entry
      int page = __ldg(a.block_table + static_cast<long long>(i) * a.bt_stride + pabs);
      if (page < 0 || page >= a.num_pages) {
        record_status(a.status, PKV_DEV_BAD_PAGE);
        page = 0;
        pabs = -1;  // take no append
      }
      pg = page;
      row = i;
      pidx = pabs;
    }
  };
  int c_pg, c_h, c_row, c_p, n_pg, n_h, n_row, n_p;
  int batch = 0;
  fetch(0, c_pg, c_h, c_row, c_p);
  int issued = 0;  // units this warp has copied
  const uint64_t policy = policy_evict_first();

  auto issue = [&]() {  // this warp's next unit, v = wt + TS issued
    const int u = issued;
    if (u >= batch + 32) {
      c_pg = n_pg;
      c_h = n_h;
      c_row = n_row;
      c_p = n_p;
      batch += 32;
      fetch(batch + 32, n_pg, n_h, n_row, n_p);
    }
    const int jj = u - batch;
    const int pg = __shfl_sync(kFull, c_pg, jj);
    const int hh = __shfl_sync(kFull, c_h, jj);
    const int pabs = __shfl_sync(kFull, c_p, jj);
    if (a.k_new != nullptr && pabs >= 0) {  // first pass: new tokens of this page first
      const int row = __shfl_sync(kFull, c_row, jj);
      const int L = lens[row], first_new = L - a.q_len;
      const int lo = max(first_new, pabs * kPage), hi = min(L, pabs * kPage + kPage);
      for (int pos = lo; pos < hi; ++pos)
        append_token<DT>(a, static_cast<long long>(row) * a.q_len + (pos - first_new), hh, pg,
                         pos % kPage, lane);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const int s = (wt + TS * u) % RT;
      const uint32_t bar = full0 + 8 * s;
      const uint32_t dst = smem_addr(ring + s * TL::kCodes);
      const int z = pg * a.n_kv + hh;
      mbar_arrive_expect_tx(bar, TL::kTx);
      tma_load_tile<DT>(dst, &maps.k, z, bar, policy);
      tma_load_tile<DT>(dst + TL::kData, &maps.v, z, bar, policy);
      if constexpr (DT == PKV_KV_Q8_0) {
        const uint32_t sdst = smem_addr(ring_sc + s * TL::kScales);
        const size_t unit = static_cast<size_t>(z);
        bulk_g2s(sdst, a.k_scales + unit * TL::kScale, TL::kScale, bar, policy);
        bulk_g2s(sdst + TL::kScale, a.v_scales + unit * TL::kScale, TL::kScale, bar, policy);
      }
    }
    ++issued;
  };
  while (issued < n_mine && wt + TS * issued < RT) issue();  // at most 32 units: batch 0
  fetch(32, n_pg, n_h, n_row, n_p);  // the next batch, once the first copies are on their way

  int consumed = 0;  // units [0, consumed) have landed (this warp waited for them)
  bool aborted = stalled;
  auto fail = [&]() {
    if (!aborted && lane == 0 && !ctl[0]) {
      ctl[0] = 1;
      record_status(a.status, PKV_DEV_TIMEOUT);
    }
    aborted = true;
  };
  MqState<DT, NT> S;

  for (long long x = c_begin; x < c_end;) {
    const int i = row_of(row_start, a.num_rows, a.n_kv, x);
    const int npg = row_start[i + 1] - row_start[i];
    const long long row_base = static_cast<long long>(a.n_kv) * row_start[i];
    const int h = static_cast<int>(x - row_base) / npg;  // x - row_base < n_kv * npg < 2^31
    const long long seg_start = row_base + static_cast<long long>(h) * npg;
    const long long seg_end = seg_start + npg;
    const long long b = min(seg_end, c_end);
    const int L = lens[i];
    const int p0 = window_start(L, plan_window) / kPage;
    const long long j = static_cast<long long>(i) * a.n_kv + h;
    int k0, k1;
    segment_chunks(*sp, i, h, row_start, pc, a.num_rows, a.n_kv, k0, k1);
    const int P0 = L - a.q_len + a.q0;  // position of the pass's first query

    // the lane's score columns cbase + 4t + tig: attended positions [col_lo, col_hi)
    int col_lo[2] = {0, 0}, col_hi[2] = {0, 0};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int c = 4 * t + tig;
      if (c < ncw) {
        const int P = P0 + (cbase + c) / G;
        col_hi[t] = P + 1;
        col_lo[t] = window_start(P + 1, a.window);
      }
    }
    // slots any of the warp's columns attends, in any page
    const int pos_lo = ncw > 0 ? window_start(P0 + cbase / G + 1, a.window) : 0;
    const int pos_hi = ncw > 0 ? P0 + (cbase + ncw - 1) / G + 1 : 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int cq = 4 * t + (gid >> 1);  // the column whose query this lane loads
      const float* qv = cq < ncw
                            ? a.q + ((static_cast<long long>(i) * a.q_len + a.q0 + (cbase + cq) / G) *
                                         a.n_q + h * G + (cbase + cq) % G) * kD
                            : nullptr;
      int e2;
      mq_load_column<DT>(qv, a.qscale, (gid & 1) != 0, tig, S.qb[t], e2);
      S.qexp[t] = ldexpf(1.0f, __shfl_sync(kFull, e2, 8 * tig));
      S.m[t] = -INFINITY;
      S.l[t] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) S.o[r][e] = 0.f;
    S.vx = kNoScale;

    for (long long pos = x; pos < b; ++pos) {
      const int v = static_cast<int>(pos - c_begin);
      const int s = v % RT;
      bool ok = !aborted && mbar_wait_bounded(full0 + 8 * s, (v / RT) & 1, ctl);
      ok = __all_sync(kFull, ok);
      if (!ok) {
        fail();
        continue;
      }
      consumed = v + 1;
      if (ncw > 0) {
        const int pf = (p0 + static_cast<int>(pos - seg_start)) * kPage;  // page's first token
        const int slot_lo = max(0, pos_lo - pf), slot_hi = min(kPage, pos_hi - pf);
        mq_process_unit<DT, NT>(ring + s * TL::kCodes, ring_sc + s * TL::kScales, pf, col_lo,
                                col_hi, slot_lo, slot_hi, ncw, lane, S);
      }
      // done with the stage; its unit's copier refills it with unit v + RT
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      if (v % TS == wt && v + RT < n_units) {
        bool e_ok = mbar_wait_bounded(empty0 + 8 * s, (v / RT) & 1, ctl);
        e_ok = __all_sync(kFull, e_ok);
        if (!e_ok) {
          fail();
          continue;
        }
        issue();
      }
    }

    // ---- piece end: this warp's columns are complete for the piece
    if (!aborted && ncw > 0) {
      float l_tot[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float vsum = S.l[t];
        vsum += __shfl_xor_sync(kFull, vsum, 4);
        vsum += __shfl_xor_sync(kFull, vsum, 8);
        vsum += __shfl_xor_sync(kFull, vsum, 16);
        l_tot[t] = vsum;
      }
      // (m, l) of the lane's V-columns 2tig + e, from the score lanes
      float mv[2], lv[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int cl = 2 * tig + e;
        mv[e] = __shfl_sync(kFull, S.m[0], cl & 3);
        lv[e] = __shfl_sync(kFull, l_tot[0], cl & 3);
        if constexpr (NT == 2) {
          const float m1 = __shfl_sync(kFull, S.m[1], cl & 3);
          const float l1 = __shfl_sync(kFull, l_tot[1], cl & 3);
          if (cl >= 4) {
            mv[e] = m1;
            lv[e] = l1;
          }
        }
      }
      const float osc = mq_o_scale<DT>(S.vx);
      const bool whole = (k0 == k1);
      auto out_col = [&](int c) {
        return a.out + ((static_cast<long long>(i) * a.q_len + a.q0 + c / G) * a.n_q + h * G +
                        c % G) * kD;
      };
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int cl = 2 * tig + e;
        if (cl >= ncw) continue;
        if (whole) {
          float* o = out_col(cbase + cl);
          const float f = osc / lv[e];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            o[mq_dim<DT>(r, 0, gid)] = S.o[r][e] * f;
            o[mq_dim<DT>(r, 2, gid)] = S.o[r][e + 2] * f;
          }
        } else {
          const long long slot = (k + j) * kMqCols + cbase + cl;
          float* acc = a.part_acc + slot * kD;
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            acc[mq_dim<DT>(r, 0, gid)] = S.o[r][e] * osc;
            acc[mq_dim<DT>(r, 2, gid)] = S.o[r][e + 2] * osc;
          }
          if (gid == 0) {
            a.part_ml[slot * 2] = mv[e];
            a.part_ml[slot * 2 + 1] = lv[e];
          }
        }
      }
      if (!whole && a.flags != nullptr) {
        __syncwarp();
        int last = 0;
        // the warp's partial (ordered by __syncwarp) is released by its arrival
        if (lane == 0) last = atomic_add_acq_rel(mq_counter(a.flags, j, wt), 1) == k1 - k0;
        last = __shfl_sync(kFull, last, 0);
        if (last) {
          __syncwarp();  // lane 0's acquire, ordered for the warp
          mq_merge_segment_warp<CW, NT == 1 ? 2 : 1>(a.part_ml, a.part_acc, j, k0, k1, cbase, nc,
                                                     out_col, lane);
          if (lane == 0) *mq_counter(a.flags, j, wt) = 0;  // ready for the next call
        }
      }
    }
    x = b;
  }

  // Copies this warp issued that no wait saw land must land before the CTA exits.
  if (aborted || ctl[0]) {
    const int zero = 0;
    for (int u = 0; u < issued; ++u) {
      const int v = wt + TS * u;
      if (v >= consumed) mbar_wait_bounded(full0 + 8 * (v % RT), (v / RT) & 1, &zero);
    }
  }
}

// ------------------------------------------------------------ launchers ----
template <class K>
static cudaError_t mq_ensure_smem(K kernel, std::atomic<size_t> (&granted)[64], size_t smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && granted[dev].load(std::memory_order_relaxed) >= smem)
    return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e == cudaSuccess && dev >= 0 && dev < 64) {
    size_t cur = granted[dev].load();
    while (cur < smem && !granted[dev].compare_exchange_weak(cur, smem)) {
    }
  }
  return e;
}

// The kernel of (dtype, kind), its dynamic shared memory for `rows` rows and
// the chunks one CTA holds.
template <int DT, int KIND>
struct MqKernel {
  static constexpr int kTeams = KIND == kMqSingle ? 1 : kWarps / kind_ts(KIND);
  static auto fn() {
    if constexpr (KIND == kMqSingle)
      return paged_decode_mq_kernel<DT>;
    else
      return paged_decode_mqt_kernel<DT, kind_nt(KIND), kind_ts(KIND)>;
  }
  static size_t smem(int rows) {
    return KIND == kMqSingle ? MqSmem<DT>::bytes(rows)
                             : MqtSmem<DT, team_stages(kind_nt(KIND))>::bytes(rows);
  }
  static cudaError_t prepare(size_t smem) {
    static std::atomic<size_t> granted[64];
    return mq_ensure_smem(fn(), granted, smem);
  }
};

template <int DT, int KIND>
static cudaError_t launch_mq_t(const DecodeArgs& a, const TileMaps& maps, int chunks,
                               cudaStream_t st) {
  using K = MqKernel<DT, KIND>;
  const size_t smem = K::smem(a.num_rows);
  cudaError_t e = K::prepare(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((chunks + K::kTeams - 1) / K::kTeams);  // a CTA holds kTeams chunks
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = PKV_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, K::fn(), a, maps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Chunks per SM: resident CTAs times the chunks a CTA holds.
template <int DT, int KIND>
static cudaError_t mq_occupancy_t(int rows, int* blocks) {
  using K = MqKernel<DT, KIND>;
  const size_t smem = K::smem(rows);
  cudaError_t e = K::prepare(smem);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, K::fn(), kThreads, smem);
  *blocks *= K::kTeams;
  return e;
}

template <int DT>
static cudaError_t launch_mq_dt(int kind, const DecodeArgs& a, const TileMaps& maps, int chunks,
                                cudaStream_t st) {
  if constexpr (DT == PKV_KV_F32) {
    return launch_mq_t<DT, kMqSingle>(a, maps, chunks, st);
  } else if constexpr (DT == PKV_KV_Q8_0) {
    if (kind == kMqSingle) return launch_mq_t<DT, kMqSingle>(a, maps, chunks, st);
    if (kind == kMqPair2) return launch_mq_t<DT, kMqPair2>(a, maps, chunks, st);
    return launch_mq_t<DT, kMqTeam2>(a, maps, chunks, st);
  } else if constexpr (DT == PKV_KV_BF16) {  // (the tensor-core kernel: launch_paged_decode_mq)
    if (kind == kMqSingle) return launch_mq_t<DT, kMqSingle>(a, maps, chunks, st);
    if (kind == kMqPair1) return launch_mq_t<DT, kMqPair1>(a, maps, chunks, st);
    return launch_mq_t<DT, kMqTeam1>(a, maps, chunks, st);
  } else {  // f16 (the tensor-core kernel is launched by launch_paged_decode_mq)
    if (kind == kMqSingle) return launch_mq_t<DT, kMqSingle>(a, maps, chunks, st);
    if (kind == kMqTeam1) return launch_mq_t<DT, kMqTeam1>(a, maps, chunks, st);
    return launch_mq_t<DT, kMqTeam2>(a, maps, chunks, st);
  }
}

template <int DT>
static cudaError_t occupancy_mq_dt(int kind, int rows, int* blocks) {
  if constexpr (DT == PKV_KV_F32) {
    return mq_occupancy_t<DT, kMqSingle>(rows, blocks);
  } else if constexpr (DT == PKV_KV_Q8_0) {
    if (kind == kMqSingle) return mq_occupancy_t<DT, kMqSingle>(rows, blocks);
    if (kind == kMqPair2) return mq_occupancy_t<DT, kMqPair2>(rows, blocks);
    return mq_occupancy_t<DT, kMqTeam2>(rows, blocks);
  } else if constexpr (DT == PKV_KV_BF16) {
    if (kind == kMqSingle) return mq_occupancy_t<DT, kMqSingle>(rows, blocks);
    if (kind == kMqPair1) return mq_occupancy_t<DT, kMqPair1>(rows, blocks);
    return mq_occupancy_t<DT, kMqTeam1>(rows, blocks);
  } else {  // f16
    if (kind == kMqSingle) return mq_occupancy_t<DT, kMqSingle>(rows, blocks);
    if (kind == kMqTeam1) return mq_occupancy_t<DT, kMqTeam1>(rows, blocks);
    return mq_occupancy_t<DT, kMqTeam2>(rows, blocks);
  }
}

cudaError_t launch_paged_decode_mq(int dtype, int group, const DecodeArgs& a, const TileMaps& maps,
                                   int chunks, cudaStream_t st) {
  if (group != 1 && group != 2 && group != 4) return cudaErrorInvalidValue;
  const int kind = mq_kind_rows(dtype, group, a.q_len, a.num_rows);
  if (kind == kMqTc) return launch_paged_decode_mqtc(dtype, a, maps, chunks, st);
  if (dtype == PKV_KV_F16) return launch_mq_dt<PKV_KV_F16>(kind, a, maps, chunks, st);
  if (dtype == PKV_KV_BF16) return launch_mq_dt<PKV_KV_BF16>(kind, a, maps, chunks, st);
  if (dtype == PKV_KV_F32) return launch_mq_dt<PKV_KV_F32>(kind, a, maps, chunks, st);
  return launch_mq_dt<PKV_KV_Q8_0>(kind, a, maps, chunks, st);
}

cudaError_t paged_decode_mq_blocks_per_sm(int dtype, int group, int q_len, int rows,
                                          int* blocks) {
  const int kind = mq_kind_rows(dtype, group, q_len, rows);
  if (kind == kMqTc) return paged_decode_mqtc_blocks_per_sm(dtype, rows, blocks);
  if (dtype == PKV_KV_F16) return occupancy_mq_dt<PKV_KV_F16>(kind, rows, blocks);
  if (dtype == PKV_KV_BF16) return occupancy_mq_dt<PKV_KV_BF16>(kind, rows, blocks);
  if (dtype == PKV_KV_F32) return occupancy_mq_dt<PKV_KV_F32>(kind, rows, blocks);
  return occupancy_mq_dt<PKV_KV_Q8_0>(kind, rows, blocks);
}

}  // namespace pkv

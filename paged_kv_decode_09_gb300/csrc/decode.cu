// decode.cu — split-KV paged decode attention, the merge of its partial
// states, and the plan kernel.
//
// The operation (tinyllm, "The repository currently provides": GQA attention,
// per-sequence block tables into a physical KV page pool; "Known limitations":
// 16-token pages, and a paged-reference decode that gathers pages before a
// dense attention): for each row i and query head g of KV head h = g / G,
//     out[i][g] = softmax_t(scale <q[i][g], K[i][h][t]>) V[i][h][t],  t < L_i.
// Here the pages are read in place.
//
// Work split.  The batch is a list of T = n_kv * sum_i ceil(L_i/16) units,
// one per (row, KV head, page) in that order, cut into contiguous chunks of
// nearly equal size, one per CTA (plan_split): uniform for q8_0 and f32 KV
// (CTA k < min(grid, T) takes [floor(kT/C), floor((k+1)T/C))), aligned to the
// (row, KV head) segments for f16 and bf16 (a split segment ends where a
// chunk ends); CTAs beyond the chunks idle.  Every CTA thus streams about the
// same number of 4 KiB (f16) or 2176-byte (q8_0) tiles whatever the length
// mix: one 40k-token row and many 16-token rows keep all SMs busy.  The units of one
// (row, head) that fall in one CTA form a "piece"; a piece that is the whole
// segment writes the output, otherwise it writes a partial state to slot
// k + (i * n_kv + h) (pieces in unit order increase k, j or both, so the slot
// is unique).  A segment spanning chunks k0..k1 has k1 - k0 + 1 pieces.  In
// the merging mode each piece then bumps the segment's arrival counter, and
// the last to arrive merges all pieces into the output and resets the
// counter; otherwise the combine kernel merges them in a second launch.
//
// Fused append: when new K/V are given, the warp that reads a row's last page
// first stores the row's new token into it (the same encoding as kv_append),
// so attention sees it without a separate launch.
//
// Inside a CTA: four warps, each feeding itself.  Warp w takes units w, w+4,
// ... of the chunk and keeps its own ring of shared-memory stages: it issues
// the tensor copies of its next units (K tile, then V tile, of one (page, KV
// head), through tensor maps that apply the 128-byte swizzle, so that the
// matrix loads below are free of bank conflicts), waits on the stage's
// mbarrier, computes, and re-issues into the stage it just read.  Each stage
// has one owner, so no empty barriers are needed and four threads per CTA
// keep copies in flight.  At the end of a piece the warps leave their states
// in a shared merge buffer; the last to arrive combines them and does the
// global writes, while the others carry on streaming.
//
// One page on the tensor cores (warp-wide mma.sync, fp32 accumulation).  The
// stored K and V values are exact in f16 (f16 KV, and the q8_0 codes, which
// are integers of at most 8 bits); the fp32 operands, q (times scale*log2 e,
// normalised per head by a power of two) and the probabilities, are each
// split into an f16 high part and the f16 rounding of the remainder, the two
// parts sitting in adjacent MMA columns, so a product keeps about 22
// significant bits.  Columns n = 2g + part, g < G (up to 8 for G = 4).
//   scores:  S[16 tokens][8 cols] = K[16 tokens][128 dims] Q^T, 8 k-steps of
//     16 dims (q8_0: one 32-dim block = 2 k-steps into a fresh accumulator,
//     then times the token's block scale).  Lane 4 gid + tig ends with head
//     tig's scores of tokens gid and gid + 8 (hi + lo columns).
//   softmax: base 2 over the page, shared by the 8 lanes of a head; the
//     running maximum is raised (and the state rescaled) only when a page
//     exceeds it by more than 8, so probabilities stay below 2^8.
//   values:  O^T[128 dims][8 cols] += V^T[128 dims][16 tokens] P^T, P^T
//     built by 4 shuffles (q8_0: times the V block scales, one B operand per
//     block).  Lane 4 gid + tig accumulates head tig's output at 16 of the
//     dims, hi and lo columns, summed at the end of the piece.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// f32 KV keeps each warp's scaled queries in shared memory, one head every
// kQStride floats (the 16-byte pad puts the heads' chunks in different banks).
constexpr int kQStride = kD + 4;

// Offsets from a 1024-byte aligned base.  The tiles come first (the swizzle
// atom is 1024 bytes), then scales, barriers, the merge buffer, (f32 KV) the
// queries, control words and the plan.
template <int DT, int G>
struct Smem {
  static constexpr int kStages = kWarps * Tiles<DT>::kRing;
  static constexpr uint32_t kAlign = 1024;
  static constexpr uint32_t kScl = kStages * Tiles<DT>::kCodes;           // [warp][ring][K, V]
  static constexpr uint32_t kBar = kScl + kStages * Tiles<DT>::kScales;   // full[warp][ring]
  static constexpr uint32_t kMrgAcc = kBar + ((kStages * 8 + 15) / 16) * 16;  // f32 [warps][G][D]
  static constexpr uint32_t kMrgMl = kMrgAcc + kWarps * G * kD * 4;        // f32 [warps][G][2]
  static constexpr uint32_t kQ = kMrgMl + kWarps * G * 2 * 4;  // f32 KV: [warps][G][kQStride] q
  static constexpr uint32_t kCtl =
      kQ + (DT == PKV_KV_F32 ? kWarps * G * kQStride * 4 : 0);             // int [4]
  static constexpr uint32_t kStall = kCtl + 16;  // the test hook's barrier (nothing completes it)
  static constexpr uint32_t kSplit = kCtl + 32;  // the work split
  static constexpr uint32_t kRows = kSplit + 16;  // int row_start[rows + 1], lens[rows], pc[rows + 1]
  static size_t bytes(int rows) {
    return kAlign + kRows + plan_ints(rows) * 4;  // kAlign: base alignment slack
  }
  static_assert(Tiles<DT>::kCodes % 1024 == 0, "tile stages keep the swizzle atom alignment");
  static_assert(kMrgAcc % 16 == 0 && kMrgMl % 16 == 0 && kQ % 16 == 0 && kCtl % 16 == 0,
                "vector accesses need 16-byte aligned regions");
};

// The same parts where `lo` differs between the lanes of a warp (the column
// a lane holds), without a branch: every lane rounds x - m f, with m = 1 for
// the remainder and m = 0 for the high part (0 f + x is x, f being finite:
// the callers keep |x| inside the f16 range, or the tf32 one).  The values
// of split_f16x2 and tf32_part, but for the sign of a zero high part.
__device__ __forceinline__ uint32_t split_f16x2_lane(float x0, float x1, bool lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 f = __half22float2(h);
  const float m = lo ? -1.0f : 0.0f;
  const float2 r = __ffma2_rn(make_float2(m, m), f, make_float2(x0, x1));
  const __half2 p = __floats2half2_rn(r.x, r.y);
  return *reinterpret_cast<const uint32_t*>(&p);
}
__device__ __forceinline__ uint32_t tf32_part_lane(float x, bool lo) {
  return to_tf32(fmaf(lo ? -1.0f : 0.0f, __uint_as_float(to_tf32(x)), x));
}

// Per-warp online softmax state for one piece.
template <int DT>
struct WarpState {
  // score k-steps (tf32: 8 dims; f32 KV: none, the products run on CUDA cores)
  static constexpr int kSteps = DT == PKV_KV_BF16 ? 16 : DT == PKV_KV_F32 ? 1 : 8;
  uint32_t qb[kSteps][2];  // B operand of the scores per k-step: column gid (head gid/2, part gid%2)
  float qexp;         // 2^e of head tig: undoes its power-of-two normalisation
  float m;            // running max (base 2) of head tig, equal on its 8 lanes
  float l;            // this lane's share of head tig's sum of probabilities
  float o[8][4];      // O^T accumulators: dims (see dim_of) x columns (tig, hi), (tig, lo)
  int vx;             // q8_0: every V block scale of the piece so far is below 2^vx
  float* qs;          // f32 KV: the warp's scaled queries [G][kQStride] in shared memory
};

template <int DT>
__device__ __forceinline__ float o_scale(const WarpState<DT>& S) {
  if constexpr (DT == PKV_KV_F16)
    return 1.0f / (1 << kPShift);
  else if constexpr (DT == PKV_KV_BF16 || DT == PKV_KV_F32)
    return 1.0f;  // tf32 parts have the fp32 exponent range; f32 products are plain fp32
  else
    return pow2i(S.vx - kPShift);
}

// The dim of accumulator o[r][e] (e = 0, 2; e + 1 is its lo column) in lane
// 4 gid + tig.
template <int DT>
__device__ __forceinline__ int dim_of(int r, int e, int gid) {
  if constexpr (DT == PKV_KV_F32)  // dims 32j + 4gid + {0,1,2,3}: o[2j][0, 2], o[2j+1][0, 2]
    return 32 * (r >> 1) + 4 * gid + 2 * (r & 1) + (e ? 1 : 0);
  else if constexpr (DT != PKV_KV_Q8_0)
    return 16 * r + gid + (e ? 8 : 0);
  else
    return 16 * r + 2 * gid + (e ? 1 : 0);
}

// Load head (gid/2)'s query for a piece into the lane's B fragments: the
// dims of k-step ks are 16ks + 2tig + {0,1} and 16ks + 2tig + 8 + {0,1}
// (f16) or 16ks + 4tig + {0,1} and {2,3} (q8_0, matching how the codes are
// placed in the A fragments).  Each head is scaled by 2^-e so that its
// largest |q| lies in [2^13, 2^14) and both f16 parts stay normal.
template <int DT, int G>
__device__ __forceinline__ void load_query(const float* qrow, float qscale, int lane,
                                           WarpState<DT>& S) {
  const int gid = lane >> 2, tig = lane & 3, g2 = gid >> 1;
  const bool lo = (gid & 1) != 0;
  if constexpr (DT == PKV_KV_F32) {
    // the G heads' q times scale * log2 e into the warp's buffer: lane l
    // writes dims 4l .. 4l + 3 of every head
    __syncwarp();  // the previous piece's reads are done
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(qrow + g * kD) + lane);
      *reinterpret_cast<float4*>(S.qs + g * kQStride + 4 * lane) =
          make_float4(x.x * qscale, x.y * qscale, x.z * qscale, x.w * qscale);
    }
    __syncwarp();
    S.qexp = 1.0f;
  } else if constexpr (DT == PKV_KV_BF16) {
    // tf32 k-steps of 8 dims: k = tig <- dim 8ks + 2tig, k = tig + 4 <- dim 8ks + 2tig + 1
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      float2 x = make_float2(0.f, 0.f);
      if (g2 < G) x = __ldg(reinterpret_cast<const float2*>(qrow + g2 * kD + 8 * ks + 2 * tig));
      S.qb[ks][0] = tf32_part_lane(x.x * qscale, lo);
      S.qb[ks][1] = tf32_part_lane(x.y * qscale, lo);
    }
    S.qexp = 1.0f;
  } else {
    float v[32];
  #pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      if (g2 < G) {
        const float* qh = qrow + g2 * kD;
        if constexpr (DT == PKV_KV_F16) {
          const float2 x = __ldg(reinterpret_cast<const float2*>(qh + 16 * ks + 2 * tig));
          const float2 y = __ldg(reinterpret_cast<const float2*>(qh + 16 * ks + 8 + 2 * tig));
          v[4 * ks] = x.x;
          v[4 * ks + 1] = x.y;
          v[4 * ks + 2] = y.x;
          v[4 * ks + 3] = y.y;
        } else {
          const float4 x = __ldg(reinterpret_cast<const float4*>(qh + 16 * ks + 4 * tig));
          v[4 * ks] = x.x;
          v[4 * ks + 1] = x.y;
          v[4 * ks + 2] = x.z;
          v[4 * ks + 3] = x.w;
        }
      } else {
  #pragma unroll
        for (int e = 0; e < 4; ++e) v[4 * ks + e] = 0.f;
      }
    }
    float amax = 0.f;
  #pragma unroll
    for (int e = 0; e < 32; ++e) {
      v[e] *= qscale;
      amax = fmaxf(amax, fabsf(v[e]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    int e2 = 0;
    if (amax > 0.f && amax <= 3.0e38f) {
      int ex;
      frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
      e2 = ex - 14;
    }
  #pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      S.qb[ks][0] = split_f16x2_lane(ldexpf(v[4 * ks], -e2), ldexpf(v[4 * ks + 1], -e2), lo);
      S.qb[ks][1] = split_f16x2_lane(ldexpf(v[4 * ks + 2], -e2), ldexpf(v[4 * ks + 3], -e2), lo);
    }
    // lane 8 tig holds head tig (gid = 2 tig)
    S.qexp = ldexpf(1.0f, __shfl_sync(kFull, e2, 8 * tig));
  }
}

// Process one staged (page, KV head) unit whose attended tokens are slots
// [tlo, nvalid) (0 <= tlo < nvalid <= 16; tlo > 0 only on the first page of
// a sliding window): tiles at shared address `st` (K, then V at + kData),
// q8_0 scales at `sc` (K, then V at + kScale).  The other rows hold whatever
// the pool holds there (possibly NaN): they are masked out of the scores, and
// f16 V rows are zeroed before the values MMA.
template <int DT, int G>
__device__ __forceinline__ void process_unit(uint8_t* st, const uint8_t* sc, int tlo, int nvalid,
                                             int lane, WarpState<DT>& S) {
  using TL = Tiles<DT>;
  const int gid = lane >> 2, tig = lane & 3;
  // ldmatrix row addresses: lane 8j + r gives row r of matrix j = token
  // r + 8 (j & 1), chunk 2c + (j >> 1) at k-step (or dim block) c.
  const int ld_tok = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int ld_chunk = lane >> 4;
  const uint32_t kt = smem_addr(st), vt = kt + TL::kData;

  // ---- scores
  float s0, s1;
  if constexpr (DT == PKV_KV_F32) {
    // CUDA cores, fp32: lane 4 gid + tig takes head tig (head 0 stands in for
    // heads >= G, whose results are never used) and tokens gid, gid + 8;
    // four partial sums per token shorten the FMA chains
    const float* qh = S.qs + (tig < G ? tig : 0) * kQStride;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll 8
    for (int c = 0; c < 32; ++c) {  // 16-byte chunks of the 128 dims
      const float4 qv = *reinterpret_cast<const float4*>(qh + 4 * c);
      const float4 k0 = *reinterpret_cast<const float4*>(st + tile_offset<DT>(gid, c));
      const float4 k1 = *reinterpret_cast<const float4*>(st + tile_offset<DT>(gid + 8, c));
      a0 = make_float4(fmaf(qv.x, k0.x, a0.x), fmaf(qv.y, k0.y, a0.y), fmaf(qv.z, k0.z, a0.z),
                       fmaf(qv.w, k0.w, a0.w));
      a1 = make_float4(fmaf(qv.x, k1.x, a1.x), fmaf(qv.y, k1.y, a1.y), fmaf(qv.z, k1.z, a1.z),
                       fmaf(qv.w, k1.w, a1.w));
    }
    s0 = (a0.x + a0.y) + (a0.z + a0.w);
    s1 = (a1.x + a1.y) + (a1.z + a1.w);
  } else if constexpr (DT == PKV_KV_BF16) {
    // bf16 pairs of an ldmatrix row widen to tf32 exactly: the low value is
    // the word shifted up, the high one the word with its low half cleared
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c2 = 0; c2 < 8; ++c2) {
      uint32_t w0, w1, w2, w3;  // tokens gid, gid+8 of chunk 2c2; the same of chunk 2c2+1
      ldsm_x4(kt + tile_offset<DT>(ld_tok, 2 * c2 + ld_chunk), w0, w1, w2, w3);
      mma_1688_tf32(c, w0 << 16, w1 << 16, w0 & 0xffff0000u, w1 & 0xffff0000u,
                    S.qb[2 * c2][0], S.qb[2 * c2][1]);
      mma_1688_tf32(c, w2 << 16, w3 << 16, w2 & 0xffff0000u, w3 & 0xffff0000u,
                    S.qb[2 * c2 + 1][0], S.qb[2 * c2 + 1][1]);
    }
    s0 = c[0] + c[1];
    s1 = c[2] + c[3];
  } else if constexpr (DT == PKV_KV_F16) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kt + tile_offset<DT>(ld_tok, 2 * ks + ld_chunk), a0, a1, a2, a3);
      mma_16816(c, a0, a1, a2, a3, S.qb[ks][0], S.qb[ks][1]);
    }
    s0 = c[0] + c[1];
    s1 = c[2] + c[3];
  } else {
    // K block scales of tokens gid and gid + 8 (four f16 each)
    const uint2 k0 = *reinterpret_cast<const uint2*>(sc + gid * 8);
    const uint2 k1 = *reinterpret_cast<const uint2*>(sc + (gid + 8) * 8);
    s0 = 0.f;
    s1 = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t w0, w1, w2, w3;  // tokens gid, gid+8 of chunk 2b; the same of chunk 2b+1
      ldsm_x4(kt + tile_offset<DT>(ld_tok, 2 * b + ld_chunk), w0, w1, w2, w3);
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(c, codes_to_f16x2<kSelB01>(w0), codes_to_f16x2<kSelB01>(w1),
                codes_to_f16x2<kSelB23>(w0), codes_to_f16x2<kSelB23>(w1), S.qb[2 * b][0],
                S.qb[2 * b][1]);
      mma_16816(c, codes_to_f16x2<kSelB01>(w2), codes_to_f16x2<kSelB01>(w3),
                codes_to_f16x2<kSelB23>(w2), codes_to_f16x2<kSelB23>(w3), S.qb[2 * b + 1][0],
                S.qb[2 * b + 1][1]);
      // (token gid, token gid + 8) scales of block b, as a pair
      const uint32_t kp = __byte_perm(b < 2 ? k0.x : k0.y, b < 2 ? k1.x : k1.y,
                                      (b & 1) ? 0x7632 : 0x5410);
      const float2 ksc = __half22float2(*reinterpret_cast<const __half2*>(&kp));
      s0 = fmaf(ksc.x, c[0] + c[1], s0);
      s1 = fmaf(ksc.y, c[2] + c[3], s1);
    }
  }
  s0 = gid >= tlo && gid < nvalid ? s0 * S.qexp : -INFINITY;
  s1 = gid + 8 >= tlo && gid + 8 < nvalid ? s1 * S.qexp : -INFINITY;

  // ---- online softmax of head tig over the page (its 8 lanes: xor 4, 8, 16)
  float mx = fmaxf(s0, s1);
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
  const bool grow = mx > S.m + 8.0f;  // true on the first page (m = -inf)
  if (__any_sync(kFull, grow)) {
    const float m_new = grow ? mx : S.m;
    const float al = ex2_ftz(S.m - m_new);  // 1 if unchanged, 0 from -inf
    S.l *= al;
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) S.o[r][e] *= al;
    S.m = m_new;
  }
  const float p0 = ex2_ftz(s0 - S.m), p1 = ex2_ftz(s1 - S.m);
  S.l += p0 + p1;

  if constexpr (DT == PKV_KV_F32) {
    // O += p_t V_t on CUDA cores: lane 4 gid + tig keeps head tig's output at
    // dims 32 j + 4 gid + {0..3}; p_t of head tig comes from lane
    // 4 (t mod 8) + tig.  Unattended slots are skipped (their V may be NaN).
    const uint8_t* vs = st + TL::kData;
    auto accumulate = [&](int t) {
      const float pt = __shfl_sync(kFull, t < 8 ? p0 : p1, 4 * (t & 7) + tig);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(vs + tile_offset<DT>(t, 8 * j + gid));
        S.o[2 * j][0] = fmaf(pt, v.x, S.o[2 * j][0]);
        S.o[2 * j][2] = fmaf(pt, v.y, S.o[2 * j][2]);
        S.o[2 * j + 1][0] = fmaf(pt, v.z, S.o[2 * j + 1][0]);
        S.o[2 * j + 1][2] = fmaf(pt, v.w, S.o[2 * j + 1][2]);
      }
    };
    if (tlo == 0 && nvalid == kPage) {
#pragma unroll
      for (int t = 0; t < kPage; ++t) accumulate(t);
    } else {
      for (int t = tlo; t < nvalid; ++t) accumulate(t);
    }
    __syncwarp();
    return;
  }

  // ---- P^T operand: column gid (head gid/2, part gid%2) at tokens 2tig,
  // 2tig+1 (b0) and 2tig+8, 2tig+9 (b1); lane 8 tig + g holds head g's
  // tokens 2tig and 2tig + 8, lane 8 tig + 4 + g tokens 2tig+1 and 2tig+9.
  const int g2 = gid >> 1;
  const bool lo = (gid & 1) != 0;
  const int src = 8 * tig + (g2 & 3);
  float pa = __shfl_sync(kFull, p0, src), pb = __shfl_sync(kFull, p0, src + 4);
  float pc = __shfl_sync(kFull, p1, src), pd = __shfl_sync(kFull, p1, src + 4);
  if (g2 >= G) pa = pb = pc = pd = 0.f;
  const int t0 = 2 * tig;

  // ---- values
  if constexpr (DT == PKV_KV_F16 || DT == PKV_KV_BF16) {
    if (tlo > 0 || nvalid < kPage) {  // zero the V rows of unattended slots (NaN * 0 is NaN)
      const int n_out = kPage - (nvalid - tlo);
      for (int x = lane; x < n_out * 16; x += 32) {
        const int r = x >> 4, t = r < tlo ? r : nvalid + (r - tlo), c = x & 15;
        *reinterpret_cast<uint4*>(st + TL::kData + (c >> 3) * 2048 + t * 128 + (c & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    if constexpr (DT == PKV_KV_F16) {
      constexpr float kUp = static_cast<float>(1 << kPShift);
      const uint32_t b0 = split_f16x2_lane(pa * kUp, pb * kUp, lo);
      const uint32_t b1 = split_f16x2_lane(pc * kUp, pd * kUp, lo);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t w0, w1, w2, w3;  // (tokens 0-7 | 8-15) x (chunk 2mt | 2mt+1), transposed
        ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * mt + ld_chunk), w0, w1, w2, w3);
        mma_16816(S.o[mt], w0, w2, w1, w3, b0, b1);
      }
    } else {
      // tf32 k-steps of 8 tokens: k = tig <- token 2tig, k = tig + 4 <- token 2tig + 1
      const uint32_t b_t0 = tf32_part_lane(pa, lo), b_t1 = tf32_part_lane(pb, lo);
      const uint32_t b_t8 = tf32_part_lane(pc, lo), b_t9 = tf32_part_lane(pd, lo);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t w0, w1, w2, w3;  // dims (16mt + gid | + 8) x tokens (2tig, 2tig+1 | + 8)
        ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * mt + ld_chunk), w0, w1, w2, w3);
        mma_1688_tf32(S.o[mt], w0 << 16, w2 << 16, w0 & 0xffff0000u, w2 & 0xffff0000u, b_t0, b_t1);
        mma_1688_tf32(S.o[mt], w1 << 16, w3 << 16, w1 & 0xffff0000u, w3 & 0xffff0000u, b_t8, b_t9);
      }
    }
  } else {
    // V block scales of tokens 2tig, 2tig+1 (va) and 2tig+8, 2tig+9 (vb): the
    // four f16 block scales of a token are 8 contiguous bytes
    uint4 va = *reinterpret_cast<const uint4*>(sc + TL::kScale + t0 * 8);
    uint4 vb = *reinterpret_cast<const uint4*>(sc + TL::kScale + (t0 + 8) * 8);
    if (tlo > 0 || nvalid < kPage) {  // masked tokens have p = 0 but their scales may be NaN
      if (t0 < tlo || t0 >= nvalid) va.x = va.y = 0u;
      if (t0 + 1 < tlo || t0 + 1 >= nvalid) va.z = va.w = 0u;
      if (t0 + 8 < tlo || t0 + 8 >= nvalid) vb.x = vb.y = 0u;
      if (t0 + 9 < tlo || t0 + 9 >= nvalid) vb.z = vb.w = 0u;
    }
    // the page's largest |scale| (non-negative f16 bit patterns order as integers)
    uint32_t mb = abs_max_f16x2(abs_max_f16x2(va.x, va.y), abs_max_f16x2(va.z, va.w));
    mb = abs_max_f16x2(mb, abs_max_f16x2(abs_max_f16x2(vb.x, vb.y), abs_max_f16x2(vb.z, vb.w)));
    mb &= 0x7fff7fffu;
    uint32_t m16 = max(mb & 0xffffu, mb >> 16);
    m16 = max(m16, __shfl_xor_sync(kFull, m16, 1));  // the page's 16 tokens: over tig
    m16 = max(m16, __shfl_xor_sync(kFull, m16, 2));
    // an f16 with biased exponent e is below 2^(e - 14) (subnormals: 2^-14)
    const int vx = static_cast<int>(m16 >> 10) - 14;
    if (vx > S.vx) {  // warp-uniform: raise the bound, rescale the accumulators
      const float r = pow2i(max(S.vx - vx, -126));
#pragma unroll
      for (int rr = 0; rr < 8; ++rr)
#pragma unroll
        for (int e = 0; e < 4; ++e) S.o[rr][e] *= r;
      S.vx = vx;
    }
    const float up = pow2i(kPShift - S.vx);  // 2^(7 - vx)
    const float2 pab = make_float2(pa * up, pb * up), pcd = make_float2(pc * up, pd * up);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      // (token t0, t0 + 1) and (t0 + 8, t0 + 9) scale pairs of block b
      const uint32_t sel = (b & 1) ? 0x7632 : 0x5410;
      const uint32_t sa = __byte_perm(b < 2 ? va.x : va.y, b < 2 ? va.z : va.w, sel);
      const uint32_t sb = __byte_perm(b < 2 ? vb.x : vb.y, b < 2 ? vb.z : vb.w, sel);
      const float2 x01 = __fmul2_rn(pab, __half22float2(*reinterpret_cast<const __half2*>(&sa)));
      const float2 x23 = __fmul2_rn(pcd, __half22float2(*reinterpret_cast<const __half2*>(&sb)));
      const float x0 = x01.x, x1 = x01.y, x2 = x23.x, x3 = x23.y;
      const uint32_t b0 = split_f16x2_lane(x0, x1, lo), b1 = split_f16x2_lane(x2, x3, lo);
      uint32_t w0, w1, w2, w3;  // (tokens 0-7 | 8-15) x (chunk 2b | 2b+1), 16-bit transposed
      ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * b + ld_chunk), w0, w1, w2, w3);
      // row gid <- dim 2gid of the chunk (bytes 0, 2), row gid + 8 <- dim 2gid+1 (bytes 1, 3)
      mma_16816(S.o[2 * b], codes_to_f16x2<kSelB02>(w0), codes_to_f16x2<kSelB13>(w0),
                codes_to_f16x2<kSelB02>(w1), codes_to_f16x2<kSelB13>(w1), b0, b1);
      mma_16816(S.o[2 * b + 1], codes_to_f16x2<kSelB02>(w2), codes_to_f16x2<kSelB13>(w2),
                codes_to_f16x2<kSelB02>(w3), codes_to_f16x2<kSelB13>(w3), b0, b1);
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------ piece merge ----
// The warp that arrives last at the end of a piece combines the four warps'
// states from shared memory: lane l owns dims 4l..4l+3 of every head.  A
// whole segment is written to the output; otherwise the piece's partial
// state goes to its workspace slot.
template <int G>
__device__ __forceinline__ void piece_merge(const float* mrg_acc, const float* mrg_ml, bool whole,
                                            float* out_seg, float* part_ml, float* part_acc,
                                            long long slot, int lane) {
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mrg_ml[(w * G + g) * 2]);
    float Ls = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = exp2f(mrg_ml[(w * G + g) * 2] - M);
      Ls = fmaf(f, mrg_ml[(w * G + g) * 2 + 1], Ls);
      const float4 x = *reinterpret_cast<const float4*>(mrg_acc + (w * G + g) * kD + lane * 4);
      A.x = fmaf(f, x.x, A.x);
      A.y = fmaf(f, x.y, A.y);
      A.z = fmaf(f, x.z, A.z);
      A.w = fmaf(f, x.w, A.w);
    }
    if (whole) {
      *reinterpret_cast<float4*>(out_seg + g * kD + lane * 4) =
          make_float4(A.x / Ls, A.y / Ls, A.z / Ls, A.w / Ls);
    } else {
      *reinterpret_cast<float4*>(part_acc + (slot * G + g) * kD + lane * 4) = A;
      if (lane == 0) {
        part_ml[(slot * G + g) * 2] = M;
        part_ml[(slot * G + g) * 2 + 1] = Ls;
      }
    }
  }
}

// --------------------------------------------------------------- kernel ----
template <int DT, int G>
__global__ void __launch_bounds__(kThreads, DT == PKV_KV_Q8_0   ? PKV_Q8_CTAS_PER_SM
                                            : DT == PKV_KV_F32 ? PKV_F32_CTAS_PER_SM
                                                               : PKV_F16_CTAS_PER_SM)
    paged_decode_kernel(const __grid_constant__ DecodeArgs a,
                        const __grid_constant__ TileMaps maps) {
  using TL = Tiles<DT>;
  using SM = Smem<DT, G>;
  constexpr int R = TL::kRing;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled tiles need a 1024-byte aligned base (the launch adds the slack)
  uint8_t* smem = smem_raw + ((SM::kAlign - (smem_addr(smem_raw) & (SM::kAlign - 1))) &
                              (SM::kAlign - 1));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // [0] abort  [1] warps arrived at the current piece end  [2] merge-buffer generation
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + SM::kCtl);
  int* row_start = reinterpret_cast<int*>(smem + SM::kRows);
  int* lens = row_start + a.num_rows + 1;
  int* pc = lens + a.num_rows;  // chunks before each row (aligned split)
  Split* split = reinterpret_cast<Split*>(smem + SM::kSplit);
  const uint32_t bar0 = smem_addr(smem + SM::kBar) + warp * R * 8;  // this warp's barriers
  uint8_t* ring = smem + static_cast<size_t>(warp) * R * TL::kCodes;  // this warp's tiles
  uint8_t* ring_sc = smem + SM::kScl + static_cast<size_t>(warp) * R * TL::kScales;  // q8_0 scales

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
  // Under programmatic dependent launch this grid may start while the
  // previous kernel of the stream still runs: nothing in global memory is
  // touched before that kernel has completed and its writes are visible.
  // The next kernel of the stream may then be scheduled at once (its blocks
  // find room as ours exit).
  grid_dependency_wait();
  grid_launch_dependents();
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, a.window, blockIdx.x == 0 ? a.status : nullptr,
            lens, row_start);

  const bool stalled = test_stall(smem_addr(smem + SM::kStall), a.test_stall_ns, ctl, a.status);
  plan_split(row_start, a.num_rows, a.n_kv, gridDim.x, a.aligned_split, split, pc);
  const Split sp = *split;
  const int k = blockIdx.x;
  long long c_begin, c_end;
  chunk_range(sp, k, row_start, pc, a.num_rows, a.n_kv, c_begin, c_end);

  // Rows without tokens attend to nothing: their output is zero.
  if (k == 0) {
    for (int i = 0; i < a.num_rows; ++i)
      if (row_start[i + 1] == row_start[i])
        for (int e = threadIdx.x; e < a.n_q * kD; e += kThreads)
          a.out[static_cast<long long>(i) * a.n_q * kD + e] = 0.f;
  }

  // This warp's units: chunk positions first + 4u, u < n_units.
  const long long first = c_begin + warp;
  const int n_units = first < c_end ? static_cast<int>((c_end - first + kWarps - 1) / kWarps) : 0;

  // Unit descriptors, 32 at a time (lane j: unit base + j): page, KV head,
  // row, and whether it is the row's last page (bad pages read page 0 and
  // take no append).  Two batches are kept: the current one and the next.
  auto fetch = [&](int base, int& pg, int& hh, int& row, int& last) {
    const int u = base + lane;
    pg = 0;
    hh = 0;
    row = 0;
    last = 0;
    if (u < n_units) {
      const long long x = first + static_cast<long long>(u) * kWarps;
      const int i = row_of(row_start, a.num_rows, a.n_kv, x);
      const int npg = row_start[i + 1] - row_start[i];
      const int off = static_cast<int>(x - static_cast<long long>(a.n_kv) * row_start[i]);
      hh = off / npg;
      const int p = off - hh * npg;  // of the pages the row reads, from window_start / 16
      int page = __ldg(a.block_table + static_cast<long long>(i) * a.bt_stride +
                       window_start(lens[i], a.window) / kPage + p);
      last = (p == npg - 1) ? 1 : 0;
      if (page < 0 || page >= a.num_pages) {
        record_status(a.status, PKV_DEV_BAD_PAGE);
        page = 0;
        last = 0;
      }
      pg = page;
      row = i;
    }
  };
  int c_pg, c_h, c_row, c_last, n_pg, n_h, n_row, n_last;
  int batch = 0;
  fetch(0, c_pg, c_h, c_row, c_last);
  int issued = 0;
  const uint64_t policy = policy_evict_first();

  // Issue unit `issued` into its stage (warp-uniform).
  auto issue = [&]() {
    const int u = issued;
    if (u >= batch + 32) {
      c_pg = n_pg;
      c_h = n_h;
      c_row = n_row;
      c_last = n_last;
      batch += 32;
      fetch(batch + 32, n_pg, n_h, n_row, n_last);
    }
    const int jj = u - batch;
    const int pg = __shfl_sync(kFull, c_pg, jj);
    const int hh = __shfl_sync(kFull, c_h, jj);
    if (a.k_new != nullptr && __shfl_sync(kFull, c_last, jj)) {
      const int row = __shfl_sync(kFull, c_row, jj);
      append_token<DT>(a, row, hh, pg, (lens[row] - 1) % kPage, lane);  // row's k_new/v_new
    }
    // The warp's earlier reads of this stage come before the copy rewrites it.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const int s = static_cast<int>(static_cast<unsigned>(u) % R);
      const uint32_t bar = bar0 + 8 * s;
      const uint32_t dst = smem_addr(ring + s * TL::kCodes);
      const int z = pg * a.n_kv + hh;  // tile index (the host checks num_pages * n_kv < 2^31)
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
  // the next batch of descriptors, once the first copies are on their way
  fetch(32, n_pg, n_h, n_row, n_last);

  const int gid = lane >> 2, tig = lane & 3;
  float* mrg_acc = reinterpret_cast<float*>(smem + SM::kMrgAcc);
  float* mrg_ml = reinterpret_cast<float*>(smem + SM::kMrgMl);
  int consumed = 0;
  bool aborted = stalled;
  WarpState<DT> S;
  S.qs = reinterpret_cast<float*>(smem + SM::kQ) + warp * G * kQStride;  // f32 KV only

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
    const int ws = window_start(L, a.window);  // first attended token of the row
    const int p0 = ws / kPage;                 // its page: the row's unit 0
    const long long j = static_cast<long long>(i) * a.n_kv + h;
    int k0, k1;
    segment_chunks(sp, i, h, row_start, pc, a.num_rows, a.n_kv, k0, k1);

    load_query<DT, G>(a.q + (static_cast<long long>(i) * a.n_q + h * G) * kD, a.qscale, lane, S);
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) S.o[r][e] = 0.f;
    S.m = -INFINITY;
    S.l = 0.f;
    S.vx = kNoScale;

    const int r = static_cast<int>((x - c_begin) % kWarps);
    // this warp's units of the piece: offsets rel in the segment (ints: a
    // segment has fewer than 2^31 units), u its index among the warp's units
    const long long pos0 = x + ((warp - r + kWarps) % kWarps);
    const int rel_end = static_cast<int>(b - seg_start);
    int u = static_cast<int>((pos0 - first) / kWarps);
    for (int rel = static_cast<int>(pos0 - seg_start); rel < rel_end; rel += kWarps, ++u) {
      const int s = static_cast<int>(static_cast<unsigned>(u) % R);
      bool ok = !aborted && mbar_wait_bounded(bar0 + 8 * s, (static_cast<unsigned>(u) / R) & 1, ctl);
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
      const int t_page = (p0 + rel) * kPage;  // page's first token
      const int nvalid = min(kPage, L - t_page);
      const int tlo = max(0, ws - t_page);
      process_unit<DT, G>(ring + s * TL::kCodes, ring_sc + s * TL::kScales, tlo, nvalid, lane, S);
      if (issued < n_units) issue();
    }

    // ---- piece end: leave this warp's state in the shared merge buffer.
    // For every piece but the chunk's last, the last warp to arrive merges
    // while the others go on streaming; the chunk's last piece is merged by
    // the whole CTA, since all its warps are done by then.
    float l_tot = S.l;  // head tig's sum over its 8 lanes
    l_tot += __shfl_xor_sync(kFull, l_tot, 4);
    l_tot += __shfl_xor_sync(kFull, l_tot, 8);
    l_tot += __shfl_xor_sync(kFull, l_tot, 16);
    const bool final_piece = (b == c_end);
    int ok = 1;
    if (lane == 0) ok = wait_merge_buffer(ctl, piece);
    ok = __shfl_sync(kFull, ok, 0);
    if (!ok && !aborted) {
      if (lane == 0 && !ctl[0]) {
        ctl[0] = 1;
        record_status(a.status, PKV_DEV_TIMEOUT);
      }
      aborted = true;
    }
    if (tig < G) {
      if (gid == 0) {
        mrg_ml[(warp * G + tig) * 2] = aborted ? -INFINITY : S.m;
        mrg_ml[(warp * G + tig) * 2 + 1] = l_tot;
      }
      float* acc_h = mrg_acc + (warp * G + tig) * kD;
      const float osc = o_scale<DT>(S);
#pragma unroll
      for (int r = 0; r < 8; ++r) {  // hi + lo columns
        acc_h[dim_of<DT>(r, 0, gid)] = (S.o[r][0] + S.o[r][1]) * osc;
        acc_h[dim_of<DT>(r, 2, gid)] = (S.o[r][2] + S.o[r][3]) * osc;
      }
    }
    const bool whole = (k0 == k1);
    float* out_seg = a.out + (static_cast<long long>(i) * a.n_q + h * G) * kD;
    if (final_piece) {
      named_barrier(1, kThreads);
      const bool live = !ctl[0];
      const int d = threadIdx.x;  // one dim per thread, all heads
      const bool split = live && !whole && a.flags != nullptr;
      // Aligned split: every piece of a split segment is the final piece of
      // its chunk, and arrives first, with a relaxed add, while its own merge
      // runs; the last arrival merges, and the others publish their partials
      // afterwards through their ready flags.  Uniform split: the segment's
      // other pieces may have ended inside their chunks, merged by one warp
      // with a release arrival (below), so this piece does the same, but first
      // asks whether the others have all arrived (then it is the last).
      // (q8_0 and f32 always take the uniform split: the aligned protocol is
      // compiled only for the 16-bit formats.)
      constexpr bool kAlignable = DT == PKV_KV_F16 || DT == PKV_KV_BF16;
      const bool aligned = kAlignable && sp.aligned;
      int arrived = -1;
      if (split && threadIdx.x == 0)
        arrived = aligned ? atomicAdd(seg_counter(a.flags, j), 1)
                          : load_acquire(seg_counter(a.flags, j));
      float M[G], Ls[G], A[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M[g] = fmaxf(M[g], mrg_ml[(w * G + g) * 2]);
        Ls[g] = 0.f;
        A[g] = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = exp2f(mrg_ml[(w * G + g) * 2] - M[g]);
          Ls[g] = fmaf(f, mrg_ml[(w * G + g) * 2 + 1], Ls[g]);
          A[g] = fmaf(f, mrg_acc[(w * G + g) * kD + d], A[g]);
        }
      }
      if (live && whole) {
#pragma unroll
        for (int g = 0; g < G; ++g) out_seg[g * kD + d] = A[g] / Ls[g];
      }
      auto write_partial = [&]() {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          a.part_acc[((k + j) * G + g) * kD + d] = A[g];
          if (d == 0) {
            a.part_ml[((k + j) * G + g) * 2] = M[g];
            a.part_ml[((k + j) * G + g) * 2 + 1] = Ls[g];
          }
        }
      };
      if (split && aligned) {
        if (threadIdx.x == 0) ctl[1] = arrived == k1 - k0;
        named_barrier(1, kThreads);  // also: the merge buffer is read
        if (ctl[1]) {  // the last arrival: merge from this piece's registers
          merge_segment_cta_ready<G, DT == PKV_KV_Q8_0 ? 2 : 3>(
              a.part_ml, a.part_acc, a.flags, j, k0, k1, k, M, Ls, A, mrg_acc, mrg_ml, out_seg,
              ctl, a.status);
          if (d == 0) *seg_counter(a.flags, j) = 0;  // ready for the next call
        } else {
          write_partial();
          named_barrier(1, kThreads);  // every thread's stores ordered before thread 0's release
          if (threadIdx.x == 0) store_release(slot_ready(a.flags, k + j), 1);
        }
      } else if (split) {
        // The last piece of a segment to finish merges it.  Every piece
        // stores its partial (the stores go out while the counter load is in
        // flight).  If the others had all arrived when asked, this piece is
        // the last one: it merges from its registers, with no arrival to
        // make (thread 0's acquire, passed on by the barrier, orders the
        // loads of the other partials).  Otherwise it arrives, releasing its
        // partial; the arrival that completes the count merges.
        write_partial();
        if (threadIdx.x == 0) ctl[1] = arrived == k1 - k0;
        named_barrier(1, kThreads);  // also: the merge buffer is read, the partial stored
        bool last = ctl[1] != 0;
        if (!last) {
          if (threadIdx.x == 0)  // the CTA's partial (ordered by the barrier) is released
            ctl[1] = atomic_add_acq_rel(seg_counter(a.flags, j), 1) == k1 - k0;
          named_barrier(1, kThreads);
          last = ctl[1] != 0;
        }
        if (last) {
          merge_segment_cta<G, DT == PKV_KV_Q8_0 ? 2 : 3>(a.part_ml, a.part_acc, j, k0, k1, k, M,
                                                           Ls, A, mrg_acc, mrg_ml, out_seg);
          if (d == 0) *seg_counter(a.flags, j) = 0;  // ready for the next call
        }
      } else if (live && !whole) {
        write_partial();  // for the combine launch
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
        if (live)
          piece_merge<G>(mrg_acc, mrg_ml, whole, out_seg, a.part_ml, a.part_acc, k + j, lane);
        __syncwarp();
        if (lane == 0) {  // release the merge buffer for the next piece
          ctl[1] = 0;
          __threadfence_block();
          ctl[2] = piece + 1;
        }
        if (live && !whole && a.flags != nullptr) {
          __syncwarp();
          int seg_last = 0;
          // the warp's partial (ordered by __syncwarp) is released by the arrival
          if (lane == 0) seg_last = atomic_add_acq_rel(seg_counter(a.flags, j), 1) == k1 - k0;
          seg_last = __shfl_sync(kFull, seg_last, 0);
          if (seg_last) {
            __syncwarp();  // lane 0's acquire, ordered for the warp
            merge_segment_warp<G>(a.part_ml, a.part_acc, j, k0, k1, out_seg, lane);
            if (lane == 0) *seg_counter(a.flags, j) = 0;  // ready for the next call
          }
        }
      }
    }
    x = b;
  }

  // Copies still in flight after an abort must land before the CTA exits.
  if (aborted || ctl[0]) {
    const int zero = 0;
    for (int u = consumed > issued - R ? consumed : issued - R; u < issued; ++u)
      if (u >= 0) mbar_wait_bounded(bar0 + 8 * (u % R), (u / R) & 1, &zero);
  }
}

// ------------------------------------------------------------ combine ----
// One CTA per (row, KV head) segment, one thread per dim: merges the pieces
// of segments split over several chunks; zeros for rows without tokens.
template <int G>
__global__ void __launch_bounds__(kD) combine_kernel(const CombineArgs a) {
  extern __shared__ int csm[];
  __shared__ Split split;
  int* row_start = csm;
  int* lens = csm + a.num_rows + 1;
  int* pc = lens + a.num_rows;
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, a.window, nullptr, lens, row_start);
  plan_split(row_start, a.num_rows, a.n_kv, a.num_chunks, a.aligned_split, &split, pc);
  const int j = blockIdx.x, i = j / a.n_kv, h = j % a.n_kv, d = threadIdx.x;
  const int npg = row_start[i + 1] - row_start[i];
  float* o = a.out + (static_cast<long long>(i) * a.n_q + h * G) * kD;
  if (npg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) o[g * kD + d] = 0.f;
    return;
  }
  int k0, k1;
  segment_chunks(split, i, h, row_start, pc, a.num_rows, a.n_kv, k0, k1);
  if (k0 == k1) return;  // one piece: the attention kernel wrote the output
  merge_segment<G>(a.part_ml, a.part_acc, j, k0, k1, o, d);
}

// ----------------------------------------------------------------- plan ----
__global__ void __launch_bounds__(256) plan_kernel(const PlanArgs a) {
  extern __shared__ int psm[];
  __shared__ Split split;
  int* row_start = psm;
  int* lens = psm + a.num_rows + 1;
  int* pc = lens + a.num_rows;
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, a.window, nullptr, lens, row_start);
  plan_split(row_start, a.num_rows, a.n_kv, a.num_chunks, a.aligned_split, &split, pc);
  for (int r = threadIdx.x; r <= a.num_rows; r += blockDim.x) a.row_page_start[r] = row_start[r];
  for (int j = threadIdx.x; j < a.num_rows * a.n_kv; j += blockDim.x) {
    const int i = j / a.n_kv, h = j % a.n_kv;
    const int npg = row_start[i + 1] - row_start[i];
    int f = -1, l = -1;
    if (npg > 0) segment_chunks(split, i, h, row_start, pc, a.num_rows, a.n_kv, f, l);
    a.seg_first_chunk[j] = f;
    a.seg_last_chunk[j] = l;
  }
}

// ------------------------------------------------------------ launchers ----
// cuTensorMapEncodeTiled, from the driver through the runtime (no link
// against the driver library).
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A layer's K or V data, [tiles][16 tokens][128 dims], as the tensor map a
// tile copy reads through (tma_load_tile), under the 128-byte swizzle:
//   f16, bf16: 4-D {64 dims, 16 tokens, 2 halves, tiles}, strides {256, 128,
//     4096} bytes, box {64, 16, 2, 1}: shared memory [half][16][64];
//   f32: 4-D {32 dims, 16 tokens, 4 quarters, tiles}, strides {512, 128,
//     8192}, box {32, 16, 4, 1}: [quarter][16][32];
//   q8_0: 3-D {128 codes, 16 tokens, tiles}, box {128, 16, 1}: [16][128].
// Each is 16 token rows of 128 bytes per box, the layout the swizzled tile
// addressing (tile_offset) reads.
static cudaError_t encode_tile_map(CUtensorMap* m, int dtype, void* base, long long tiles) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint32_t esize = dtype == PKV_KV_F32 ? 4u : dtype == PKV_KV_Q8_0 ? 1u : 2u;  // bytes
  const cuuint32_t row = 128u / esize;   // elements in a 128-byte row
  const cuuint32_t parts = kD / row;     // rows of a token: 1 (q8_0), 2 (16-bit), 4 (f32)
  const cuuint64_t tok = static_cast<cuuint64_t>(kD) * esize;  // bytes of a token
  const cuuint32_t estride[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapDataType type = dtype == PKV_KV_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                   : dtype == PKV_KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dtype == PKV_KV_F32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                          : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r;
  if (parts == 1) {
    const cuuint64_t dims[3] = {row, static_cast<cuuint64_t>(kPage), static_cast<cuuint64_t>(tiles)};
    const cuuint64_t strides[2] = {tok, tok * kPage};
    const cuuint32_t box[3] = {row, static_cast<cuuint32_t>(kPage), 1u};
    r = fn(m, type, 3, base, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[4] = {row, static_cast<cuuint64_t>(kPage), parts,
                                static_cast<cuuint64_t>(tiles)};
    const cuuint64_t strides[3] = {tok, 128u, tok * kPage};
    const cuuint32_t box[4] = {row, static_cast<cuuint32_t>(kPage), parts, 1u};
    r = fn(m, type, 4, base, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A 16-bit layer's K or V data as 5-D tiles [2 token groups][2 halves][8
// tokens][64 dims] (strides 2048, 128, 256 bytes): one copy lands a tile as
// four 1 KiB blocks, each 8 tokens of one 64-dim half under the 128-byte
// swizzle, so that the 8-token groups of consecutive tiles of one half sit a
// uniform 2 KiB apart in shared memory.
static cudaError_t encode_page_map(CUtensorMap* m, int dtype, void* base, long long tiles) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[5] = {64u, 8u, 2u, 2u, static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[4] = {kD * 2, 128u, 8 * kD * 2, kD * kPage * 2};
  const cuuint32_t box[5] = {64u, 8u, 2u, 2u, 1u};
  const cuuint32_t estride[5] = {1u, 1u, 1u, 1u, 1u};
  const CUresult r = fn(m, dtype == PKV_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        5, base, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tile_maps(int dtype, void* k_data, void* v_data, long long tiles,
                             TileMaps* maps) {
  if (tiles <= 0 || tiles >= (1ll << 31)) return cudaErrorInvalidValue;  // int tile index
  cudaError_t e = encode_tile_map(&maps->k, dtype, k_data, tiles);
  if (e == cudaSuccess) e = encode_tile_map(&maps->v, dtype, v_data, tiles);
  if (dtype == PKV_KV_F16 || dtype == PKV_KV_BF16) {
    if (e == cudaSuccess) e = encode_page_map(&maps->kp, dtype, k_data, tiles);
    if (e == cudaSuccess) e = encode_page_map(&maps->vp, dtype, v_data, tiles);
  } else {
    maps->kp = maps->k;
    maps->vp = maps->v;
  }
  return e;
}

// The kernel's dynamic shared-memory limit, raised only when a call needs
// more than any earlier call (per device).
template <int DT, int G>
static cudaError_t ensure_smem(size_t smem) {
  static std::atomic<size_t> granted[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && granted[dev].load(std::memory_order_relaxed) >= smem)
    return cudaSuccess;
  e = cudaFuncSetAttribute(paged_decode_kernel<DT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e == cudaSuccess && dev >= 0 && dev < 64) {
    size_t cur = granted[dev].load();
    while (cur < smem && !granted[dev].compare_exchange_weak(cur, smem)) {
    }
  }
  return e;
}

template <int DT, int G>
static cudaError_t launch_decode_t(const DecodeArgs& a, const TileMaps& maps, int chunks,
                                   cudaStream_t st) {
  const size_t smem = Smem<DT, G>::bytes(a.num_rows);
  cudaError_t e = ensure_smem<DT, G>(smem);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the grid may be scheduled while the
  // previous kernel of the stream finishes; the kernel itself waits for that
  // kernel's completion before its first global access.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(chunks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = PKV_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, paged_decode_kernel<DT, G>, a, maps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DT, int G>
static cudaError_t occupancy_t(int rows, int* blocks) {
  const size_t smem = Smem<DT, G>::bytes(rows);
  cudaError_t e = ensure_smem<DT, G>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, paged_decode_kernel<DT, G>,
                                                       kThreads, smem);
}

#define PKV_DISPATCH(DT_, G_, CALL)          \
  do {                                       \
    if ((DT_) == PKV_KV_F16) {               \
      if ((G_) == 1) return CALL(0, 1);      \
      if ((G_) == 2) return CALL(0, 2);      \
      if ((G_) == 4) return CALL(0, 4);      \
    } else if ((DT_) == PKV_KV_BF16) {       \
      if ((G_) == 1) return CALL(2, 1);      \
      if ((G_) == 2) return CALL(2, 2);      \
      if ((G_) == 4) return CALL(2, 4);      \
    } else if ((DT_) == PKV_KV_F32) {        \
      if ((G_) == 1) return CALL(3, 1);      \
      if ((G_) == 2) return CALL(3, 2);      \
      if ((G_) == 4) return CALL(3, 4);      \
    } else {                                 \
      if ((G_) == 1) return CALL(1, 1);      \
      if ((G_) == 2) return CALL(1, 2);      \
      if ((G_) == 4) return CALL(1, 4);      \
    }                                        \
    return cudaErrorInvalidValue;            \
  } while (0)

cudaError_t launch_paged_decode(int dtype, int group, const DecodeArgs& a, const TileMaps& maps,
                                int chunks, cudaStream_t st) {
#define PKV_CALL(D, G) launch_decode_t<D, G>(a, maps, chunks, st)
  PKV_DISPATCH(dtype, group, PKV_CALL);
#undef PKV_CALL
}

cudaError_t paged_decode_blocks_per_sm(int dtype, int group, int rows, int* blocks) {
#define PKV_CALL(D, G) occupancy_t<D, G>(rows, blocks)
  PKV_DISPATCH(dtype, group, PKV_CALL);
#undef PKV_CALL
}

cudaError_t launch_combine(int group, const CombineArgs& a, cudaStream_t st) {
  const int segs = a.num_rows * a.n_kv;
  if (segs == 0) return cudaSuccess;
  const size_t smem = plan_ints(a.num_rows) * sizeof(int);
  if (group == 1)
    combine_kernel<1><<<segs, kD, smem, st>>>(a);
  else if (group == 2)
    combine_kernel<2><<<segs, kD, smem, st>>>(a);
  else if (group == 4)
    combine_kernel<4><<<segs, kD, smem, st>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t st) {
  const size_t smem = plan_ints(a.num_rows) * sizeof(int);
  plan_kernel<<<1, 256, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv

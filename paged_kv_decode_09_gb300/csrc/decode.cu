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
// one per (row, KV head, page) in that order.  With C = min(grid, T) chunks,
// CTA k < C takes units [floor(kT/C), floor((k+1)T/C)) (never empty; CTAs
// k >= C idle), so every CTA streams the same number of
// 4 KiB (f16) or 2176-byte (q8_0) tiles whatever the length mix: one 40k-token
// row and many 16-token rows keep all SMs equally busy.  The units of one
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
struct Tiles<PKV_KV_Q8_0> {
  static constexpr uint32_t kData = kPage * kD;                   // 2048 codes
  static constexpr uint32_t kScale = kPage * (kD / kQBlock) * 2;  // 128 bytes of f16 scales
  static constexpr uint32_t kCodes = 2 * kData;
  static constexpr uint32_t kScales = 2 * kScale;  // K scales then V scales
  static constexpr uint32_t kTx = kCodes + kScales;
  static constexpr int kRing = PKV_Q8_RING;  // stages per warp
};

// Offsets from a 1024-byte aligned base.  The tiles come first (the swizzle
// atom is 1024 bytes), then scales, barriers, the merge buffer, control
// words and the plan.
template <int DT, int G>
struct Smem {
  static constexpr int kStages = kWarps * Tiles<DT>::kRing;
  static constexpr uint32_t kAlign = 1024;
  static constexpr uint32_t kScl = kStages * Tiles<DT>::kCodes;           // [warp][ring][K, V]
  static constexpr uint32_t kBar = kScl + kStages * Tiles<DT>::kScales;   // full[warp][ring]
  static constexpr uint32_t kMrgAcc = kBar + ((kStages * 8 + 15) / 16) * 16;  // f32 [warps][G][D]
  static constexpr uint32_t kMrgMl = kMrgAcc + kWarps * G * kD * 4;        // f32 [warps][G][2]
  static constexpr uint32_t kCtl = kMrgMl + kWarps * G * 2 * 4;            // int [4]
  static constexpr uint32_t kRows = kCtl + 16;  // int row_start[rows + 1], lens[rows]
  static size_t bytes(int rows) {
    return kAlign + kRows + (2 * static_cast<size_t>(rows) + 1) * 4;  // kAlign: base alignment slack
  }
  static_assert(Tiles<DT>::kCodes % 1024 == 0, "tile stages keep the swizzle atom alignment");
  static_assert(kMrgAcc % 16 == 0 && kMrgMl % 16 == 0 && kCtl % 16 == 0,
                "vector accesses need 16-byte aligned regions");
};

// ------------------------------------------------------------ operands ----
// Byte offset of the 16-byte chunk c (8 f16 or 16 int8 values) of token row t
// in a swizzled tile: 128-byte rows, chunk index xor (row mod 8); f16 tiles
// keep dims 64..127 in a second 2 KiB half.
template <int DT>
__device__ __forceinline__ uint32_t tile_offset(int t, int c) {
  if constexpr (DT != PKV_KV_Q8_0)
    return (c >> 3) * 2048 + t * 128 + (((c & 7) ^ (t & 7)) << 4);
  else
    return t * 128 + ((c ^ (t & 7)) << 4);
}

// Two signed 8-bit codes of `u` (the word xor 0x80808080, i.e. code + 128 in
// each byte) as an exact f16 pair: the bytes chosen by `sel` go into the low
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

// Per-warp online softmax state for one piece.
template <int DT>
struct WarpState {
  static constexpr int kSteps = DT == PKV_KV_BF16 ? 16 : 8;  // score k-steps (tf32: 8 dims)
  uint32_t qb[kSteps][2];  // B operand of the scores per k-step: column gid (head gid/2, part gid%2)
  float qexp;         // 2^e of head tig: undoes its power-of-two normalisation
  float m;            // running max (base 2) of head tig, equal on its 8 lanes
  float l;            // this lane's share of head tig's sum of probabilities
  float o[8][4];      // O^T accumulators: dims (see dim_of) x columns (tig, hi), (tig, lo)
  int vx;             // q8_0: every V block scale of the piece so far is below 2^vx
};

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
template <int DT>
__device__ __forceinline__ float o_scale(const WarpState<DT>& S) {
  if constexpr (DT == PKV_KV_F16)
    return 1.0f / (1 << kPShift);
  else if constexpr (DT == PKV_KV_BF16)
    return 1.0f;  // tf32 parts have the fp32 exponent range: no scaling
  else
    return pow2i(S.vx - kPShift);
}

// The dim of accumulator o[r][e] (e = 0, 2; e + 1 is its lo column) in lane
// 4 gid + tig.
template <int DT>
__device__ __forceinline__ int dim_of(int r, int e, int gid) {
  if constexpr (DT != PKV_KV_Q8_0)
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
  if constexpr (DT == PKV_KV_BF16) {
    // tf32 k-steps of 8 dims: k = tig <- dim 8ks + 2tig, k = tig + 4 <- dim 8ks + 2tig + 1
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      float2 x = make_float2(0.f, 0.f);
      if (g2 < G) x = __ldg(reinterpret_cast<const float2*>(qrow + g2 * kD + 8 * ks + 2 * tig));
      S.qb[ks][0] = tf32_part(x.x * qscale, lo);
      S.qb[ks][1] = tf32_part(x.y * qscale, lo);
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
      S.qb[ks][0] = split_f16x2(ldexpf(v[4 * ks], -e2), ldexpf(v[4 * ks + 1], -e2), lo);
      S.qb[ks][1] = split_f16x2(ldexpf(v[4 * ks + 2], -e2), ldexpf(v[4 * ks + 3], -e2), lo);
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
  if constexpr (DT == PKV_KV_BF16) {
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
      w0 ^= 0x80808080u;
      w1 ^= 0x80808080u;
      w2 ^= 0x80808080u;
      w3 ^= 0x80808080u;
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
    const float al = exp2f(S.m - m_new);  // 1 if unchanged, 0 from -inf
    S.l *= al;
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) S.o[r][e] *= al;
    S.m = m_new;
  }
  const float p0 = exp2f(s0 - S.m), p1 = exp2f(s1 - S.m);
  S.l += p0 + p1;

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
  if constexpr (DT != PKV_KV_Q8_0) {
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
      const uint32_t b0 = split_f16x2(pa * kUp, pb * kUp, lo);
      const uint32_t b1 = split_f16x2(pc * kUp, pd * kUp, lo);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t w0, w1, w2, w3;  // (tokens 0-7 | 8-15) x (chunk 2mt | 2mt+1), transposed
        ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * mt + ld_chunk), w0, w1, w2, w3);
        mma_16816(S.o[mt], w0, w2, w1, w3, b0, b1);
      }
    } else {
      // tf32 k-steps of 8 tokens: k = tig <- token 2tig, k = tig + 4 <- token 2tig + 1
      const uint32_t b_t0 = tf32_part(pa, lo), b_t1 = tf32_part(pb, lo);
      const uint32_t b_t8 = tf32_part(pc, lo), b_t9 = tf32_part(pd, lo);
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
    // the page's largest |scale|: non-negative f16 bit patterns order as integers
    uint32_t mb = __vmaxu2(__vmaxu2(va.x & 0x7fff7fffu, va.y & 0x7fff7fffu),
                           __vmaxu2(va.z & 0x7fff7fffu, va.w & 0x7fff7fffu));
    mb = __vmaxu2(mb, __vmaxu2(__vmaxu2(vb.x & 0x7fff7fffu, vb.y & 0x7fff7fffu),
                               __vmaxu2(vb.z & 0x7fff7fffu, vb.w & 0x7fff7fffu)));
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
      const uint32_t b0 = split_f16x2(x0, x1, lo), b1 = split_f16x2(x2, x3, lo);
      uint32_t w0, w1, w2, w3;  // (tokens 0-7 | 8-15) x (chunk 2b | 2b+1), 16-bit transposed
      ldsm_x4_trans(vt + tile_offset<DT>(ld_tok, 2 * b + ld_chunk), w0, w1, w2, w3);
      w0 ^= 0x80808080u;
      w1 ^= 0x80808080u;
      w2 ^= 0x80808080u;
      w3 ^= 0x80808080u;
      // row gid <- dim 2gid of the chunk (bytes 0, 2), row gid + 8 <- dim 2gid+1 (bytes 1, 3)
      mma_16816(S.o[2 * b], codes_to_f16x2<kSelB02>(w0), codes_to_f16x2<kSelB13>(w0),
                codes_to_f16x2<kSelB02>(w1), codes_to_f16x2<kSelB13>(w1), b0, b1);
      mma_16816(S.o[2 * b + 1], codes_to_f16x2<kSelB02>(w2), codes_to_f16x2<kSelB13>(w2),
                codes_to_f16x2<kSelB02>(w3), codes_to_f16x2<kSelB13>(w3), b0, b1);
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------- merge ----
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

// ------------------------------------------------------------- append ----
// A warp stores row i's new K and V token of KV head h into slot (L - 1) % 16
// of tile (page, h) just before it bulk-copies that tile: 4 dims per lane;
// q8_0 blocks of 32 dims span 8 lanes.  Same encoding as kv_append.
template <int DT>
__device__ __forceinline__ void append_token(const DecodeArgs& a, int i, int h, int page,
                                                   int slot, int lane) {
  using TL = Tiles<DT>;
  const size_t tile = static_cast<size_t>(page) * a.n_kv + h;
  const long long src = (static_cast<long long>(i) * a.n_kv + h) * kD + lane * 4;
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
      *reinterpret_cast<uint32_t*>(data + tile * TL::kData + slot * kD + lane * 4) = packed;
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

// --------------------------------------------------------------- kernel ----
template <int DT, int G>
__global__ void __launch_bounds__(kThreads, DT != PKV_KV_Q8_0 ? PKV_F16_CTAS_PER_SM
                                                              : PKV_Q8_CTAS_PER_SM)
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
  const uint32_t bar0 = smem_addr(smem + SM::kBar) + warp * R * 8;  // this warp's barriers
  uint8_t* ring = smem + static_cast<size_t>(warp) * R * TL::kCodes;  // this warp's tiles
  uint8_t* ring_sc = smem + SM::kScl + static_cast<size_t>(warp) * R * TL::kScales;  // q8_0 scales

  if (threadIdx.x == 0) {
    ctl[0] = 0;
    ctl[1] = 0;
    ctl[2] = 0;
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

  const long long T = static_cast<long long>(a.n_kv) * row_start[a.num_rows];
  const int C = used_chunks(T, gridDim.x), k = blockIdx.x;
  const long long c_begin = k < C ? static_cast<long long>(k) * T / C : T;
  const long long c_end = k < C ? static_cast<long long>(k + 1) * T / C : T;

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
  fetch(32, n_pg, n_h, n_row, n_last);
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
      append_token<DT>(a, row, hh, pg, (lens[row] - 1) % kPage, lane);
    }
    // The warp's earlier reads of this stage come before the copy rewrites it.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const int s = u % R;
      const uint32_t bar = bar0 + 8 * s;
      const uint32_t dst = smem_addr(ring + s * TL::kCodes);
      const int z = pg * a.n_kv + hh;  // tile index (the host checks num_pages * n_kv < 2^31)
      mbar_arrive_expect_tx(bar, TL::kTx);
      if constexpr (DT != PKV_KV_Q8_0) {
        tma_load_3d(dst, &maps.k, 0, 0, z, bar, policy);
        tma_load_3d(dst + 2048, &maps.k, 64, 0, z, bar, policy);
        tma_load_3d(dst + TL::kData, &maps.v, 0, 0, z, bar, policy);
        tma_load_3d(dst + TL::kData + 2048, &maps.v, 64, 0, z, bar, policy);
      } else {
        const uint32_t sdst = smem_addr(ring_sc + s * TL::kScales);
        const size_t unit = static_cast<size_t>(z);
        tma_load_3d(dst, &maps.k, 0, 0, z, bar, policy);
        bulk_g2s(sdst, a.k_scales + unit * TL::kScale, TL::kScale, bar, policy);
        tma_load_3d(dst + TL::kData, &maps.v, 0, 0, z, bar, policy);
        bulk_g2s(sdst + TL::kScale, a.v_scales + unit * TL::kScale, TL::kScale, bar, policy);
      }
    }
    ++issued;
  };
  while (issued < n_units && issued < R) issue();

  const int gid = lane >> 2, tig = lane & 3;
  float* mrg_acc = reinterpret_cast<float*>(smem + SM::kMrgAcc);
  float* mrg_ml = reinterpret_cast<float*>(smem + SM::kMrgMl);
  bool aborted = false;
  int consumed = 0;
  WarpState<DT> S;

  int piece = 0;
  for (long long x = c_begin; x < c_end; ++piece) {
    const int i = row_of(row_start, a.num_rows, a.n_kv, x);
    const int npg = row_start[i + 1] - row_start[i];
    const long long row_base = static_cast<long long>(a.n_kv) * row_start[i];
    const int h = static_cast<int>((x - row_base) / npg);
    const long long seg_start = row_base + static_cast<long long>(h) * npg;
    const long long seg_end = seg_start + npg;
    const long long b = min(seg_end, c_end);
    const int L = lens[i];
    const int ws = window_start(L, a.window);  // first attended token of the row
    const int p0 = ws / kPage;                 // its page: the row's unit 0
    const long long j = static_cast<long long>(i) * a.n_kv + h;
    const int k0 = chunk_of(seg_start, T, C), k1 = chunk_of(seg_end - 1, T, C);

    load_query<DT, G>(a.q + (static_cast<long long>(i) * a.n_q + h * G) * kD, a.qscale, lane, S);
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) S.o[r][e] = 0.f;
    S.m = -INFINITY;
    S.l = 0.f;
    S.vx = kNoScale;

    const int r = static_cast<int>((x - c_begin) % kWarps);
    for (long long pos = x + ((warp - r + kWarps) % kWarps); pos < b; pos += kWarps) {
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
      const int t_page = (p0 + static_cast<int>(pos - seg_start)) * kPage;  // page's first token
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
      if (live) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mrg_ml[(w * G + g) * 2]);
          float Ls = 0.f, A = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(mrg_ml[(w * G + g) * 2] - M);
            Ls = fmaf(f, mrg_ml[(w * G + g) * 2 + 1], Ls);
            A = fmaf(f, mrg_acc[(w * G + g) * kD + d], A);
          }
          if (whole) {
            out_seg[g * kD + d] = A / Ls;
          } else {
            a.part_acc[((k + j) * G + g) * kD + d] = A;
            if (d == 0) {
              a.part_ml[((k + j) * G + g) * 2] = M;
              a.part_ml[((k + j) * G + g) * 2 + 1] = Ls;
            }
          }
        }
      }
      const bool counted = live && !whole && a.counters != nullptr;
      named_barrier(1, kThreads);
      if (threadIdx.x == 0) {
        int seg_last = 0;
        if (counted) {
          __threadfence();  // the CTA's partial (ordered by the barrier) before the arrival
          seg_last = atomicAdd(a.counters + j, 1) == k1 - k0;
        }
        ctl[1] = seg_last;
      }
      named_barrier(1, kThreads);
      if (ctl[1]) {
        __threadfence();
        merge_segment<G, DT != PKV_KV_Q8_0 ? PKV_MERGE_BATCH : PKV_MERGE_BATCH / 2>(
            a.part_ml, a.part_acc, j, k0, k1, out_seg, d);
        if (d == 0) a.counters[j] = 0;  // ready for the next call
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
        if (live && !whole && a.counters != nullptr) {
          __syncwarp();
          int seg_last = 0;
          if (lane == 0) {
            __threadfence();  // the warp's partial (ordered by __syncwarp) before the arrival
            seg_last = atomicAdd(a.counters + j, 1) == k1 - k0;
          }
          seg_last = __shfl_sync(kFull, seg_last, 0);
          if (seg_last) {
            __threadfence();
            merge_segment_warp<G>(a.part_ml, a.part_acc, j, k0, k1, out_seg, lane);
            if (lane == 0) a.counters[j] = 0;  // ready for the next call
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
  int* row_start = csm;
  int* lens = csm + a.num_rows + 1;
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, a.window, nullptr, lens, row_start);
  const int j = blockIdx.x, i = j / a.n_kv, h = j % a.n_kv, d = threadIdx.x;
  const int npg = row_start[i + 1] - row_start[i];
  float* o = a.out + (static_cast<long long>(i) * a.n_q + h * G) * kD;
  if (npg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) o[g * kD + d] = 0.f;
    return;
  }
  const long long T = static_cast<long long>(a.n_kv) * row_start[a.num_rows];
  const int C = used_chunks(T, a.num_chunks);
  const long long s0 = static_cast<long long>(a.n_kv) * row_start[i] + static_cast<long long>(h) * npg;
  const int k0 = chunk_of(s0, T, C), k1 = chunk_of(s0 + npg - 1, T, C);
  if (k0 == k1) return;  // one piece: the attention kernel wrote the output
  merge_segment<G>(a.part_ml, a.part_acc, j, k0, k1, o, d);
}

// ----------------------------------------------------------------- plan ----
__global__ void __launch_bounds__(256) plan_kernel(const PlanArgs a) {
  extern __shared__ int psm[];
  int* row_start = psm;
  int* lens = psm + a.num_rows + 1;
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, a.window, nullptr, lens, row_start);
  for (int r = threadIdx.x; r <= a.num_rows; r += blockDim.x) a.row_page_start[r] = row_start[r];
  const long long T = static_cast<long long>(a.n_kv) * row_start[a.num_rows];
  const int C = used_chunks(T, a.num_chunks);
  for (int j = threadIdx.x; j < a.num_rows * a.n_kv; j += blockDim.x) {
    const int i = j / a.n_kv, h = j % a.n_kv;
    const int npg = row_start[i + 1] - row_start[i];
    int f = -1, l = -1;
    if (npg > 0) {
      const long long s0 = static_cast<long long>(a.n_kv) * row_start[i] + static_cast<long long>(h) * npg;
      f = chunk_of(s0, T, C);
      l = chunk_of(s0 + npg - 1, T, C);
    }
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

// A layer's K or V data as a 3-D tensor [tiles][16 tokens][128 dims] read in
// [16][64] (f16) or [16][128] (q8_0 codes) boxes of 128-byte rows under the
// 128-byte swizzle.
static cudaError_t encode_tile_map(CUtensorMap* m, int dtype, void* base, long long tiles) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const bool f16 = dtype != PKV_KV_Q8_0;  // 16-bit values (f16, bf16)
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(kPage),
                              static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[2] = {f16 ? 256u : 128u, f16 ? 4096u : 2048u};  // bytes
  const cuuint32_t box[3] = {f16 ? 64u : 128u, static_cast<cuuint32_t>(kPage), 1u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUresult r =
      fn(m, dtype == PKV_KV_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
            : dtype == PKV_KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8,
         3, base, dims,
         strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tile_maps(int dtype, void* k_data, void* v_data, long long tiles,
                             TileMaps* maps) {
  if (tiles <= 0 || tiles >= (1ll << 31)) return cudaErrorInvalidValue;  // int tile index
  cudaError_t e = encode_tile_map(&maps->k, dtype, k_data, tiles);
  if (e == cudaSuccess) e = encode_tile_map(&maps->v, dtype, v_data, tiles);
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
  const size_t smem = (2 * static_cast<size_t>(a.num_rows) + 1) * sizeof(int);
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
  const size_t smem = (2 * static_cast<size_t>(a.num_rows) + 1) * sizeof(int);
  plan_kernel<<<1, 256, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv

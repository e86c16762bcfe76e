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
// the 1-D bulk async copies of its next units (K tile, then V tile, of one
// (page, KV head)), waits on the stage's mbarrier, computes, and re-issues
// into the stage it just read.  Each stage has one owner, so no empty
// barriers are needed and four threads per CTA keep copies in flight.  Each
// warp keeps a base-2 online softmax in fp32 for the G query heads of the
// unit's KV head, sharing every K and V element it converts across the group.
// At the end of a piece the warps leave their states in a shared merge
// buffer; the last to arrive combines them and does the global writes,
// while the others carry on streaming.
//
// Lane layout of a warp on one 16-token page (lane = 8 tg + dj):
//   scores: lane handles tokens 4tg..4tg+3 and 16 of the 128 dims (f16: two
//     8-dim chunks dj and dj+8; q8_0: the 16 dims 16dj..16dj+15, inside one
//     32-wide q8_0 block), for all G heads; the 8 lanes of a token group then
//     reduce-scatter their 4G partial dot products (3 shuffle steps), leaving
//     each lane max(G/2, 1) complete scores of one head.
//   values: lane owns dims 4 lane .. 4 lane + 3 of the accumulator for all G
//     heads and walks all 16 tokens, reading the probabilities from shared
//     memory.
#include <cmath>
#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// Build-time knobs (defaults are the tuned values): consumer warps per CTA,
// shared-memory stages per dtype, and the minimum CTAs per SM the register
// allocation must allow.
#ifndef PKV_F16_RING
#define PKV_F16_RING 2
#endif
#ifndef PKV_Q8_RING
#define PKV_Q8_RING 3
#endif
#ifndef PKV_MIN_CTAS_PER_SM
#define PKV_MIN_CTAS_PER_SM 3
#endif
#ifndef PKV_MERGE_BATCH
#define PKV_MERGE_BATCH 8
#endif

constexpr int kWarps = 4;  // warps per CTA; the piece merge gives each lane 4 of the 128 dims
constexpr int kThreads = kWarps * 32;

// Shared-memory stage of one unit: the K tile then the V tile of one
// (page, KV head); q8_0 tiles are codes followed by their block scales.
template <int DT>
struct Tiles;
template <>
struct Tiles<PKV_KV_F16> {
  static constexpr uint32_t kData = kPage * kD * 2;  // 4096
  static constexpr uint32_t kScale = 0;
  static constexpr uint32_t kTile = kData;
  static constexpr uint32_t kStage = 2 * kTile;
  static constexpr int kRing = PKV_F16_RING;  // stages per warp
};
template <>
struct Tiles<PKV_KV_Q8_0> {
  static constexpr uint32_t kData = kPage * kD;                   // 2048 codes
  static constexpr uint32_t kScale = kPage * (kD / kQBlock) * 2;  // 128 bytes of f16 scales
  static constexpr uint32_t kTile = kData + kScale;
  static constexpr uint32_t kStage = 2 * kTile;
  static constexpr int kRing = PKV_Q8_RING;  // stages per warp
};

// Lane bookkeeping of the score phase for a GQA group of G query heads.
template <int G>
struct Group {
  static_assert(G == 1 || G == 2 || G == 4, "group of 1, 2 or 4 query heads");
  static constexpr int kLog2 = G == 1 ? 0 : (G == 2 ? 1 : 2);
  static constexpr int kVals = 4 * G;              // partial dot products per lane
  static constexpr int kSpl = G >= 2 ? G / 2 : 1;  // complete scores per lane afterwards
  static constexpr int kTokLanes = 4 / kSpl;       // lanes (low dj bits) splitting a head's 4 tokens
};

template <int DT, int G>
struct Smem {
  static constexpr int kStages = kWarps * Tiles<DT>::kRing;
  static constexpr uint32_t kBar = kStages * Tiles<DT>::kStage;           // full[warp][ring]
  static constexpr uint32_t kMrgAcc = kBar + ((kStages * 8 + 15) / 16) * 16;  // f32 [warps][G][D]
  static constexpr uint32_t kMrgMl = kMrgAcc + kWarps * G * kD * 4;        // f32 [warps][G][2]
  // probabilities per warp: f16 [G][16]; q8_0 [4 blocks][G][16] (pre-scaled by V block scales)
  static constexpr int kProbPerWarp = (DT == PKV_KV_F16 ? 1 : kD / kQBlock) * G * kPage;
  static constexpr uint32_t kProb = kMrgMl + kWarps * G * 2 * 4;           // f32 [warps][kProbPerWarp]
  static constexpr uint32_t kAlpha = kProb + kWarps * kProbPerWarp * 4;    // f32 [warps][4]
  static constexpr uint32_t kCtl = kAlpha + kWarps * 4 * 4;                // int [4]
  static constexpr uint32_t kRows = kCtl + 16;  // int row_start[rows + 1], lens[rows]
  static size_t bytes(int rows) { return kRows + (2 * static_cast<size_t>(rows) + 1) * 4; }
  static_assert(kMrgAcc % 16 == 0 && kMrgMl % 16 == 0 && kProb % 16 == 0 && kAlpha % 16 == 0,
                "vector accesses need 16-byte aligned regions");
};

// ---------------------------------------------------------- conversions ----
__device__ __forceinline__ void f16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ void f16x4_to_f32(const uint2& u, float* f) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

// Four signed bytes to floats, exactly: bias each byte to b + 128 (xor 0x80),
// place it in the low mantissa byte of 2^23 (the float 2^23 + b + 128), and
// subtract 2^23 + 128 -- one byte permute per value and one packed subtract
// per pair instead of integer-to-float conversions.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float* f) {
  const uint32_t u = w ^ 0x80808080u;
  const float2 bias = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  const float2 lo = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                           __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441))),
                               bias);
  const float2 hi = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                           __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443))),
                               bias);
  f[0] = lo.x;
  f[1] = lo.y;
  f[2] = hi.x;
  f[3] = hi.y;
}

// ------------------------------------------------------- warp reductions ----
// One reduce-scatter step over lane bit `mask`: N values in, N/2 out.  Lanes
// with the bit set keep the upper half, the others the lower half, each
// adding its partner's copy.
template <int N>
__device__ __forceinline__ void rs_step(float* v, int mask, int lane) {
  const bool up = (lane & mask) != 0;
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    const float send = up ? v[k] : v[k + N / 2];
    const float keep = up ? v[k + N / 2] : v[k];
    v[k] = keep + __shfl_xor_sync(kFull, send, mask);
  }
}

// Full dot products of the 8 lanes of a token group: v[g*4 + j] (token
// 4tg + j, head g) in, Group<G>::kSpl complete scores out in v[0..kSpl): head
// dj >> (3 - log2 G), tokens 4tg + (dj & (kTokLanes-1)) * kSpl + s.
template <int G>
__device__ __forceinline__ void reduce_scores(float* v, int lane) {
  if constexpr (G == 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] += __shfl_xor_sync(kFull, v[k], 4);
    rs_step<4>(v, 2, lane);
    rs_step<2>(v, 1, lane);
  } else {
    rs_step<4 * G>(v, 4, lane);
    rs_step<2 * G>(v, 2, lane);
    rs_step<G>(v, 1, lane);
  }
}

// Sum (or max) over the lanes holding distinct tokens of the lane's head.
template <int G>
__device__ __forceinline__ float head_sum(float x) {
#pragma unroll
  for (int m = 1; m < Group<G>::kTokLanes; m <<= 1) x += __shfl_xor_sync(kFull, x, m);
  x += __shfl_xor_sync(kFull, x, 8);
  x += __shfl_xor_sync(kFull, x, 16);
  return x;
}
template <int G>
__device__ __forceinline__ float head_max(float x) {
#pragma unroll
  for (int m = 1; m < Group<G>::kTokLanes; m <<= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, m));
  x = fmaxf(x, __shfl_xor_sync(kFull, x, 8));
  x = fmaxf(x, __shfl_xor_sync(kFull, x, 16));
  return x;
}

// Per-consumer-warp online softmax state for one piece.
template <int G>
struct WarpState {
  float2 q[G][8];    // this lane's 16 dims of each query head (pairs), times scale*log2(e)
  float m;           // running max (base 2) of the lane's head
  float l;           // running sum of the lane's own tokens (reduced at the end)
  float2 acc[G][2];  // dims 4 lane .. 4 lane + 3 of each head (pairs)
};

// The dims of q a lane's 16 score-phase registers hold.
template <int DT>
__device__ __forceinline__ int q_dim(int dj, int e) {
  if constexpr (DT == PKV_KV_F16)
    return (e < 8) ? dj * 8 + e : 64 + dj * 8 + (e - 8);
  else
    return dj * 16 + e;
}

// Process one staged (page, KV head) unit of nvalid tokens (1..16).
template <int DT, int G>
__device__ __forceinline__ void process_unit(const uint8_t* st, int nvalid, int lane,
                                             WarpState<G>& S, float* prob, float* alpha) {
  using GR = Group<G>;
  using TL = Tiles<DT>;
  const int tg = lane >> 3, dj = lane & 7;

  // ---- scores: 4 tokens x 16 dims x G heads per lane
  float v[GR::kVals];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int t = tg * 4 + j;
    float kf[16];
    float ksc = 1.0f;
    if constexpr (DT == PKV_KV_F16) {
      const uint4 a = *reinterpret_cast<const uint4*>(st + t * 256 + dj * 16);
      const uint4 b = *reinterpret_cast<const uint4*>(st + t * 256 + 128 + dj * 16);
      f16x8_to_f32(a, kf);
      f16x8_to_f32(b, kf + 8);
    } else {
      const uint4 c = *reinterpret_cast<const uint4*>(st + t * kD + dj * 16);
      i8x4_to_f32(c.x, kf);
      i8x4_to_f32(c.y, kf + 4);
      i8x4_to_f32(c.z, kf + 8);
      i8x4_to_f32(c.w, kf + 12);
      const __half* sc = reinterpret_cast<const __half*>(st + TL::kData);
      ksc = __half2float(sc[t * (kD / kQBlock) + (dj >> 1)]);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      // packed fp32 FMA on dim pairs: one pair accumulator per (head, token)
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        s2 = __ffma2_rn(S.q[g][e], make_float2(kf[2 * e], kf[2 * e + 1]), s2);
      v[g * 4 + j] = (s2.x + s2.y) * ksc;
    }
  }
  reduce_scores<G>(v, lane);

  // ---- online softmax of the lane's head over this page
  const int g_lane = dj >> (3 - GR::kLog2);
  const int t0 = tg * 4 + (dj & (GR::kTokLanes - 1)) * GR::kSpl;
  float mx = -INFINITY;
#pragma unroll
  for (int s = 0; s < GR::kSpl; ++s) {
    if (t0 + s >= nvalid) v[s] = -INFINITY;
    mx = fmaxf(mx, v[s]);
  }
  mx = head_max<G>(mx);
  const float m_new = fmaxf(S.m, mx);
  const float al = exp2f(S.m - m_new);
  float psum = 0.f;
#pragma unroll
  for (int s = 0; s < GR::kSpl; ++s) {
    const float p = exp2f(v[s] - m_new);
    psum += p;
    if constexpr (DT == PKV_KV_F16) {
      prob[g_lane * kPage + t0 + s] = p;
    } else {
      // q8_0: fold the V block scales of token t0+s into its probability:
      // prob[block][head][token] = p * scale(V, token, block).
      const int t = t0 + s;
      const uint2 sc4 = *reinterpret_cast<const uint2*>(st + TL::kTile + TL::kData +
                                                        t * (kD / kQBlock) * 2);
      const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sc4.x));
      const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&sc4.y));
      prob[(0 * G + g_lane) * kPage + t] = p * s01.x;
      prob[(1 * G + g_lane) * kPage + t] = p * s01.y;
      prob[(2 * G + g_lane) * kPage + t] = p * s23.x;
      prob[(3 * G + g_lane) * kPage + t] = p * s23.y;
    }
  }
  S.l = S.l * al + psum;
  S.m = m_new;
  if (tg == 0 && (dj & (GR::kTokLanes - 1)) == 0) alpha[g_lane] = al;
  __syncwarp();

  // ---- values: acc[g][dims of lane] = acc * alpha + sum_t p[g][t] V[t]
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float2 a2 = make_float2(alpha[g], alpha[g]);
    S.acc[g][0] = __fmul2_rn(S.acc[g][0], a2);
    S.acc[g][1] = __fmul2_rn(S.acc[g][1], a2);
  }
  const uint8_t* vt = st + TL::kTile;
  // f16: prob[head][token]; q8_0: prob[block][head][token], block of this lane's dims
  const float* pl = (DT == PKV_KV_F16) ? prob : prob + (lane >> 3) * G * kPage;
  if (nvalid == kPage) {
#pragma unroll
    for (int t4 = 0; t4 < kPage; t4 += 4) {
      float4 p4[G];
#pragma unroll
      for (int g = 0; g < G; ++g) p4[g] = *reinterpret_cast<const float4*>(pl + g * kPage + t4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = t4 + u;
        float vf[4];
        if constexpr (DT == PKV_KV_F16)
          f16x4_to_f32(*reinterpret_cast<const uint2*>(vt + t * 256 + lane * 8), vf);
        else
          i8x4_to_f32(*reinterpret_cast<const uint32_t*>(vt + t * kD + lane * 4), vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = (&p4[g].x)[u];
          const float2 p2 = make_float2(p, p);
          S.acc[g][0] = __ffma2_rn(p2, make_float2(vf[0], vf[1]), S.acc[g][0]);
          S.acc[g][1] = __ffma2_rn(p2, make_float2(vf[2], vf[3]), S.acc[g][1]);
        }
      }
    }
  } else {
#pragma unroll 1
    for (int t = 0; t < nvalid; ++t) {
      float vf[4];
      if constexpr (DT == PKV_KV_F16)
        f16x4_to_f32(*reinterpret_cast<const uint2*>(vt + t * 256 + lane * 8), vf);
      else
        i8x4_to_f32(*reinterpret_cast<const uint32_t*>(vt + t * kD + lane * 4), vf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = pl[g * kPage + t];
        const float2 p2 = make_float2(p, p);
        S.acc[g][0] = __ffma2_rn(p2, make_float2(vf[0], vf[1]), S.acc[g][0]);
        S.acc[g][1] = __ffma2_rn(p2, make_float2(vf[2], vf[3]), S.acc[g][1]);
      }
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
template <int G>
__device__ __forceinline__ void merge_segment(const float* part_ml, const float* part_acc,
                                              long long j, int k0, int k1, float* o, int d) {
  constexpr int kBatch = PKV_MERGE_BATCH;  // pieces loaded per round trip, all G heads at once
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
__global__ void __launch_bounds__(kThreads, PKV_MIN_CTAS_PER_SM)
    paged_decode_kernel(const DecodeArgs a) {
  using TL = Tiles<DT>;
  using SM = Smem<DT, G>;
  using GR = Group<G>;
  constexpr int R = TL::kRing;
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // [0] abort  [1] warps arrived at the current piece end  [2] merge-buffer generation
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + SM::kCtl);
  int* row_start = reinterpret_cast<int*>(smem + SM::kRows);
  int* lens = row_start + a.num_rows + 1;
  const uint32_t bar0 = smem_addr(smem + SM::kBar) + warp * R * 8;  // this warp's barriers
  uint8_t* ring = smem + static_cast<size_t>(warp) * R * TL::kStage;  // this warp's stages

  if (threadIdx.x == 0) {
    ctl[0] = 0;
    ctl[1] = 0;
    ctl[2] = 0;
  }
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, blockIdx.x == 0 ? a.status : nullptr, lens,
            row_start);

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
      const int p = off - hh * npg;
      int page = __ldg(a.block_table + static_cast<long long>(i) * a.bt_stride + p);
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
      const uint32_t dst = smem_addr(ring + s * TL::kStage);
      const size_t unit = static_cast<size_t>(pg) * a.n_kv + hh;
      mbar_arrive_expect_tx(bar, TL::kStage);
      bulk_g2s(dst, a.k_data + unit * TL::kData, TL::kData, bar, policy);
      if constexpr (DT == PKV_KV_Q8_0)
        bulk_g2s(dst + TL::kData, a.k_scales + unit * TL::kScale, TL::kScale, bar, policy);
      bulk_g2s(dst + TL::kTile, a.v_data + unit * TL::kData, TL::kData, bar, policy);
      if constexpr (DT == PKV_KV_Q8_0)
        bulk_g2s(dst + TL::kTile + TL::kData, a.v_scales + unit * TL::kScale, TL::kScale, bar,
                 policy);
    }
    ++issued;
  };
  while (issued < n_units && issued < R) issue();

  const int tg = lane >> 3, dj = lane & 7;
  float* mrg_acc = reinterpret_cast<float*>(smem + SM::kMrgAcc);
  float* mrg_ml = reinterpret_cast<float*>(smem + SM::kMrgMl);
  float* prob = reinterpret_cast<float*>(smem + SM::kProb) + warp * SM::kProbPerWarp;
  float* alpha = reinterpret_cast<float*>(smem + SM::kAlpha) + warp * 4;
  const int g_lane = dj >> (3 - GR::kLog2);
  const bool head_writer = tg == 0 && (dj & (GR::kTokLanes - 1)) == 0 && (G > 1 || dj < 4);
  bool aborted = false;
  int consumed = 0;
  WarpState<G> S;

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
    const long long j = static_cast<long long>(i) * a.n_kv + h;
    const int k0 = chunk_of(seg_start, T, C), k1 = chunk_of(seg_end - 1, T, C);

    const float* qrow = a.q + (static_cast<long long>(i) * a.n_q + h * G) * kD;
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(qrow + g * kD + q_dim<DT>(dj, e)));
        S.q[g][e / 2] = make_float2(f.x * a.qscale, f.y * a.qscale);
        S.q[g][e / 2 + 1] = make_float2(f.z * a.qscale, f.w * a.qscale);
      }
      S.acc[g][0] = make_float2(0.f, 0.f);
      S.acc[g][1] = make_float2(0.f, 0.f);
    }
    S.m = -INFINITY;
    S.l = 0.f;

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
      const int nvalid = min(kPage, L - static_cast<int>(pos - seg_start) * kPage);
      process_unit<DT, G>(ring + s * TL::kStage, nvalid, lane, S, prob, alpha);
      if (issued < n_units) issue();
    }

    // ---- piece end: leave this warp's state in the shared merge buffer.
    // For every piece but the chunk's last, the last warp to arrive merges
    // while the others go on streaming; the chunk's last piece is merged by
    // the whole CTA, since all its warps are done by then.
    const float l_tot = head_sum<G>(S.l);
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
    if (head_writer) {
      mrg_ml[(warp * G + g_lane) * 2] = aborted ? -INFINITY : S.m;
      mrg_ml[(warp * G + g_lane) * 2 + 1] = l_tot;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
      *reinterpret_cast<float4*>(mrg_acc + (warp * G + g) * kD + lane * 4) =
          make_float4(S.acc[g][0].x, S.acc[g][0].y, S.acc[g][1].x, S.acc[g][1].y);
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
        merge_segment<G>(a.part_ml, a.part_acc, j, k0, k1, out_seg, d);
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
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, nullptr, lens, row_start);
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
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, nullptr, lens, row_start);
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
template <int DT, int G>
static cudaError_t launch_decode_t(const DecodeArgs& a, int chunks, cudaStream_t st) {
  const size_t smem = Smem<DT, G>::bytes(a.num_rows);
  cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<DT, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  paged_decode_kernel<DT, G><<<chunks, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int DT, int G>
static cudaError_t occupancy_t(int rows, int* blocks) {
  const size_t smem = Smem<DT, G>::bytes(rows);
  cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<DT, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
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
    } else {                                 \
      if ((G_) == 1) return CALL(1, 1);      \
      if ((G_) == 2) return CALL(1, 2);      \
      if ((G_) == 4) return CALL(1, 4);      \
    }                                        \
    return cudaErrorInvalidValue;            \
  } while (0)

cudaError_t launch_paged_decode(int dtype, int group, const DecodeArgs& a, int chunks,
                                cudaStream_t st) {
#define PKV_CALL(D, G) launch_decode_t<D, G>(a, chunks, st)
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

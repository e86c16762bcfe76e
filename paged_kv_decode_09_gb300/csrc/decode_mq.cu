// decode_mq.cu — paged decode attention with several queries per row: the
// verification step of speculative decoding and small chunks of chunked
// prefill (Leone, "What ships": chunked prefill, exact speculative
// verification; LeatEngine, "Capabilities": chunked prefill, speculative
// decoding).
//
// A row of L tokens whose last q_len are new has one query per new token:
// query j sits at position P = L - q_len + j and attends causally to
// [max(0, P + 1 - W), P + 1) under a window W (all of [0, P + 1) without
// one).  Every (row, KV head) page is read once per pass for all the pass's
// queries: a pass carries up to 8 (query, head) columns (f16, q8_0; 4 for
// bf16), so a step with q_len * G larger than that takes several passes over
// the same plan, each reading the pages again.  The new tokens are appended
// in the first pass, by the warp that reads their page, before its copy.
//
// The work split, the warps' rings, the tensor copies and the merges are the
// single-query kernel's (decode.cu); what differs is the page's MMA layout:
//   scores: S[16 tokens][cols] = K Q^T as there, with the columns split over
//     NT score n-tiles of 4 (query, head) columns x {hi, lo} parts; lane
//     4 gid + tig ends with the scores of columns tig and 4 + tig.
//   values: O^T[128 dims][cols] += V^T P^T with one B operand per part of P
//     (two MMAs into the same accumulator), so the 8 columns of an n-tile are
//     8 (query, head) pairs and O stays 32 registers a lane.
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
constexpr int mq_tiles() {
  return DT == PKV_KV_BF16 ? 1 : 2;
}

int mq_pass_queries(int dtype, int group) {
  const int cols = dtype == PKV_KV_BF16 ? 4 : 8;
  return cols / group > 0 ? cols / group : 1;
}

template <int DT>
struct MqSmem {
  static constexpr int kStages = kWarps * Tiles<DT>::kRing;
  static constexpr uint32_t kAlign = 1024;
  static constexpr uint32_t kScl = kStages * Tiles<DT>::kCodes;
  static constexpr uint32_t kBar = kScl + kStages * Tiles<DT>::kScales;
  static constexpr uint32_t kMrgAcc = kBar + ((kStages * 8 + 15) / 16) * 16;  // f32 [warps][8][D]
  static constexpr uint32_t kMrgMl = kMrgAcc + kWarps * kMqCols * kD * 4;      // f32 [warps][8][2]
  static constexpr uint32_t kCtl = kMrgMl + kWarps * kMqCols * 2 * 4;
  static constexpr uint32_t kRows = kCtl + 16;
  static size_t bytes(int rows) { return kAlign + kRows + (2 * static_cast<size_t>(rows) + 1) * 4; }
  static_assert(Tiles<DT>::kCodes % 1024 == 0, "tile stages keep the swizzle atom alignment");
};

template <int DT>
struct MqState {
  static constexpr int NT = mq_tiles<DT>();
  static constexpr int kSteps = DT == PKV_KV_BF16 ? 16 : 8;
  uint32_t qb[NT][kSteps][2];  // score B operands of n-tile t: column gid -> (4t + gid/2, part gid%2)
  float qexp[NT];              // 2^e of the lane's score column 4t + tig
  float m[NT], l[NT];          // softmax state of the lane's score columns
  float o[8][4];               // O^T: dims x V-columns 2tig (o[.][0, 2]) and 2tig + 1 (o[.][1, 3])
  int vx;                      // q8_0: bound on the piece's V block scales (as decode.cu)
};

template <int DT>
__device__ __forceinline__ float mq_o_scale(int vx) {
  if constexpr (DT == PKV_KV_F16)
    return 1.0f / (1 << kPShift);
  else if constexpr (DT == PKV_KV_BF16)
    return 1.0f;
  else
    return pow2i(vx - kPShift);
}

// Dim of O row r, element e (0: c0/c1, 2: c2/c3) in lane 4 gid + tig (as decode.cu).
template <int DT>
__device__ __forceinline__ int mq_dim(int r, int e, int gid) {
  if constexpr (DT != PKV_KV_Q8_0)
    return 16 * r + gid + (e ? 8 : 0);
  else
    return 16 * r + 2 * gid + (e ? 1 : 0);
}

// One column's query (qv, nullptr for an unused column) into the score B
// operands of the lane (part `lo`), with the dims mapping of the single-query
// kernel, normalised by a power of two per column (f16, q8_0).
template <int DT>
__device__ __forceinline__ void mq_load_column(const float* qv, float qscale, bool lo, int tig,
                                               uint32_t (&qb)[MqState<DT>::kSteps][2], int& e2) {
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
template <int DT>
__device__ __forceinline__ void mq_process_unit(uint8_t* st, const uint8_t* sc, int pf,
                                                const int (&col_lo)[2], const int (&col_hi)[2],
                                                int slot_lo, int slot_hi, int nc, int lane,
                                                MqState<DT>& S) {
  using TL = Tiles<DT>;
  constexpr int NT = MqState<DT>::NT;
  const int gid = lane >> 2, tig = lane & 3;
  const int ld_tok = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int ld_chunk = lane >> 4;
  const uint32_t kt = smem_addr(st), vt = kt + TL::kData;

  // ---- scores of the lane's columns 4t + tig, tokens gid and gid + 8
  float s[NT][2];
  if constexpr (DT == PKV_KV_BF16) {
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
      w0 ^= 0x80808080u;
      w1 ^= 0x80808080u;
      w2 ^= 0x80808080u;
      w3 ^= 0x80808080u;
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
    alpha[t] = grow ? exp2f(S.m[t] - mx) : 1.0f;
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
    p[t][0] = exp2f(s[t][0] - mu);
    p[t][1] = exp2f(s[t][1] - mu);
    S.l[t] += p[t][0] + p[t][1];
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
  if constexpr (DT != PKV_KV_Q8_0) {
    if (slot_lo > 0 || slot_hi < kPage) {  // zero the V rows of slots no column attends
      const int n_out = kPage - (slot_hi - slot_lo);
      for (int x = lane; x < n_out * 16; x += 32) {
        const int r = x >> 4, tt = r < slot_lo ? r : slot_hi + (r - slot_lo), c = x & 15;
        *reinterpret_cast<uint4*>(st + TL::kData + (c >> 3) * 2048 + tt * 128 + (c & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
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
        const uint32_t x0 = w0 << 16, x1 = w2 << 16, x2 = w0 & 0xffff0000u, x3 = w2 & 0xffff0000u;
        const uint32_t y0 = w1 << 16, y1 = w3 << 16, y2 = w1 & 0xffff0000u, y3 = w3 & 0xffff0000u;
        mma_1688_tf32(S.o[mt], x0, x1, x2, x3, h0, h1);
        mma_1688_tf32(S.o[mt], x0, x1, x2, x3, l0, l1);
        mma_1688_tf32(S.o[mt], y0, y1, y2, y3, h8, h9);
        mma_1688_tf32(S.o[mt], y0, y1, y2, y3, l8, l9);
      }
    }
  } else {
    uint4 va = *reinterpret_cast<const uint4*>(sc + TL::kScale + t0 * 8);
    uint4 vb = *reinterpret_cast<const uint4*>(sc + TL::kScale + (t0 + 8) * 8);
    if (slot_lo > 0 || slot_hi < kPage) {  // unattended slots: P = 0, scales may be NaN
      if (t0 < slot_lo || t0 >= slot_hi) va.x = va.y = 0u;
      if (t0 + 1 < slot_lo || t0 + 1 >= slot_hi) va.z = va.w = 0u;
      if (t0 + 8 < slot_lo || t0 + 8 >= slot_hi) vb.x = vb.y = 0u;
      if (t0 + 9 < slot_lo || t0 + 9 >= slot_hi) vb.z = vb.w = 0u;
    }
    uint32_t mb = __vmaxu2(__vmaxu2(va.x & 0x7fff7fffu, va.y & 0x7fff7fffu),
                           __vmaxu2(va.z & 0x7fff7fffu, va.w & 0x7fff7fffu));
    mb = __vmaxu2(mb, __vmaxu2(__vmaxu2(vb.x & 0x7fff7fffu, vb.y & 0x7fff7fffu),
                               __vmaxu2(vb.z & 0x7fff7fffu, vb.w & 0x7fff7fffu)));
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
      w0 ^= 0x80808080u;
      w1 ^= 0x80808080u;
      w2 ^= 0x80808080u;
      w3 ^= 0x80808080u;
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

// Merge the pieces k0..k1 of segment j (slots k + j, kMqCols columns each),
// one warp, lane l: dims 4l..4l+3; column c of the pass goes to out_col(c).
template <class OutCol>
__device__ __forceinline__ void mq_merge_segment_warp(const float* part_ml, const float* part_acc,
                                                      long long j, int k0, int k1, int nc,
                                                      OutCol&& out_col, int lane) {
  for (int c = 0; c < nc; ++c) {
    float M = -INFINITY, Ls = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int kk = k0; kk <= k1; ++kk) {
      const long long slot = (kk + j) * kMqCols + c;
      const float m = __ldcg(part_ml + slot * 2), l = __ldcg(part_ml + slot * 2 + 1);
      const float4 x = __ldcg(reinterpret_cast<const float4*>(part_acc + slot * kD) + lane);
      const float bm = fmaxf(M, m);
      if (bm == -INFINITY) continue;  // no token of this query in either
      const float f0 = exp2f(M - bm), f1 = exp2f(m - bm);
      Ls = Ls * f0 + l * f1;
      A = make_float4(A.x * f0 + x.x * f1, A.y * f0 + x.y * f1, A.z * f0 + x.z * f1,
                      A.w * f0 + x.w * f1);
      M = bm;
    }
    const float inv = 1.0f / Ls;
    *reinterpret_cast<float4*>(out_col(c) + lane * 4) =
        make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
  }
}

// --------------------------------------------------------------- kernel ----
template <int DT, int G>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_mq_kernel(const __grid_constant__ DecodeArgs a,
                           const __grid_constant__ TileMaps maps) {
  using TL = Tiles<DT>;
  using SM = MqSmem<DT>;
  constexpr int R = TL::kRing;
  constexpr int NT = MqState<DT>::NT;
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
  const int nc = a.nq * G;  // columns of this pass
  // the pages read cover the first query's window: [L - q_len + 1 - W, L)
  const int plan_window = a.window > 0 ? a.window + a.q_len - 1 : 0;

  if (threadIdx.x == 0) {
    ctl[0] = 0;
    ctl[1] = 0;
    ctl[2] = 0;
  }
  if (lane == 0) {
    for (int s = 0; s < R; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  plan_rows(a.seq_lens, a.num_rows, a.bt_stride, plan_window,
            blockIdx.x == 0 ? a.status : nullptr, lens, row_start, a.q_len);

  const long long T = static_cast<long long>(a.n_kv) * row_start[a.num_rows];
  const int C = used_chunks(T, gridDim.x), k = blockIdx.x;
  const long long c_begin = k < C ? static_cast<long long>(k) * T / C : T;
  const long long c_end = k < C ? static_cast<long long>(k + 1) * T / C : T;

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
  fetch(32, n_pg, n_h, n_row, n_p);
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

  float* mrg_acc = reinterpret_cast<float*>(smem + SM::kMrgAcc);
  float* mrg_ml = reinterpret_cast<float*>(smem + SM::kMrgMl);
  bool aborted = false;
  int consumed = 0;
  MqState<DT> S;

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
    const int p0 = window_start(L, plan_window) / kPage;
    const long long j = static_cast<long long>(i) * a.n_kv + h;
    const int k0 = chunk_of(seg_start, T, C), k1 = chunk_of(seg_end - 1, T, C);

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
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int cq = 4 * t + (gid >> 1);  // the column whose query this lane loads
      const float* qv = cq < nc
                            ? a.q + ((static_cast<long long>(i) * a.q_len + a.q0 + cq / G) * a.n_q +
                                     h * G + cq % G) * kD
                            : nullptr;
      int e2;
      mq_load_column<DT>(qv, a.qscale, (gid & 1) != 0, tig, S.qb[t], e2);
      S.qexp[t] = ldexpf(1.0f, __shfl_sync(kFull, e2, 8 * tig));  // lane 8 tig loads column 4t + tig
      S.m[t] = -INFINITY;
      S.l[t] = 0.f;
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
      mq_process_unit<DT>(ring + s * TL::kCodes, ring_sc + s * TL::kScales, pf, col_lo, col_hi,
                          slot_lo, slot_hi, nc, lane, S);
      if (issued < n_units) issue();
    }

    // ---- piece end (as the single-query kernel, kMqCols columns)
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
        mrg_ml[(warp * kMqCols + c) * 2] = aborted ? -INFINITY : S.m[t];
        mrg_ml[(warp * kMqCols + c) * 2 + 1] = l_tot[t];
      }
    }
    {
      const float osc = mq_o_scale<DT>(S.vx);
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 2 * tig + (e & 1);
          mrg_acc[(warp * kMqCols + c) * kD + mq_dim<DT>(r, e & 2, gid)] = S.o[r][e] * osc;
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
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mrg_ml[(w * kMqCols + c) * 2]);
      Ls = 0.f;
      A = 0.f;
      if (M == -INFINITY) return;  // no token of this query in the piece
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(mrg_ml[(w * kMqCols + c) * 2] - M);
        Ls = fmaf(f, mrg_ml[(w * kMqCols + c) * 2 + 1], Ls);
        A = fmaf(f, mrg_acc[(w * kMqCols + c) * kD + d], A);
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
      const bool counted = live && !whole && a.counters != nullptr;
      named_barrier(1, kThreads);
      if (threadIdx.x == 0) {
        int seg_last = 0;
        if (counted) {
          __threadfence();
          seg_last = atomicAdd(a.counters + j, 1) == k1 - k0;
        }
        ctl[1] = seg_last;
      }
      named_barrier(1, kThreads);
      if (ctl[1] && warp == 0) {
        __threadfence();
        mq_merge_segment_warp(a.part_ml, a.part_acc, j, k0, k1, nc, out_col, lane);
        if (lane == 0) a.counters[j] = 0;
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
        if (live && !whole && a.counters != nullptr) {
          __syncwarp();
          int seg_last = 0;
          if (lane == 0) {
            __threadfence();
            seg_last = atomicAdd(a.counters + j, 1) == k1 - k0;
          }
          seg_last = __shfl_sync(kFull, seg_last, 0);
          if (seg_last) {
            __threadfence();
            mq_merge_segment_warp(a.part_ml, a.part_acc, j, k0, k1, nc, out_col, lane);
            if (lane == 0) a.counters[j] = 0;
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

// ------------------------------------------------------------ launchers ----
template <int DT, int G>
static cudaError_t mq_ensure_smem(size_t smem) {
  static std::atomic<size_t> granted[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && granted[dev].load(std::memory_order_relaxed) >= smem)
    return cudaSuccess;
  e = cudaFuncSetAttribute(paged_decode_mq_kernel<DT, G>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess && dev >= 0 && dev < 64) {
    size_t cur = granted[dev].load();
    while (cur < smem && !granted[dev].compare_exchange_weak(cur, smem)) {
    }
  }
  return e;
}

template <int DT, int G>
static cudaError_t launch_mq_t(const DecodeArgs& a, const TileMaps& maps, int chunks,
                               cudaStream_t st) {
  const size_t smem = MqSmem<DT>::bytes(a.num_rows);
  cudaError_t e = mq_ensure_smem<DT, G>(smem);
  if (e != cudaSuccess) return e;
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
  e = cudaLaunchKernelEx(&cfg, paged_decode_mq_kernel<DT, G>, a, maps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DT>
static cudaError_t mq_occupancy_t(int rows, int* blocks) {
  const size_t smem = MqSmem<DT>::bytes(rows);
  cudaError_t e = mq_ensure_smem<DT, 4>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, paged_decode_mq_kernel<DT, 4>,
                                                       kThreads, smem);
}

cudaError_t launch_paged_decode_mq(int dtype, int group, const DecodeArgs& a, const TileMaps& maps,
                                   int chunks, cudaStream_t st) {
#define PKV_MQ(D, G_)                                   \
  if (group == (G_)) return launch_mq_t<D, G_>(a, maps, chunks, st)
  if (dtype == PKV_KV_F16) {
    PKV_MQ(PKV_KV_F16, 1);
    PKV_MQ(PKV_KV_F16, 2);
    PKV_MQ(PKV_KV_F16, 4);
  } else if (dtype == PKV_KV_BF16) {
    PKV_MQ(PKV_KV_BF16, 1);
    PKV_MQ(PKV_KV_BF16, 2);
    PKV_MQ(PKV_KV_BF16, 4);
  } else {
    PKV_MQ(PKV_KV_Q8_0, 1);
    PKV_MQ(PKV_KV_Q8_0, 2);
    PKV_MQ(PKV_KV_Q8_0, 4);
  }
#undef PKV_MQ
  return cudaErrorInvalidValue;
}

cudaError_t paged_decode_mq_blocks_per_sm(int dtype, int rows, int* blocks) {
  if (dtype == PKV_KV_F16) return mq_occupancy_t<PKV_KV_F16>(rows, blocks);
  if (dtype == PKV_KV_BF16) return mq_occupancy_t<PKV_KV_BF16>(rows, blocks);
  return mq_occupancy_t<PKV_KV_Q8_0>(rows, blocks);
}

}  // namespace pkv

// append.cu — kv_append: store each row's new K and V token into its page
// slot (tinyllm, "The repository currently provides": per-sequence block
// tables into a physical page pool; Leone, "What ships" and LeatEngine, "Run":
// f16 and q8_0 KV storage).
//
// Row i with L = seq_lens[i] >= 1 writes position L - 1: page
// block_table[i][(L-1)/16], slot (L-1) % 16.  One CTA per (row, KV head), one
// thread per dim; K and V in turn.
//   f16 : binary16 rounded to nearest even.
//   bf16: bfloat16 rounded to nearest even.
//   f32 : the fp32 value itself.
//   q8_0: each warp holds one 32-wide block: amax by warp reduction,
//         d = amax / 127 (IEEE division), codes round(x / d) with ties away
//         from zero (roundf), stored scale binary16(d); amax = 0 gives zeros.
#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

template <int DT>
__global__ void __launch_bounds__(kD) append_kernel(const AppendArgs a) {
  const int i = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int L = a.seq_lens[i];
  if (L <= 0) return;
  if (L > a.bt_stride * kPage) {
    if (d == 0 && h == 0) record_status(a.status, PKV_DEV_BAD_LENGTH);
    return;
  }
  const int pos = L - 1;
  const int page = a.block_table[static_cast<long long>(i) * a.bt_stride + pos / kPage];
  if (page < 0 || page >= a.num_pages) {
    if (d == 0 && h == 0) record_status(a.status, PKV_DEV_BAD_PAGE);
    return;
  }
  const long long slot_row = (static_cast<long long>(page) * a.n_kv + h) * kPage + pos % kPage;
  const long long src = (static_cast<long long>(i) * a.n_kv + h) * kD + d;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const float x = which == 0 ? a.k_new[src] : a.v_new[src];
    uint8_t* data = which == 0 ? a.k_data : a.v_data;
    if constexpr (DT == PKV_KV_F16) {
      reinterpret_cast<__half*>(data)[slot_row * kD + d] = __float2half_rn(x);
    } else if constexpr (DT == PKV_KV_BF16) {
      reinterpret_cast<__nv_bfloat16*>(data)[slot_row * kD + d] = __float2bfloat16_rn(x);
    } else if constexpr (DT == PKV_KV_F32) {
      reinterpret_cast<float*>(data)[slot_row * kD + d] = x;
    } else {
      float amax = fabsf(x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      const float dq = amax / 127.0f;  // IEEE division (no fast-math in this build)
      float c = 0.0f;
      if (dq != 0.0f) c = fminf(fmaxf(roundf(x / dq), -127.0f), 127.0f);
      // stored offset-binary: code + 128 (the int8 code with its top bit flipped)
      data[slot_row * kD + d] = static_cast<uint8_t>(static_cast<int>(c) + 128);
      if ((d & 31) == 0) {
        uint8_t* sc = which == 0 ? a.k_scales : a.v_scales;
        reinterpret_cast<__half*>(sc)[slot_row * (kD / kQBlock) + d / kQBlock] =
            __float2half_rn(dq);
      }
    }
  }
}

cudaError_t launch_append(int dtype, const AppendArgs& a, cudaStream_t st) {
  if (a.num_rows == 0) return cudaSuccess;
  const dim3 grid(a.num_rows, a.n_kv);
  if (dtype == PKV_KV_F16)
    append_kernel<PKV_KV_F16><<<grid, kD, 0, st>>>(a);
  else if (dtype == PKV_KV_BF16)
    append_kernel<PKV_KV_BF16><<<grid, kD, 0, st>>>(a);
  else if (dtype == PKV_KV_F32)
    append_kernel<PKV_KV_F32><<<grid, kD, 0, st>>>(a);
  else
    append_kernel<PKV_KV_Q8_0><<<grid, kD, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv

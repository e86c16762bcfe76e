// pkv_internal.h — argument blocks and launchers shared between the C-ABI
// layer (api.cu) and the kernel files (append.cu, decode.cu).  Not installed.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// Arguments of the split-KV decode kernel.  Pool pointers already point at
// the layer's arrays.
struct DecodeArgs {
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_scales;  // q8_0 only
  uint8_t* v_scales;  // q8_0 only
  const float* k_new;  // non-null: append each row's new token first (fused step)
  const float* v_new;
  int num_pages;
  int n_kv;
  const float* q;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;
  int num_rows;
  int n_q;
  float qscale;  // softmax scale * log2(e): scores are kept in base 2
  int window;    // > 0: each row attends to its last `window` tokens
  int q_len;     // queries (new tokens) per row; q, out [rows][q_len][n_q][128]
  int q0, nq;    // several-query kernel: this pass's queries q0 .. q0 + nq - 1
  int vchunks;   // chunks of the work split (several-query kernels: a CTA may hold 2)
  int aligned_split;  // 1: the split may align chunks to segments (single-query kernel)
  float* out;
  float* part_ml;   // [slots][G][2]
  float* part_acc;  // [slots][G][128]
  // Non-null: merge in-kernel, and the end of the workspace.  The merge's
  // flags sit below it at places that do not depend on the call's rows or
  // chunks (see flag_bytes): the arrival counter of segment j at flags[-1 - 2j]
  // and the ready flag of partial slot s at flags[-2 - 2s] (single-query
  // kernel); the counter of (segment j, column group w) at
  // flags[-1 - (kMqCounters j + w)] (several-query kernels).
  int32_t* flags;
  int32_t* status;  // optional device status word
  unsigned long long test_stall_ns;  // test hook (kv_pool_set_test_stall); 0: off
};

struct CombineArgs {
  const int32_t* seq_lens;
  int window;
  int num_rows;
  int n_q;
  int n_kv;
  int bt_stride;
  int num_chunks;
  int aligned_split;  // the attention call's split (see DecodeArgs)
  const float* part_ml;
  const float* part_acc;
  float* out;
};

struct PlanArgs {
  const int32_t* seq_lens;
  int window;
  int num_rows;
  int n_kv;
  int bt_stride;
  int num_chunks;
  int aligned_split;
  int32_t* row_page_start;
  int32_t* seg_first_chunk;
  int32_t* seg_last_chunk;
};

struct AppendArgs {
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_scales;
  uint8_t* v_scales;
  int num_pages;
  int n_kv;
  const float* k_new;
  const float* v_new;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;
  int num_rows;
  int32_t* status;
};

// Workspace layout (see paged_decode_workspace_bytes): the partial states
// from the start (part_ml, then part_acc), and the merge's int32 flags down
// from the end.  The flags of a segment or slot keep their place whatever
// the call's shape, so a workspace sized for the largest call serves calls of
// any smaller shape: no call's partial states land on another call's flags.
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
// ints of a single-query CTA's plan in shared memory: row_start[rows + 1],
// lens[rows] and the chunks before each row pc[rows + 1]
inline size_t plan_ints(int rows) { return 3 * static_cast<size_t>(rows) + 2; }
// the single-query flags of a call with `slots` partial slots (segments <=
// slots): a counter and a ready flag interleaved per index
inline size_t flag_bytes(long long slots) {
  return align256(static_cast<size_t>(slots) * 2 * sizeof(int32_t));
}
// the end of a workspace of `bytes` bytes, where the flags start (downwards)
inline int32_t* flags_end(void* ws, size_t bytes) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + (bytes & ~size_t(255)));
}
inline size_t part_ml_bytes(long long slots, int group) {
  return align256(static_cast<size_t>(slots) * group * 2 * sizeof(float));
}
inline size_t part_acc_bytes(long long slots, int group) {
  return align256(static_cast<size_t>(slots) * group * PKV_HEAD_DIM * sizeof(float));
}

// Helpers the C-ABI layer exports to the other translation units.
int pool_kv_heads(const pkv_pool* pool);                 // n_kv_heads of a pool descriptor
// The host-side checks of paged_decode_attention's arguments other than the
// workspace (PKV_OK, or the status that call would return).
pkv_status check_attention_args(const pkv_pool* pool, int layer, const float* q,
                                const int32_t* block_table, int bt_stride,
                                const int32_t* seq_lens, int num_rows, int n_q_heads,
                                const float* out, int num_chunks);
pkv_status record_error(pkv_status s, const char* msg);  // sets pkv_last_error_message

// Tensor maps of one layer's K and V data, [tiles][16 tokens][128 dims]
// under the 128-byte swizzle (encoded once per layer when a pool is created).
struct TileMaps {
  CUtensorMap k;
  CUtensorMap v;
  // 16-bit formats also: a tile as [2 token groups][2 halves][8 tokens][64
  // dims], one copy per tile (the tensor-core several-query kernel)
  CUtensorMap kp;
  CUtensorMap vp;
};
cudaError_t encode_tile_maps(int dtype, void* k_data, void* v_data, long long tiles,
                             TileMaps* maps);

cudaError_t launch_paged_decode(int dtype, int group, const DecodeArgs& a, const TileMaps& maps,
                                int chunks, cudaStream_t stream);
cudaError_t paged_decode_blocks_per_sm(int dtype, int group, int rows, int* blocks);
// The several-query kernels: one pass of up to mq_pass_queries(dtype, group,
// q_len) queries (a.q0, a.nq) over the same plan; the kernel is chosen by
// q_len * group (the same for every pass of a call).
int mq_pass_queries(int dtype, int group, int q_len, int rows);
cudaError_t launch_paged_decode_mq(int dtype, int group, const DecodeArgs& a, const TileMaps& maps,
                                   int chunks, cudaStream_t stream);
cudaError_t paged_decode_mq_blocks_per_sm(int dtype, int group, int q_len, int rows, int* blocks);
// The tensor-core several-query kernel (f16 and bf16 KV, passes of up to 32
// columns).
cudaError_t launch_paged_decode_mqtc(int dtype, const DecodeArgs& a, const TileMaps& maps,
                                     int chunks, cudaStream_t stream);
cudaError_t paged_decode_mqtc_blocks_per_sm(int dtype, int rows, int* blocks);
int paged_decode_mqtc_max_rows(int dtype);  // rows per call the tensor-core kernel takes
constexpr int kMqCols = 32;  // partial-state columns of a several-query workspace slot
constexpr int kMqCounters = 4;  // arrival counters per (row, KV head): one per warp's columns
inline size_t mq_flag_bytes(long long segments) {
  return align256(static_cast<size_t>(segments) * kMqCounters * sizeof(int32_t));
}
cudaError_t launch_combine(int group, const CombineArgs& a, cudaStream_t stream);
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);
cudaError_t launch_append(int dtype, const AppendArgs& a, cudaStream_t stream);

}  // namespace pkv

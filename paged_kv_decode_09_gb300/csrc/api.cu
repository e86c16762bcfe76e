// api.cu — the C ABI of libpkv.so (declared in include/pkv.h): host-side
// validation, the pool descriptor, and the kernel launches.  Nothing here
// allocates device memory or synchronises a stream, except
// kv_pool_read_status, which is documented to.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>

#include "pkv.h"
#include "pkv_internal.h"

struct pkv_pool {
  int num_layers;
  int num_pages;
  int n_kv;
  int head_dim;
  pkv_kv_dtype dtype;
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_scales;
  uint8_t* v_scales;
  int32_t* status;
  size_t layer_data_bytes;
  size_t layer_scale_bytes;
  // Per layer, the tensor maps through which the attention kernel reads the
  // K and V tiles: encoded on the layer's first attention call (host only),
  // so that creating a descriptor needs no driver.
  pkv::TileMaps* maps;       // [num_layers]
  std::atomic<int>* ready;   // [num_layers]: 1 once maps[layer] is valid
  std::mutex maps_mutex;
  int* window;               // [num_layers]: sliding window of the layer (0: none)
  unsigned long long test_stall_ns = 0;  // test hook (kv_pool_set_test_stall); 0: off
  ~pkv_pool() {
    delete[] maps;
    delete[] ready;
    delete[] window;
  }
};

namespace {

thread_local char g_last_error[256] = "";

pkv_status fail(pkv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

size_t data_bytes_per_layer(int num_pages, int n_kv, int head_dim, pkv_kv_dtype dtype) {
  const size_t elems = static_cast<size_t>(num_pages) * n_kv * PKV_PAGE_TOKENS * head_dim;
  return dtype == PKV_KV_Q8_0 ? elems : dtype == PKV_KV_F32 ? elems * 4 : elems * 2;  // f16, bf16: 2
}

size_t scale_bytes_per_layer(int num_pages, int n_kv, int head_dim, pkv_kv_dtype dtype) {
  if (dtype != PKV_KV_Q8_0) return 0;
  return static_cast<size_t>(num_pages) * n_kv * PKV_PAGE_TOKENS * (head_dim / PKV_Q8_BLOCK) * 2;
}

pkv_status check_geometry(int n_q, int n_kv, int head_dim) {
  if (n_kv <= 0 || n_q <= 0) return fail(PKV_ERR_INVALID_ARG, "head counts must be positive");
  if (n_q % n_kv) return fail(PKV_ERR_INVALID_ARG, "n_q_heads %% n_kv_heads != 0");
  const int g = n_q / n_kv;
  if (g != 1 && g != 2 && g != 4)
    return fail(PKV_ERR_UNSUPPORTED, "GQA group %d not in {1,2,4}", g);
  if (head_dim != PKV_HEAD_DIM) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d != 128", head_dim);
  return PKV_OK;
}

bool known_dtype(pkv_kv_dtype d) {
  return d == PKV_KV_F16 || d == PKV_KV_Q8_0 || d == PKV_KV_BF16 || d == PKV_KV_F32;
}

// Whether the single-query split may align its chunks to segments for this
// KV format: the 16-bit formats.  q8_0 chunks finish by launch order
// (instruction issue), not by the pieces they hold, and f32 chunks are twice
// as long, so for both equal chunks serve better.
int split_may_align(pkv_kv_dtype d) { return d == PKV_KV_F16 || d == PKV_KV_BF16; }

pkv_status check_rows(int num_rows, int bt_stride, const int32_t* bt, const int32_t* sl,
                      int max_rows = PKV_MAX_ROWS) {
  if (num_rows < 0) return fail(PKV_ERR_INVALID_ARG, "num_rows < 0");
  if (num_rows > max_rows)
    return fail(PKV_ERR_UNSUPPORTED, "num_rows %d > %d", num_rows, max_rows);
  if (num_rows > 0 && (!bt || !sl)) return fail(PKV_ERR_INVALID_ARG, "null block table or seq_lens");
  if (bt_stride < 1) return fail(PKV_ERR_INVALID_ARG, "bt_stride < 1");
  if (!aligned(bt, 4) || !aligned(sl, 4))
    return fail(PKV_ERR_INVALID_ARG, "block table / seq_lens not 4-byte aligned");
  return PKV_OK;
}

pkv_status check_pool_layer(const pkv_pool* p, int layer) {
  if (!p) return fail(PKV_ERR_INVALID_ARG, "null pool");
  if (layer < 0 || layer >= p->num_layers)
    return fail(PKV_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, p->num_layers);
  return PKV_OK;
}

long long partial_slots(int num_chunks, int num_rows, int n_kv) {
  return static_cast<long long>(num_chunks) + static_cast<long long>(num_rows) * n_kv;
}

size_t workspace_needed(int num_rows, int n_q, int n_kv, int num_chunks) {
  const long long slots = partial_slots(num_chunks, num_rows, n_kv);
  const int g = n_q / n_kv;
  return pkv::part_ml_bytes(slots, g) + pkv::part_acc_bytes(slots, g) + pkv::flag_bytes(slots);
}

// Workspace parts for a call: part_ml, part_acc, and the end the flags hang from.
struct WsParts {
  float* part_ml;
  float* part_acc;
  int32_t* flags;
};
WsParts workspace_parts(void* ws, size_t bytes, int num_rows, int n_q, int n_kv, int num_chunks) {
  const long long slots = partial_slots(num_chunks, num_rows, n_kv);
  uint8_t* p = static_cast<uint8_t*>(ws);
  WsParts w;
  w.part_ml = reinterpret_cast<float*>(p);
  p += pkv::part_ml_bytes(slots, n_q / n_kv);
  w.part_acc = reinterpret_cast<float*>(p);
  w.flags = pkv::flags_end(ws, bytes);
  return w;
}

pkv_status default_chunks(const pkv_pool* p, int n_q, int rows, int* chunks) {
  int dev = 0, sms = 0, blocks = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  e = pkv::paged_decode_blocks_per_sm(p->dtype, n_q / p->n_kv, rows, &blocks);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  if (blocks < 1) return fail(PKV_ERR_UNSUPPORTED, "attention kernel does not fit on an SM");
  *chunks = sms * blocks;
  return PKV_OK;
}

// The layer's tensor maps, encoded on first use.
pkv_status layer_maps(const pkv_pool* pool, int layer, const pkv::TileMaps** maps) {
  pkv_pool* p = const_cast<pkv_pool*>(pool);
  if (!p->ready[layer].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(p->maps_mutex);
    if (!p->ready[layer].load(std::memory_order_relaxed)) {
      const cudaError_t e = pkv::encode_tile_maps(
          p->dtype, p->k_data + layer * p->layer_data_bytes, p->v_data + layer * p->layer_data_bytes,
          static_cast<long long>(p->num_pages) * p->n_kv, &p->maps[layer]);
      if (e != cudaSuccess) return cuda_fail(e, "tensor maps of the pool layer");
      p->ready[layer].store(1, std::memory_order_release);
    }
  }
  *maps = &p->maps[layer];
  return PKV_OK;
}

enum class Mode { kMerged, kSplitOnly };

// One launch of the decode kernel: kMerged merges split segments in-kernel
// (arrival counters) and, given k_new/v_new, appends the new tokens first;
// kSplitOnly leaves the partial states for paged_decode_combine.
// The checks of an attention call's arguments other than the workspace.
pkv_status check_attention(const pkv_pool* pool, int layer, const float* q,
                           const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                           int num_rows, int n_q, const float* out, int num_chunks) {
  pkv_status s = check_pool_layer(pool, layer);
  if (s) return s;
  if ((s = check_geometry(n_q, pool->n_kv, pool->head_dim))) return s;
  if ((s = check_rows(num_rows, bt_stride, block_table, seq_lens))) return s;
  if (num_rows > 0 && (!q || !out)) return fail(PKV_ERR_INVALID_ARG, "null q or out");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(PKV_ERR_INVALID_ARG, "q / out not 16-byte aligned");
  if (num_chunks < 0) return fail(PKV_ERR_INVALID_ARG, "num_chunks < 0");
  if (num_chunks > PKV_MAX_CHUNKS) return fail(PKV_ERR_UNSUPPORTED, "num_chunks > %d", PKV_MAX_CHUNKS);
  return PKV_OK;
}

pkv_status attention_impl(const pkv_pool* pool, int layer, const float* q, const float* k_new,
                          const float* v_new, const int32_t* block_table, int bt_stride,
                          const int32_t* seq_lens, int num_rows, int n_q, float scale, float* out,
                          void* workspace, size_t workspace_bytes, int num_chunks, void* stream,
                          Mode mode) {
  pkv_status s =
      check_attention(pool, layer, q, block_table, bt_stride, seq_lens, num_rows, n_q, out, num_chunks);
  if (s) return s;
  if (num_rows == 0) return PKV_OK;
  if (num_chunks == 0 && (s = default_chunks(pool, n_q, num_rows, &num_chunks))) return s;
  const size_t need = workspace_needed(num_rows, n_q, pool->n_kv, num_chunks);
  if (!workspace || workspace_bytes < need)
    return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace not 256-byte aligned");

  const int g = n_q / pool->n_kv;
  const WsParts w = workspace_parts(workspace, workspace_bytes, num_rows, n_q, pool->n_kv, num_chunks);
  pkv::DecodeArgs a;
  a.k_data = pool->k_data + layer * pool->layer_data_bytes;
  a.v_data = pool->v_data + layer * pool->layer_data_bytes;
  a.k_scales = pool->k_scales ? pool->k_scales + layer * pool->layer_scale_bytes : nullptr;
  a.v_scales = pool->v_scales ? pool->v_scales + layer * pool->layer_scale_bytes : nullptr;
  a.k_new = mode == Mode::kMerged ? k_new : nullptr;
  a.v_new = mode == Mode::kMerged ? v_new : nullptr;
  a.num_pages = pool->num_pages;
  a.n_kv = pool->n_kv;
  a.q = q;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.num_rows = num_rows;
  a.n_q = n_q;
  a.qscale = scale * 1.4426950408889634f;  // log2(e): base-2 softmax
  a.window = pool->window[layer];
  a.q_len = 1;
  a.q0 = 0;
  a.nq = 1;
  a.vchunks = num_chunks;
  a.aligned_split = split_may_align(pool->dtype);
  a.out = out;
  a.part_ml = w.part_ml;
  a.part_acc = w.part_acc;
  a.flags = mode == Mode::kMerged ? w.flags : nullptr;
  a.status = pool->status;
  a.test_stall_ns = pool->test_stall_ns;
  const pkv::TileMaps* maps = nullptr;
  if ((s = layer_maps(pool, layer, &maps))) return s;
  cudaError_t e = pkv::launch_paged_decode(pool->dtype, g, a, *maps, num_chunks,
                                           as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged decode launch");
  return PKV_OK;
}


// ------------------------------------------------- several queries per row
size_t workspace_needed_mq(int num_rows, int n_kv, int num_chunks) {
  const long long slots = partial_slots(num_chunks, num_rows, n_kv);
  return pkv::part_ml_bytes(slots, pkv::kMqCols) + pkv::part_acc_bytes(slots, pkv::kMqCols) +
         pkv::mq_flag_bytes(static_cast<long long>(num_rows) * n_kv);
}

pkv_status default_chunks_mq(const pkv_pool* p, int group, int q_len, int rows, int* chunks) {
  int dev = 0, sms = 0, blocks = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  e = pkv::paged_decode_mq_blocks_per_sm(p->dtype, group, q_len, rows, &blocks);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  if (blocks < 1) return fail(PKV_ERR_UNSUPPORTED, "attention kernel does not fit on an SM");
  *chunks = sms * blocks;
  return PKV_OK;
}

// ceil(q_len * G / columns) launches over the same plan; the first appends.
pkv_status attention_mq_impl(const pkv_pool* pool, int layer, const float* q, const float* k_new,
                             const float* v_new, const int32_t* block_table, int bt_stride,
                             const int32_t* seq_lens, int num_rows, int q_len, int n_q,
                             float scale, float* out, void* workspace, size_t workspace_bytes,
                             int num_chunks, void* stream) {
  pkv_status s = check_pool_layer(pool, layer);
  if (s) return s;
  if ((s = check_geometry(n_q, pool->n_kv, pool->head_dim))) return s;
  if ((s = check_rows(num_rows, bt_stride, block_table, seq_lens))) return s;
  if (q_len < 1 || q_len > PKV_MAX_Q_LEN)
    return fail(PKV_ERR_UNSUPPORTED, "q_len %d outside [1, %d]", q_len, PKV_MAX_Q_LEN);
  if (num_rows > 0 && (!q || !out)) return fail(PKV_ERR_INVALID_ARG, "null q or out");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(PKV_ERR_INVALID_ARG, "q / out not 16-byte aligned");
  if (num_chunks < 0) return fail(PKV_ERR_INVALID_ARG, "num_chunks < 0");
  if (num_chunks > PKV_MAX_CHUNKS) return fail(PKV_ERR_UNSUPPORTED, "num_chunks > %d", PKV_MAX_CHUNKS);
  if (num_rows == 0) return PKV_OK;
  const int g = n_q / pool->n_kv;
  if (num_chunks == 0 && (s = default_chunks_mq(pool, g, q_len, num_rows, &num_chunks))) return s;
  const size_t need = workspace_needed_mq(num_rows, pool->n_kv, num_chunks);
  if (!workspace || workspace_bytes < need)
    return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace not 256-byte aligned");

  const long long slots = partial_slots(num_chunks, num_rows, pool->n_kv);
  uint8_t* wp = static_cast<uint8_t*>(workspace);
  pkv::DecodeArgs a;
  a.flags = pkv::flags_end(workspace, workspace_bytes);
  a.part_ml = reinterpret_cast<float*>(wp);
  wp += pkv::part_ml_bytes(slots, pkv::kMqCols);
  a.part_acc = reinterpret_cast<float*>(wp);
  a.k_data = pool->k_data + layer * pool->layer_data_bytes;
  a.v_data = pool->v_data + layer * pool->layer_data_bytes;
  a.k_scales = pool->k_scales ? pool->k_scales + layer * pool->layer_scale_bytes : nullptr;
  a.v_scales = pool->v_scales ? pool->v_scales + layer * pool->layer_scale_bytes : nullptr;
  a.num_pages = pool->num_pages;
  a.n_kv = pool->n_kv;
  a.q = q;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.num_rows = num_rows;
  a.n_q = n_q;
  a.qscale = scale * 1.4426950408889634f;  // log2(e): base-2 softmax
  a.window = pool->window[layer];
  a.q_len = q_len;
  a.vchunks = num_chunks;
  a.aligned_split = split_may_align(pool->dtype);
  a.out = out;
  a.status = pool->status;
  a.test_stall_ns = pool->test_stall_ns;
  const pkv::TileMaps* maps = nullptr;
  if ((s = layer_maps(pool, layer, &maps))) return s;
  const int per_pass = pkv::mq_pass_queries(pool->dtype, g, q_len, num_rows);
  for (int q0 = 0; q0 < q_len; q0 += per_pass) {
    a.q0 = q0;
    a.nq = q_len - q0 < per_pass ? q_len - q0 : per_pass;
    a.k_new = q0 == 0 ? k_new : nullptr;  // the new tokens are stored once, in the first pass
    a.v_new = q0 == 0 ? v_new : nullptr;
    cudaError_t e = pkv::launch_paged_decode_mq(pool->dtype, g, a, *maps, num_chunks,
                                                as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged decode (several queries) launch");
  }
  return PKV_OK;
}

}  // namespace

namespace pkv {
int pool_kv_heads(const pkv_pool* pool) { return pool ? pool->n_kv : 0; }
pkv_status check_attention_args(const pkv_pool* pool, int layer, const float* q,
                                const int32_t* block_table, int bt_stride,
                                const int32_t* seq_lens, int num_rows, int n_q_heads,
                                const float* out, int num_chunks) {
  return check_attention(pool, layer, q, block_table, bt_stride, seq_lens, num_rows, n_q_heads, out,
                         num_chunks);
}
pkv_status record_error(pkv_status s, const char* msg) { return fail(s, "%s", msg); }
}  // namespace pkv

extern "C" {

size_t kv_pool_bytes(int num_layers, int num_pages, int n_kv_heads, int head_dim,
                     pkv_kv_dtype dtype, int which) {
  if (num_layers <= 0 || num_pages <= 0 || n_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % PKV_Q8_BLOCK ||
      (dtype != PKV_KV_F16 && dtype != PKV_KV_Q8_0 && dtype != PKV_KV_BF16 &&
       dtype != PKV_KV_F32))
    return 0;
  const size_t per = which == 0 ? data_bytes_per_layer(num_pages, n_kv_heads, head_dim, dtype)
                                : scale_bytes_per_layer(num_pages, n_kv_heads, head_dim, dtype);
  return per * num_layers;
}

pkv_status kv_pool_create(pkv_pool** out, int num_layers, int num_pages, int n_kv_heads,
                          int head_dim, pkv_kv_dtype dtype, void* k_data, void* v_data,
                          void* k_scales, void* v_scales, int32_t* device_status) {
  if (!out) return fail(PKV_ERR_INVALID_ARG, "null output pointer");
  *out = nullptr;
  if (num_layers <= 0 || num_pages <= 0 || n_kv_heads <= 0)
    return fail(PKV_ERR_INVALID_ARG, "pool sizes must be positive");
  if (dtype != PKV_KV_F16 && dtype != PKV_KV_Q8_0 && dtype != PKV_KV_BF16 &&
      dtype != PKV_KV_F32)
    return fail(PKV_ERR_INVALID_ARG, "unknown KV dtype %d", static_cast<int>(dtype));
  if (head_dim != PKV_HEAD_DIM) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d != 128", head_dim);
  if (!k_data || !v_data) return fail(PKV_ERR_INVALID_ARG, "null K or V data");
  if (!aligned(k_data, 16) || !aligned(v_data, 16))
    return fail(PKV_ERR_INVALID_ARG, "K / V data not 16-byte aligned");
  if (dtype == PKV_KV_Q8_0) {
    if (!k_scales || !v_scales) return fail(PKV_ERR_INVALID_ARG, "q8_0 pool needs scale arrays");
    if (!aligned(k_scales, 16) || !aligned(v_scales, 16))
      return fail(PKV_ERR_INVALID_ARG, "scale arrays not 16-byte aligned");
  } else if (k_scales || v_scales) {
    return fail(PKV_ERR_INVALID_ARG, "f16, bf16 and f32 pools take no scale arrays");
  }
  if (device_status && !aligned(device_status, 4))
    return fail(PKV_ERR_INVALID_ARG, "status word not 4-byte aligned");
  pkv_pool* p = new (std::nothrow) pkv_pool();
  if (!p) return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  p->num_layers = num_layers;
  p->num_pages = num_pages;
  p->n_kv = n_kv_heads;
  p->head_dim = head_dim;
  p->dtype = dtype;
  p->k_data = static_cast<uint8_t*>(k_data);
  p->v_data = static_cast<uint8_t*>(v_data);
  p->k_scales = static_cast<uint8_t*>(k_scales);
  p->v_scales = static_cast<uint8_t*>(v_scales);
  p->status = device_status;
  p->layer_data_bytes = data_bytes_per_layer(num_pages, n_kv_heads, head_dim, dtype);
  p->layer_scale_bytes = scale_bytes_per_layer(num_pages, n_kv_heads, head_dim, dtype);
  p->maps = nullptr;
  p->ready = nullptr;
  p->window = nullptr;
  if (static_cast<long long>(num_pages) * n_kv_heads >= (1ll << 31)) {
    delete p;
    return fail(PKV_ERR_UNSUPPORTED, "num_pages * n_kv_heads must be below 2^31");
  }
  p->maps = new (std::nothrow) pkv::TileMaps[num_layers];
  p->ready = new (std::nothrow) std::atomic<int>[num_layers];
  p->window = new (std::nothrow) int[num_layers];
  if (!p->maps || !p->ready || !p->window) {
    delete p;
    return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  }
  for (int l = 0; l < num_layers; ++l) {
    p->ready[l].store(0);
    p->window[l] = 0;
  }
  *out = p;
  return PKV_OK;
}

void kv_pool_destroy(pkv_pool* pool) { delete pool; }

pkv_status kv_pool_set_window(pkv_pool* pool, int layer, int window) {
  pkv_status s = check_pool_layer(pool, layer);
  if (s) return s;
  if (window < 0) return fail(PKV_ERR_INVALID_ARG, "window < 0");
  pool->window[layer] = window;
  return PKV_OK;
}

pkv_status kv_pool_get_window(const pkv_pool* pool, int layer, int* window) {
  pkv_status s = check_pool_layer(pool, layer);
  if (s) return s;
  if (!window) return fail(PKV_ERR_INVALID_ARG, "null window pointer");
  *window = pool->window[layer];
  return PKV_OK;
}

pkv_status kv_pool_set_test_stall(pkv_pool* pool, unsigned long long stall_ns) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "null pool");
  if (stall_ns > PKV_DEFAULT_WAIT_NS)
    return fail(PKV_ERR_INVALID_ARG, "stall_ns above PKV_DEFAULT_WAIT_NS");
  pool->test_stall_ns = stall_ns;
  return PKV_OK;
}

pkv_status kv_pool_read_status(const pkv_pool* pool, void* stream, int32_t* status) {
  if (!pool || !status) return fail(PKV_ERR_INVALID_ARG, "null pool or status pointer");
  *status = 0;
  if (!pool->status) return PKV_OK;
  cudaError_t e = cudaMemcpyAsync(status, pool->status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  as_stream(stream));
  if (e == cudaSuccess)
    e = cudaMemsetAsync(pool->status, 0, sizeof(int32_t), as_stream(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  return PKV_OK;
}

pkv_status kv_append(const pkv_pool* pool, int layer, const float* k_new, const float* v_new,
                     const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                     int num_rows, void* stream) {
  pkv_status s = check_pool_layer(pool, layer);
  if (s) return s;
  if ((s = check_rows(num_rows, bt_stride, block_table, seq_lens, 1 << 24))) return s;
  if (num_rows > 0 && (!k_new || !v_new)) return fail(PKV_ERR_INVALID_ARG, "null k_new or v_new");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_new / v_new not 16-byte aligned");
  if (num_rows == 0) return PKV_OK;
  pkv::AppendArgs a;
  a.k_data = pool->k_data + layer * pool->layer_data_bytes;
  a.v_data = pool->v_data + layer * pool->layer_data_bytes;
  a.k_scales = pool->k_scales ? pool->k_scales + layer * pool->layer_scale_bytes : nullptr;
  a.v_scales = pool->v_scales ? pool->v_scales + layer * pool->layer_scale_bytes : nullptr;
  a.num_pages = pool->num_pages;
  a.n_kv = pool->n_kv;
  a.k_new = k_new;
  a.v_new = v_new;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.num_rows = num_rows;
  a.status = pool->status;
  cudaError_t e = pkv::launch_append(pool->dtype, a, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return PKV_OK;
}

pkv_status paged_decode_default_chunks(const pkv_pool* pool, int n_q_heads, int max_rows,
                                       int* chunks) {
  if (!pool || !chunks) return fail(PKV_ERR_INVALID_ARG, "null pool or output pointer");
  pkv_status s = check_geometry(n_q_heads, pool->n_kv, pool->head_dim);
  if (s) return s;
  if (max_rows < 1 || max_rows > PKV_MAX_ROWS)
    return fail(PKV_ERR_UNSUPPORTED, "max_rows %d outside [1, %d]", max_rows, PKV_MAX_ROWS);
  return default_chunks(pool, n_q_heads, max_rows, chunks);
}

size_t paged_decode_workspace_bytes(int max_rows, int n_q_heads, int n_kv_heads, int head_dim,
                                    int num_chunks) {
  if (max_rows < 0 || num_chunks < 1 || num_chunks > PKV_MAX_CHUNKS || n_kv_heads <= 0 || n_q_heads <= 0 ||
      n_q_heads % n_kv_heads || head_dim != PKV_HEAD_DIM)
    return 0;
  return workspace_needed(max_rows, n_q_heads, n_kv_heads, num_chunks);
}

pkv_status paged_decode_attention(const pkv_pool* pool, int layer, const float* q,
                                  const int32_t* block_table, int bt_stride,
                                  const int32_t* seq_lens, int num_rows, int n_q_heads,
                                  float scale, float* out, void* workspace,
                                  size_t workspace_bytes, int num_chunks, void* stream) {
  return attention_impl(pool, layer, q, nullptr, nullptr, block_table, bt_stride, seq_lens,
                        num_rows, n_q_heads, scale, out, workspace, workspace_bytes, num_chunks,
                        stream, Mode::kMerged);
}

pkv_status paged_decode_split(const pkv_pool* pool, int layer, const float* q,
                              const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                              int num_rows, int n_q_heads, float scale, float* out,
                              void* workspace, size_t workspace_bytes, int num_chunks,
                              void* stream) {
  return attention_impl(pool, layer, q, nullptr, nullptr, block_table, bt_stride, seq_lens,
                        num_rows, n_q_heads, scale, out, workspace, workspace_bytes, num_chunks,
                        stream, Mode::kSplitOnly);
}

pkv_status paged_decode_plan(const int32_t* seq_lens, int num_rows, int n_kv_heads,
                             int bt_stride, int window, int num_chunks, pkv_kv_dtype kv_dtype,
                             int32_t* row_page_start, int32_t* seg_first_chunk,
                             int32_t* seg_last_chunk, void* stream) {
  pkv_status s = check_rows(num_rows, bt_stride, seq_lens, seq_lens);
  if (s) return s;
  if (!known_dtype(kv_dtype)) return fail(PKV_ERR_INVALID_ARG, "unknown KV dtype %d", static_cast<int>(kv_dtype));
  if (window < 0) return fail(PKV_ERR_INVALID_ARG, "window < 0");
  if (n_kv_heads <= 0 || num_chunks < 1)
    return fail(PKV_ERR_INVALID_ARG, "n_kv_heads and num_chunks must be positive");
  if (num_chunks > PKV_MAX_CHUNKS) return fail(PKV_ERR_UNSUPPORTED, "num_chunks > %d", PKV_MAX_CHUNKS);
  if (!row_page_start || (num_rows > 0 && (!seg_first_chunk || !seg_last_chunk)))
    return fail(PKV_ERR_INVALID_ARG, "null plan output");
  pkv::PlanArgs a{seq_lens,  window,         num_rows,        n_kv_heads,     bt_stride,
                  num_chunks, split_may_align(kv_dtype), row_page_start, seg_first_chunk,
                  seg_last_chunk};
  cudaError_t e = pkv::launch_plan(a, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  return PKV_OK;
}

pkv_status paged_decode_combine(const int32_t* seq_lens, int num_rows, int n_q_heads,
                                int n_kv_heads, int head_dim, int bt_stride, int window,
                                int num_chunks, pkv_kv_dtype kv_dtype, const void* workspace,
                                size_t workspace_bytes, float* out, void* stream) {
  pkv_status s = check_geometry(n_q_heads, n_kv_heads, head_dim);
  if (s) return s;
  if (!known_dtype(kv_dtype)) return fail(PKV_ERR_INVALID_ARG, "unknown KV dtype %d", static_cast<int>(kv_dtype));
  if (window < 0) return fail(PKV_ERR_INVALID_ARG, "window < 0");
  if ((s = check_rows(num_rows, bt_stride, seq_lens, seq_lens))) return s;
  if (num_chunks < 1) return fail(PKV_ERR_INVALID_ARG, "num_chunks < 1");
  if (num_chunks > PKV_MAX_CHUNKS) return fail(PKV_ERR_UNSUPPORTED, "num_chunks > %d", PKV_MAX_CHUNKS);
  if (num_rows > 0 && !out) return fail(PKV_ERR_INVALID_ARG, "null out");
  const size_t need = workspace_needed(num_rows, n_q_heads, n_kv_heads, num_chunks);
  if (!workspace || workspace_bytes < need)
    return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (num_rows == 0) return PKV_OK;
  const int g = n_q_heads / n_kv_heads;
  const WsParts w = workspace_parts(const_cast<void*>(workspace), workspace_bytes, num_rows,
                                    n_q_heads, n_kv_heads, num_chunks);
  pkv::CombineArgs c;
  c.seq_lens = seq_lens;
  c.window = window;
  c.num_rows = num_rows;
  c.n_q = n_q_heads;
  c.n_kv = n_kv_heads;
  c.bt_stride = bt_stride;
  c.num_chunks = num_chunks;
  c.aligned_split = split_may_align(kv_dtype);
  c.part_ml = w.part_ml;
  c.part_acc = w.part_acc;
  c.out = out;
  cudaError_t e = pkv::launch_combine(g, c, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return PKV_OK;
}

pkv_status pkv_decode_step(const pkv_pool* pool, int layer, const float* q, const float* k_new,
                           const float* v_new, const int32_t* block_table, int bt_stride,
                           const int32_t* seq_lens, int num_rows, int n_q_heads, float scale,
                           float* out, void* workspace, size_t workspace_bytes, int num_chunks,
                           void* stream) {
  // One launch: the kernel stores each row's new token into its last page
  // just before reading that page, then attends and merges.
  if (num_rows > 0 && (!k_new || !v_new)) return fail(PKV_ERR_INVALID_ARG, "null k_new or v_new");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_new / v_new not 16-byte aligned");
  return attention_impl(pool, layer, q, k_new, v_new, block_table, bt_stride, seq_lens, num_rows,
                        n_q_heads, scale, out, workspace, workspace_bytes, num_chunks, stream,
                        Mode::kMerged);
}

size_t paged_decode_workspace_bytes_mq(int max_rows, int n_q_heads, int n_kv_heads, int head_dim,
                                       int num_chunks) {
  if (max_rows < 0 || num_chunks < 1 || num_chunks > PKV_MAX_CHUNKS || n_kv_heads <= 0 || n_q_heads <= 0 ||
      n_q_heads % n_kv_heads || head_dim != PKV_HEAD_DIM)
    return 0;
  return workspace_needed_mq(max_rows, n_kv_heads, num_chunks);
}

pkv_status paged_decode_default_chunks_mq(const pkv_pool* pool, int n_q_heads, int max_rows,
                                          int q_len, int* chunks) {
  if (!pool || !chunks) return fail(PKV_ERR_INVALID_ARG, "null pool or output pointer");
  pkv_status s = check_geometry(n_q_heads, pool->n_kv, pool->head_dim);
  if (s) return s;
  if (max_rows < 1 || max_rows > PKV_MAX_ROWS)
    return fail(PKV_ERR_UNSUPPORTED, "max_rows %d outside [1, %d]", max_rows, PKV_MAX_ROWS);
  if (q_len < 1 || q_len > PKV_MAX_Q_LEN)
    return fail(PKV_ERR_UNSUPPORTED, "q_len %d outside [1, %d]", q_len, PKV_MAX_Q_LEN);
  return default_chunks_mq(pool, n_q_heads / pool->n_kv, q_len, max_rows, chunks);
}

pkv_status paged_decode_attention_mq(const pkv_pool* pool, int layer, const float* q,
                                     const int32_t* block_table, int bt_stride,
                                     const int32_t* seq_lens, int num_rows, int q_len,
                                     int n_q_heads, float scale, float* out, void* workspace,
                                     size_t workspace_bytes, int num_chunks, void* stream) {
  return attention_mq_impl(pool, layer, q, nullptr, nullptr, block_table, bt_stride, seq_lens,
                           num_rows, q_len, n_q_heads, scale, out, workspace, workspace_bytes,
                           num_chunks, stream);
}

pkv_status pkv_decode_step_mq(const pkv_pool* pool, int layer, const float* q, const float* k_new,
                              const float* v_new, const int32_t* block_table, int bt_stride,
                              const int32_t* seq_lens, int num_rows, int q_len, int n_q_heads,
                              float scale, float* out, void* workspace, size_t workspace_bytes,
                              int num_chunks, void* stream) {
  if (num_rows > 0 && (!k_new || !v_new)) return fail(PKV_ERR_INVALID_ARG, "null k_new or v_new");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_new / v_new not 16-byte aligned");
  return attention_mq_impl(pool, layer, q, k_new, v_new, block_table, bt_stride, seq_lens,
                           num_rows, q_len, n_q_heads, scale, out, workspace, workspace_bytes,
                           num_chunks, stream);
}

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_CAPACITY: return "PKV_ERR_CAPACITY";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
  }
  return "PKV_ERR_UNKNOWN";
}

const char* pkv_last_error_message(void) { return g_last_error; }

}  // extern "C"

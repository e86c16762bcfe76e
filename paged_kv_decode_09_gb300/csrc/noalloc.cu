// noalloc.cu — paged_decode_attention_static: paged_decode_attention with its
// workspace in a fixed array inside this library, for callers that cannot
// allocate device memory when they decode.
//
// Who needs it: a serving process that reserves all of its device memory up
// front (the KV page pool plus a caching allocator take nearly the whole
// GPU, so a later cudaMalloc fails or fragments the reservation), and code
// running where a cudaMalloc is not allowed or would stall the device
// (cudaMalloc may synchronise implicitly).  Such callers still pass their own
// inputs and outputs; only the scratch lives here.
//
// The scratch is a file-scope __device__ array: every GPU that loads
// libpkv.so holds PKV_STATIC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so the first call on each device, with that
// device current, looks the address up with cudaGetSymbolAddress and keeps
// it; that first call should come before any stream capture.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_addr[kMaxDevices] = {};

thread_local char g_static_error[160] = "";

}  // namespace

extern "C" pkv_status paged_decode_attention_static(const pkv_pool* pool, int layer,
                                                    const float* q, const int32_t* block_table,
                                                    int bt_stride, const int32_t* seq_lens,
                                                    int num_rows, int n_q_heads, float scale,
                                                    float* out, int num_chunks, void* stream) {
  if (!pool) return pkv::record_error(PKV_ERR_INVALID_ARG, "null pool");
  if (num_rows < 0 || num_rows > PKV_MAX_ROWS)
    return pkv::record_error(PKV_ERR_UNSUPPORTED, "num_rows outside [0, PKV_MAX_ROWS]");
  if (num_rows == 0)
    return paged_decode_attention(pool, layer, q, block_table, bt_stride, seq_lens, 0, n_q_heads,
                                  scale, out, nullptr, 0, num_chunks, stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return pkv::record_error(PKV_ERR_CUDA, "paged_decode_attention_static: no current device");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
        return pkv::record_error(PKV_ERR_CUDA,
                                 "paged_decode_attention_static: cudaGetSymbolAddress failed");
      g_addr[dev] = p;
    }
    base = g_addr[dev];
  }
  // The chunk count fixes the workspace size; resolve the default here.
  if (num_chunks == 0) {
    pkv_status s = paged_decode_default_chunks(pool, n_q_heads, num_rows, &num_chunks);
    if (s != PKV_OK) return s;
  }
  const int n_kv = pkv::pool_kv_heads(pool);
  const size_t need =
      paged_decode_workspace_bytes(num_rows, n_q_heads, n_kv, PKV_HEAD_DIM, num_chunks);
  if (need > PKV_STATIC_SCRATCH_BYTES) {
    snprintf(g_static_error, sizeof(g_static_error),
             "paged_decode_attention_static: this call needs %zu bytes of scratch; the "
             "static array holds %u (fewer rows or chunks fit)",
             need, static_cast<unsigned>(PKV_STATIC_SCRATCH_BYTES));
    return pkv::record_error(PKV_ERR_WORKSPACE, g_static_error);
  }
  // The arrival counters must start at zero.  Completed calls leave them at
  // zero, but a call that timed out may not have: clear them every time.
  if (need > 0) {
    const size_t counters =
        pkv::counter_bytes(static_cast<long long>(num_rows) * n_kv);
    if (cudaMemsetAsync(base, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return pkv::record_error(PKV_ERR_CUDA, "paged_decode_attention_static: clearing counters");
  }
  // need == 0 means invalid geometry: the regular entry point reports it.
  return paged_decode_attention(pool, layer, q, block_table, bt_stride, seq_lens, num_rows,
                                n_q_heads, scale, out, base, PKV_STATIC_SCRATCH_BYTES, num_chunks,
                                stream);
}

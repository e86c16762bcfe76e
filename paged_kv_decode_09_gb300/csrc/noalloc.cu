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
// it; that first call should come before any stream capture.  The address
// is kept together with the id of the CUDA context it belongs to: after a
// device reset the runtime creates a new context, loads the module again
// (the array may then sit elsewhere), and the next call looks it up anew.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx[kMaxDevices] = {};  // id of the context g_addr[dev] belongs to

thread_local char g_static_error[160] = "";

// The id of the calling thread's current CUDA context, through the driver
// (reached via the runtime, no link against the driver library); false if
// there is none yet or the driver cannot say.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

extern "C" pkv_status paged_decode_attention_static(const pkv_pool* pool, int layer,
                                                    const float* q, const int32_t* block_table,
                                                    int bt_stride, const int32_t* seq_lens,
                                                    int num_rows, int n_q_heads, float scale,
                                                    float* out, int num_chunks, void* stream) {
  // Every check of the regular entry point comes first: a call that will not
  // launch leaves the shared array alone.
  pkv_status st = pkv::check_attention_args(pool, layer, q, block_table, bt_stride, seq_lens,
                                            num_rows, n_q_heads, out, num_chunks);
  if (st != PKV_OK) return st;
  if (num_rows == 0)
    return paged_decode_attention(pool, layer, q, block_table, bt_stride, seq_lens, 0, n_q_heads,
                                  scale, out, nullptr, 0, num_chunks, stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return pkv::record_error(PKV_ERR_CUDA, "paged_decode_attention_static: no current device");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    unsigned long long id = 0;
    const bool known = current_context_id(&id);
    if (!g_addr[dev] || !known || g_ctx[dev] != id) {
      void* p = nullptr;
      // also creates the device's context if the thread has none yet
      if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
        return pkv::record_error(PKV_ERR_CUDA,
                                 "paged_decode_attention_static: cudaGetSymbolAddress failed");
      // without a context id from the driver, nothing is kept (the next call
      // looks the address up again)
      g_addr[dev] = current_context_id(&id) ? p : nullptr;
      g_ctx[dev] = id;
      base = p;
    } else {
      base = g_addr[dev];
    }
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
  // The merge's flags (arrival counters and ready flags, at the end of the
  // array) must start at zero.  Completed calls leave them at zero, but a call
  // that timed out may not have: clear this call's flags every time.
  if (need > 0) {
    const long long slots = static_cast<long long>(num_chunks) + static_cast<long long>(num_rows) * n_kv;
    const size_t flags = pkv::flag_bytes(slots);
    uint8_t* end = reinterpret_cast<uint8_t*>(pkv::flags_end(base, PKV_STATIC_SCRATCH_BYTES));
    if (cudaMemsetAsync(end - flags, 0, flags, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return pkv::record_error(PKV_ERR_CUDA, "paged_decode_attention_static: clearing counters");
  }
  // need == 0 means invalid geometry: the regular entry point reports it.
  return paged_decode_attention(pool, layer, q, block_table, bt_stride, seq_lens, num_rows,
                                n_q_heads, scale, out, base, PKV_STATIC_SCRATCH_BYTES, num_chunks,
                                stream);
}

/*
 * pkv.h — C ABI of libpkv.so: one decode step of paged-KV attention on a
 * GB300 GPU (sm_103a).
 *
 * What it computes.  Rows (active sequences) are decoded together in one batch
 * (Leone, "What ships": continuous decode batching across active requests;
 * tinyllm, "The repository currently provides": variable-length batched decode
 * for several active sequences).  Each row's K/V live in a shared pool of
 * fixed 16-token physical pages, reached through that row's block table
 * (tinyllm, "The repository currently provides": a runner-owned physical KV
 * page pool and a logical block table per active sequence; "Known
 * limitations": 16-token pages).  Attention is GQA (tinyllm, "The repository
 * currently provides": GQA attention), and K/V are stored as f16 or q8_0
 * (Leone, "What ships": f16 and q8 KV storage; LeatEngine, "Run": the q8_0
 * KV cache, as llama.cpp keeps it, in about half the memory of f16).  For
 * row i and query head g, with G = n_q_heads / n_kv_heads and h = g / G:
 *
 *     out[i][g] = sum_{t < L_i} softmax_t(scale * <q[i][g], K[i][h][t]>) V[i][h][t]
 *
 * where K and V are the stored values and L_i = seq_lens[i].  tinyllm's own
 * paged path gathers a row's pages and right-pads them before dense attention
 * ("Known limitations"); this library reads the pages in place instead.
 *
 * Conventions (readings where the pages are silent):
 *   - seq_lens[i] counts the tokens row i attends to, INCLUDING the token
 *     appended this step; kv_append writes position seq_lens[i] - 1.
 *   - Block table: int32 [num_rows][bt_stride]; entry p of row i is the
 *     physical page of tokens 16p .. 16p + 15.  Only the first
 *     ceil(seq_lens[i] / 16) entries are read.
 *   - Pool, per layer, per K and per V (layer l starts at l times the
 *     per-layer size):
 *       f16 : data   [num_pages][n_kv_heads][16][head_dim]  binary16
 *       bf16: data   [num_pages][n_kv_heads][16][head_dim]  bfloat16
 *       f32 : data   [num_pages][n_kv_heads][16][head_dim]  binary32
 *       q8_0: data   [num_pages][n_kv_heads][16][head_dim]  code + 128 (uint8)
 *             scales [num_pages][n_kv_heads][16][head_dim/32] binary16
 *     q8_0 value = scale of the element's 32-wide block (along head_dim)
 *     times its code.  Encoding: d = amax / 127 (fp32, IEEE division), stored
 *     scale = binary16(d) rounded to nearest even, code = round(x / d) with
 *     ties away from zero (using the fp32 d); amax = 0 gives d = 0, codes 0.
 *     The data byte is code + 128 (offset-binary: the int8 code's top bit
 *     flipped).
 *   - q, out: fp32 [num_rows][n_q_heads][head_dim].  k_new, v_new: fp32
 *     [num_rows][n_kv_heads][head_dim].
 *   - head_dim must be 128; n_q_heads / n_kv_heads must be 1, 2 or 4.
 *
 * Ownership and threading.  Every data pointer is a DEVICE pointer that the
 * caller allocates and frees; the library allocates no device memory, frees
 * nothing and never synchronises a stream on the decode path.  `stream` is a
 * cudaStream_t (NULL: the legacy default stream); all work is queued on it and
 * the calls return before it runs.  The opaque pkv_pool is a small host-side
 * descriptor; it holds the caller's pointers, not copies.
 *
 * Errors.  Every call checks its arguments on the host and returns a status
 * before queueing anything; a failed launch returns PKV_ERR_CUDA.  Problems
 * only the device can see (a block-table entry outside the pool, a length
 * beyond the block table, a bounded wait that gave up) do not fault: the
 * kernels clamp or skip the access and record a PKV_DEV_* bit in the pool's
 * optional device status word, which kv_pool_read_status returns.
 * pkv_last_error_message gives a one-line reason for the calling thread's
 * last failed call.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_PAGE_TOKENS 16
#define PKV_HEAD_DIM 128
#define PKV_Q8_BLOCK 32
#define PKV_MAX_ROWS 2048 /* rows per call (per-CTA row tables live in shared memory) */
#define PKV_MAX_CHUNKS (1 << 24) /* work chunks per call (PKV_ERR_UNSUPPORTED above) */

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, bad layer */
    PKV_ERR_UNSUPPORTED = 2,  /* head_dim != 128, GQA group not in {1,2,4}, too many rows */
    PKV_ERR_CAPACITY = 3,     /* more pages than the pool holds */
    PKV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
    PKV_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
} pkv_status;

/* Bits the kernels OR into the pool's device status word. */
#define PKV_DEV_BAD_PAGE 1u   /* block-table entry outside [0, num_pages): page 0 read instead, or write skipped */
#define PKV_DEV_BAD_LENGTH 2u /* seq_lens[i] < 0 or > 16 * bt_stride: clamped */
#define PKV_DEV_TIMEOUT 4u    /* a bounded wait on a shared-memory barrier gave up */

/* How long (ns) a warp of the attention kernels waits on a shared-memory
 * barrier (a tile copy, a peer warp) before the kernel gives up. */
#define PKV_DEFAULT_WAIT_NS (1ull << 30)

/* Stored KV formats: binary16; q8_0 (codes in [-127, 127] + one binary16
 * scale per 32 values along head_dim, value = scale * code); bfloat16,
 * rounded to nearest even, and binary32, stored as given (tinyllm, "The
 * repository currently provides": BF16/F32 KV caching).  Data arrays hold 2
 * bytes per value (f16, bf16), 4 (f32) or 1 (q8_0: the code stored
 * offset-binary, as the unsigned byte code + 128, i.e. the int8 code with its
 * top bit flipped, which the attention kernels widen to f16 without a
 * per-byte sign fix). */
typedef enum pkv_kv_dtype {
    PKV_KV_F16 = 0,
    PKV_KV_Q8_0 = 1,
    PKV_KV_BF16 = 2,
    PKV_KV_F32 = 3,
} pkv_kv_dtype;

typedef struct pkv_pool pkv_pool;

/* Bytes of one pool array for all layers: which = 0 the data array (K or V),
 * which = 1 the q8_0 scale array (0 for f16 and bf16).  Returns 0 for
 * invalid sizes. */
size_t kv_pool_bytes(int num_layers, int num_pages, int n_kv_heads, int head_dim,
                     pkv_kv_dtype dtype, int which);

/* Describe a caller-owned KV page pool (tinyllm, "The repository currently
 * provides": one runner-owned physical KV page pool).
 *   k_data, v_data     device arrays of kv_pool_bytes(..., 0) bytes, 16-byte aligned
 *   k_scales, v_scales q8_0: device arrays of kv_pool_bytes(..., 1) bytes,
 *                      16-byte aligned; f16, bf16, f32: must be NULL
 *   device_status      optional device int32 (NULL: none), zero before first
 *                      use; kernels OR PKV_DEV_* bits into it.
 * num_pages * n_kv_heads must be below 2^31 (PKV_ERR_UNSUPPORTED).  Creating
 * a descriptor touches no device memory and needs no driver; the first
 * attention call on a layer encodes that layer's tensor maps (host only)
 * into the descriptor and reports PKV_ERR_CUDA if the driver cannot.
 * On success *out receives a descriptor to free with kv_pool_destroy. */
pkv_status kv_pool_create(pkv_pool **out, int num_layers, int num_pages, int n_kv_heads,
                          int head_dim, pkv_kv_dtype dtype, void *k_data, void *v_data,
                          void *k_scales, void *v_scales, int32_t *device_status);

/* Free a descriptor (not the caller's arrays).  NULL is allowed. */
void kv_pool_destroy(pkv_pool *pool);

/* Sliding window of a layer (LeatEngine, "Capabilities": sliding-window KV
 * caches).  With window W > 0, every attention call on the layer lets a row
 * of L tokens attend to its last W tokens, [max(0, L - W), L), the token
 * appended this step included, and reads only the pages holding them:
 * block-table entries floor(max(0, L - W) / 16) onwards.  W = 0 (the
 * default) attends to all L tokens.  Host-side descriptor state, read when a
 * call is queued; kv_append is unaffected.  W < 0 -> PKV_ERR_INVALID_ARG. */
pkv_status kv_pool_set_window(pkv_pool *pool, int layer, int window);
pkv_status kv_pool_get_window(const pkv_pool *pool, int layer, int *window);

/* Test hook, not part of the method: it lets the kernels' give-up path be
 * run on a real GPU, with no hang and no fault.  With stall_ns > 0, every
 * attention call queued on this descriptor from now on makes each warp of
 * the kernel, once it has queued its first tile copies, wait up to stall_ns
 * on a barrier that nothing completes, as it would on a copy that never
 * lands.  That wait runs out, and the kernel gives up as on a real timeout:
 * it stops reading, ORs PKV_DEV_TIMEOUT into the status word, waits for the
 * copies it has in flight to land (each up to PKV_DEFAULT_WAIT_NS), and
 * returns.  The call's outputs are then undefined and its workspace may hold
 * non-zero arrival counters: zero the workspace before the next call uses
 * it.  stall_ns = 0 (the default) turns the hook off; values above
 * PKV_DEFAULT_WAIT_NS return PKV_ERR_INVALID_ARG.  Host-side descriptor
 * state; setting it while another thread queues calls is a data race. */
pkv_status kv_pool_set_test_stall(pkv_pool *pool, unsigned long long stall_ns);

/* Wait for `stream`, copy the pool's device status word into *status and
 * reset it to 0.  This call synchronises; it is not part of the decode path.
 * Without a status word, *status = 0. */
pkv_status kv_pool_read_status(const pkv_pool *pool, void *stream, int32_t *status);

/* kv_append — store one new K and V token per row into its page slot
 * (tinyllm, "The repository currently provides": an incremental decoder per
 * active sequence writing through its block table; Leone, "What ships" and
 * LeatEngine, "Run": f16 and q8_0 KV storage).
 * For each row i with L = seq_lens[i] >= 1 and each KV head h, encodes
 * k_new[i][h][:] and v_new[i][h][:] (fp32, 16-byte aligned) into page
 * block_table[i][(L - 1) / 16], slot (L - 1) % 16 of `layer`.  Rows with
 * L == 0 write nothing.  num_rows is not limited by PKV_MAX_ROWS (up to 2^24).
 * One launch; asynchronous on `stream`. */
pkv_status kv_append(const pkv_pool *pool, int layer, const float *k_new, const float *v_new,
                     const int32_t *block_table, int bt_stride, const int32_t *seq_lens,
                     int num_rows, void *stream);

/* Number of work chunks (one per resident CTA of the attention kernel) that
 * fills this GPU, for calls of up to max_rows rows with this pool and
 * n_q_heads.  Queries the current device. */
pkv_status paged_decode_default_chunks(const pkv_pool *pool, int n_q_heads, int max_rows,
                                       int *chunks);

/* Workspace bytes paged_decode_attention needs for up to max_rows rows with
 * num_chunks chunks.  Layout for a call of num_rows rows, with S = num_chunks
 * + num_rows * n_kv_heads partial slots and G = n_q / n_kv, from the start:
 *     part_ml  float [S][G][2]  (m2, l) per slot and query head of the group
 *     part_acc float [S][G][head_dim]  (at the next 256-byte boundary)
 * and down from the end E (workspace_bytes rounded down to a multiple of 256),
 * int32 flags: the arrival count of (row, KV head) j at E - 4 (2j + 1), and
 * the ready flag of slot s (its partial state is complete) at E - 4 (2s + 2).
 * The flags keep their places whatever the call's rows and chunks, so one
 * workspace sized for the largest call serves every smaller call.  It must
 * be zero-filled once before its first use (the flags must start at 0);
 * every call that completes leaves them at 0 again.
 * After a call that reported PKV_DEV_TIMEOUT, zero it again.  Calls that
 * share a workspace must not run concurrently.  Returns 0 for invalid sizes. */
size_t paged_decode_workspace_bytes(int max_rows, int n_q_heads, int n_kv_heads, int head_dim,
                                    int num_chunks);

/* paged_decode_attention — decode attention for a batch of variable-length
 * rows straight from the paged pool (the operation tinyllm's paged-reference
 * path computes by gathering and right-padding, "Known limitations").
 *   q            fp32 [num_rows][n_q_heads][128], 16-byte aligned
 *   block_table  int32 [num_rows][bt_stride]; seq_lens int32 [num_rows]
 *   scale        softmax scale (1/sqrt(head_dim) for the usual attention)
 *   out          fp32 [num_rows][n_q_heads][128], 16-byte aligned
 *   workspace    device scratch of paged_decode_workspace_bytes(num_rows ...)
 *                bytes, 256-byte aligned, zero-filled before its first use
 *   num_chunks   work chunks (0: paged_decode_default_chunks for num_rows)
 * The T (row, KV head, page) tiles of the batch are split into at most
 * num_chunks contiguous chunks, one per CTA, as paged_decode_plan describes;
 * a CTA streams its tiles through shared memory, keeps a base-2 online softmax in fp32 for the
 * G query heads of the tile's KV head, and writes either the final output
 * (when it holds a whole (row, KV head)) or a partial state (m2, l, acc) to
 * slot chunk + row * n_kv_heads + head of the workspace.  The last CTA to
 * finish a piece of a split (row, KV head) merges all its pieces into the
 * output.  Rows with seq_lens[i] == 0 get zeros.  A layer with a sliding
 * window (kv_pool_set_window) attends to each row's last `window` tokens and
 * counts only the pages holding them.  One launch, no host
 * synchronisation. */
pkv_status paged_decode_attention(const pkv_pool *pool, int layer, const float *q,
                                  const int32_t *block_table, int bt_stride,
                                  const int32_t *seq_lens, int num_rows, int n_q_heads,
                                  float scale, float *out, void *workspace,
                                  size_t workspace_bytes, int num_chunks, void *stream);

/* paged_decode_split — paged_decode_attention without the in-kernel merge
 * (same arguments): every piece that holds a whole (row, KV head) writes
 * `out`, the others leave their partial states in the workspace, and
 * paged_decode_combine with the same seq_lens, num_chunks and workspace
 * completes the call.  The counters are not used.  One launch. */
pkv_status paged_decode_split(const pkv_pool *pool, int layer, const float *q,
                              const int32_t *block_table, int bt_stride, const int32_t *seq_lens,
                              int num_rows, int n_q_heads, float scale, float *out,
                              void *workspace, size_t workspace_bytes, int num_chunks,
                              void *stream);

/* paged_decode_plan — the work split paged_decode_attention uses on a pool of
 * KV format kv_dtype, written out for inspection.  Units are (row, KV head,
 * page) tiles in that order; row i reads the pages holding its attended
 * tokens [a_i, L_i), a_i = max(0, L_i - window) (0 for window 0):
 * npg_i = ceil(L_i / 16) - floor(a_i / 16) pages; the units of one (row, KV
 * head) form a segment; T = n_kv_heads * total pages; C = num_chunks.
 *   Aligned split (f16 and bf16 KV, when it balances): for a cap of t
 *   units a chunk, a row with npg_i >= t gives each of its segments
 *   c = ceil(npg_i / t) chunks, the q-th covering the segment's pages
 *   [floor(q npg_i / c), floor((q + 1) npg_i / c)); a row with npg_i < t gives
 *   ceil(n_kv_heads / m) chunks of m = floor(t / npg_i) whole segments (the
 *   last fewer).  Chunks are numbered in unit order.  t is the smallest
 *   integer from ceil(T / C) for which all rows need at most C chunks; the
 *   split is used when t <= floor(11 T / (10 C)), floor(11 T / (10 C)) >
 *   ceil(T / C) and T < 2^31.  No segment split over several chunks ends
 *   inside a chunk.
 *   Uniform split (q8_0 and f32 KV, or when the aligned one does not
 *   balance): of C
 *   chunks C' = min(C, T) are used, chunk k covering units
 *   [floor(k T / C'), floor((k + 1) T / C')).
 * `window` must be the layer's window of the call the plan describes.
 *   row_page_start  int32 [num_rows + 1]: exclusive prefix sum of pages
 *   seg_first_chunk, seg_last_chunk  int32 [num_rows * n_kv_heads]: first and
 *                   last chunk meeting segment (row, head) (-1 if empty)
 * One single-CTA launch. */
pkv_status paged_decode_plan(const int32_t *seq_lens, int num_rows, int n_kv_heads,
                             int bt_stride, int window, int num_chunks, pkv_kv_dtype kv_dtype,
                             int32_t *row_page_start, int32_t *seg_first_chunk,
                             int32_t *seg_last_chunk, void *stream);

/* paged_decode_combine — merge the base-2 partial states of every
 * (row, query head) split over several chunks:
 *     M = max_s m2_s,  out = sum_s 2^(m2_s - M) acc_s / sum_s 2^(m2_s - M) l_s
 * over the slots chunk + row * n_kv_heads + head of the chunks the plan
 * assigns to the segment.  Segments held whole by one chunk are left as they
 * are; rows with seq_lens[i] == 0 get zeros.  The workspace layout is the one
 * paged_decode_workspace_bytes describes; `window` is the layer's window and
 * kv_dtype the pool's KV format of the paged_decode_split call being
 * completed.  One launch. */
pkv_status paged_decode_combine(const int32_t *seq_lens, int num_rows, int n_q_heads,
                                int n_kv_heads, int head_dim, int bt_stride, int window,
                                int num_chunks, pkv_kv_dtype kv_dtype, const void *workspace,
                                size_t workspace_bytes, float *out, void *stream);

/* pkv_decode_step — one decode step of one layer: the new K/V token of every
 * row is stored as kv_append would store it, and attention runs over the
 * lengths that include it (paged_decode_attention).  One launch: the CTA
 * that reads a row's last page stores the new token there just before
 * reading it.  A row's last page must not be shared with another row (full
 * pages may be).  Same arguments as the two calls. */
pkv_status pkv_decode_step(const pkv_pool *pool, int layer, const float *q, const float *k_new,
                           const float *v_new, const int32_t *block_table, int bt_stride,
                           const int32_t *seq_lens, int num_rows, int n_q_heads, float scale,
                           float *out, void *workspace, size_t workspace_bytes, int num_chunks,
                           void *stream);

/* Several queries per row: the verification step of speculative decoding and
 * short chunks of chunked prefill (Leone, "What ships": chunked prefill and
 * exact speculative verification; LeatEngine, "Capabilities": chunked
 * prefill, speculative decoding).
 *
 * Each row i has q_len (1 .. PKV_MAX_Q_LEN) new tokens, the last q_len of its
 * L = seq_lens[i] >= q_len tokens.  Query j (0 <= j < q_len) sits at position
 * P = L - q_len + j and attends causally to [max(0, P + 1 - W), P + 1), W the
 * layer's window (0: [0, P + 1)):
 *
 *     out[i][j][g] = sum_{t in that range} softmax_t(scale * <q[i][j][g], K[i][h][t]>) V[i][h][t]
 *
 *   q, out        fp32 [num_rows][q_len][n_q_heads][128], 16-byte aligned
 *   k_new, v_new  fp32 [num_rows][q_len][n_kv_heads][128] (pkv_decode_step_mq):
 *                 token j of row i is stored at position L - q_len + j
 * Rows with L == 0 get zeros; rows with 0 < L < q_len get zeros and set
 * PKV_DEV_BAD_LENGTH.  A row reads the pages holding [L - q_len + 1 - W, L)
 * (all of [0, L) without a window), split into chunks as in
 * paged_decode_attention.  Every page is read once per pass; a pass carries
 * the (query, query head) pairs of a KV head, C = q_len * G in all:
 *     C <= 8 (bf16: 4), and f32: passes of 8 pairs (bf16: 4), the CTA's
 *     warps reading different pages;
 *     otherwise teams of warps reading every page together, each warp a
 *     share of the pairs: f16 passes of 16 (C <= 16) or 32 (four warps);
 *     q8_0 passes of 16 (C <= 16, two warps) or 32 (four warps); bf16 one
 *     pass for C <= 8 (two warps), passes of 16 beyond (four warps);
 * each pass one launch on `stream`.  pkv_decode_step_mq stores the new tokens
 * in the first pass, just before their pages are read; the last q_len
 * positions' pages must not be shared with another row.
 * Workspace (paged_decode_workspace_bytes_mq): as paged_decode_attention's
 * with 32 partial-state columns per slot instead of G and 4 counters per
 * (row, KV head):
 *     counters int32 [num_rows * n_kv_heads * 4]
 *     part_ml  float [S][32][2];  part_acc float [S][32][head_dim]
 * zero-filled once before first use; not shared by concurrent calls. */
#define PKV_MAX_Q_LEN 64

size_t paged_decode_workspace_bytes_mq(int max_rows, int n_q_heads, int n_kv_heads, int head_dim,
                                       int num_chunks);

/* Chunks (resident CTAs of the several-query kernel that q_len selects) that
 * fill this GPU. */
pkv_status paged_decode_default_chunks_mq(const pkv_pool *pool, int n_q_heads, int max_rows,
                                          int q_len, int *chunks);

pkv_status paged_decode_attention_mq(const pkv_pool *pool, int layer, const float *q,
                                     const int32_t *block_table, int bt_stride,
                                     const int32_t *seq_lens, int num_rows, int q_len,
                                     int n_q_heads, float scale, float *out, void *workspace,
                                     size_t workspace_bytes, int num_chunks, void *stream);

pkv_status pkv_decode_step_mq(const pkv_pool *pool, int layer, const float *q, const float *k_new,
                              const float *v_new, const int32_t *block_table, int bt_stride,
                              const int32_t *seq_lens, int num_rows, int q_len, int n_q_heads,
                              float scale, float *out, void *workspace, size_t workspace_bytes,
                              int num_chunks, void *stream);

/* Bytes of scratch held by paged_decode_attention_static (per GPU that
 * loads the library, for the life of the process). */
#define PKV_STATIC_SCRATCH_BYTES (8u << 20)

/* paged_decode_attention_static — paged_decode_attention for callers that
 * cannot allocate device memory when they decode: a serving process whose
 * device memory is all reserved up front by its KV pool and caching
 * allocator, or code where a cudaMalloc is not allowed or would stall the
 * device.  The pages describe no such entry point; it has no counterpart
 * there.  Same arguments as paged_decode_attention without the workspace:
 * the scratch is a PKV_STATIC_SCRATCH_BYTES array inside the library, and
 * the call allocates and frees nothing.
 *   - Calls whose paged_decode_workspace_bytes(num_rows, n_q_heads, n_kv,
 *     128, num_chunks) exceed PKV_STATIC_SCRATCH_BYTES return
 *     PKV_ERR_WORKSPACE (for example, with G = 4 and the default chunks of
 *     a GB300, a few hundred rows of 8 KV heads fit).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept with the id of the
 *     CUDA context it belongs to: after a device reset, the first call in
 *     the new context looks it up again (also before any capture).
 *   - Every argument is checked as paged_decode_attention checks it before
 *     the array is touched, so a rejected call leaves it as it was.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's partial states; each call clears the arrival counters first
 *     (one cudaMemsetAsync on `stream`).  Calls that overlap on the GPU
 *     (other streams, other host threads) race on it: serialise them. */
pkv_status paged_decode_attention_static(const pkv_pool *pool, int layer, const float *q,
                                         const int32_t *block_table, int bt_stride,
                                         const int32_t *seq_lens, int num_rows, int n_q_heads,
                                         float scale, float *out, int num_chunks, void *stream);

/* Name of a status code ("PKV_OK", ...). */
const char *pkv_status_string(pkv_status status);

/* One-line reason for the calling thread's last failed call ("" if none). */
const char *pkv_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */

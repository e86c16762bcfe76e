/* pkv_alloc.h — host-side page allocator for the paged KV pool of libpkv.so.
 *
 * The ownership side of the pool (tinyllm, "The repository currently
 * provides": one runner-owned physical KV page pool, a worker-owned allocator
 * and a logical block table per active sequence, with deterministic
 * reserve/commit/release; "Known limitations": 16-token pages, only complete
 * pages are shared and a non-aligned suffix is recomputed; Leone, "What
 * ships" and the introduction: page-rounded KV admission that returns typed
 * overload errors before the configured capacity is exceeded, forked
 * generation sessions).
 *
 * Model.  The allocator owns page ids 0 .. num_pages - 1 of a pool (the same
 * ids for every layer) and up to max_seqs sequences.  A sequence holds an
 * ordered list of pages (its block table), `committed` tokens written and
 * `reserved` further token slots it may write.  Its page count is always
 * ceil((committed + reserved) / 16).  A page has a reference count: the
 * number of sequences holding it; it is free at 0.
 *
 *   reserve(s, n)    make room for n more tokens: take the pages
 *                    ceil((committed + reserved + n) / 16) needs beyond those
 *                    s holds, lowest free ids first, appended in increasing
 *                    id order; all or nothing: if the pool has too few free
 *                    pages, or s would exceed max_pages_per_seq, nothing
 *                    changes and PKV_ERR_CAPACITY is returned.
 *   commit(s, n)     n <= reserved of the reserved slots now hold tokens:
 *                    committed += n, reserved -= n.
 *   unreserve(s, n)  n <= reserved slots are given back (for example the
 *                    rejected tokens of a speculative step): reserved -= n,
 *                    and the pages past ceil((committed + reserved) / 16) are
 *                    released.
 *   fork(p, &c)      a new sequence c sharing p's complete committed pages:
 *                    the first floor(committed_p / 16) pages of p, each
 *                    referenced once more; committed_c = 16 * that count,
 *                    reserved_c = 0.  The rest of p's tokens (a non-aligned
 *                    suffix) are not shared: the caller writes them again.
 *                    Shared pages are full and committed, so no sequence
 *                    ever writes into one.
 *   release(s)       every page of s is referenced once less (freed at 0);
 *                    s is closed and its id may be reused.
 *
 * Sequence ids: open() and fork() return the lowest closed id.  All results
 * are deterministic functions of the call sequence.  Not thread-safe: one
 * owner (the scheduler thread) calls it.  No device memory is touched; the
 * block tables it writes are host arrays the caller copies to the device.
 * Status codes are those of pkv.h: PKV_ERR_INVALID_ARG for a null pointer,
 * an id that is not open, a negative count or n > reserved;
 * PKV_ERR_CAPACITY as above. */
#ifndef PKV_ALLOC_H
#define PKV_ALLOC_H

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_alloc pkv_alloc;

/* num_pages, max_seqs, max_pages_per_seq >= 1.  *out gets an allocator with
 * every page free and no sequence open. */
pkv_status pkv_alloc_create(pkv_alloc **out, int num_pages, int max_seqs, int max_pages_per_seq);
void pkv_alloc_destroy(pkv_alloc *a); /* NULL is allowed */

pkv_status pkv_alloc_open(pkv_alloc *a, int *seq);
pkv_status pkv_alloc_reserve(pkv_alloc *a, int seq, int n_tokens);
pkv_status pkv_alloc_commit(pkv_alloc *a, int seq, int n_tokens);
pkv_status pkv_alloc_unreserve(pkv_alloc *a, int seq, int n_tokens);
pkv_status pkv_alloc_fork(pkv_alloc *a, int parent, int *child);
pkv_status pkv_alloc_release(pkv_alloc *a, int seq);

/* The same for a batch: reserve_many gives each of seqs[0 .. num_seqs) n_tokens
 * more token slots, or nobody any (a refused admission changes nothing:
 * PKV_ERR_CAPACITY or PKV_ERR_INVALID_ARG); commit_many commits n_tokens for
 * each (all validated first).  A sequence may appear once per call. */
pkv_status pkv_alloc_reserve_many(pkv_alloc *a, const int *seqs, int num_seqs, int n_tokens);
pkv_status pkv_alloc_commit_many(pkv_alloc *a, const int *seqs, int num_seqs, int n_tokens);

/* committed and reserved token counts and page count of an open sequence
 * (any output pointer may be NULL). */
pkv_status pkv_alloc_seq_info(const pkv_alloc *a, int seq, int *committed, int *reserved,
                              int *pages);

/* The block table of `seq` into row[0 .. stride): its page ids in order, then
 * -1.  stride must be at least its page count (else PKV_ERR_INVALID_ARG). */
pkv_status pkv_alloc_block_table(const pkv_alloc *a, int seq, int32_t *row, int stride);

/* Block tables and attention lengths of a decode batch: row r of
 * block_table (stride bt_stride) gets seqs[r]'s table and seq_lens[r] =
 * committed + extra, the length a step that writes `extra` of its reserved
 * tokens attends over (extra <= reserved for every row, else
 * PKV_ERR_INVALID_ARG and nothing is written). */
pkv_status pkv_alloc_batch(const pkv_alloc *a, const int *seqs, int num_rows, int extra,
                           int32_t *block_table, int bt_stride, int32_t *seq_lens);

/* Pages with reference count 0, >= 1 and >= 2 (any pointer may be NULL). */
pkv_status pkv_alloc_stats(const pkv_alloc *a, int *free_pages, int *used_pages,
                           int *shared_pages);

/* Reference count of one page (0 .. num_pages - 1). */
pkv_status pkv_alloc_page_refs(const pkv_alloc *a, int page, int *refs);

#ifdef __cplusplus
}
#endif

#endif /* PKV_ALLOC_H */

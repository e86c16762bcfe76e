// alloc.cu — the host page allocator declared in include/pkv_alloc.h (host
// code only; no device memory).
//
// Free page ids and closed sequence ids are kept in min-heaps, so "lowest id
// first" costs O(log n) per page; a sequence's pages are a vector in block
// table order.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <vector>

#include "pkv.h"
#include "pkv_alloc.h"
#include "pkv_internal.h"

namespace {

constexpr int kPage = PKV_PAGE_TOKENS;

using MinHeap = std::priority_queue<int, std::vector<int>, std::greater<int>>;

struct Seq {
  bool open = false;
  long long committed = 0;
  long long reserved = 0;
  std::vector<int32_t> pages;
};

long long pages_for(long long tokens) { return (tokens + kPage - 1) / kPage; }

}  // namespace

struct pkv_alloc {
  int num_pages;
  int max_pages_per_seq;
  std::vector<int> refs;  // per page
  MinHeap free_pages;
  std::vector<Seq> seqs;
  MinHeap closed;
  int shared = 0;  // pages with refs >= 2
  int used = 0;    // pages with refs >= 1
  std::vector<int> mark;  // per sequence id: the batch call that last named it
  int mark_gen = 0;

  void ref(int p) {
    if (refs[p] == 0) ++used;
    if (refs[p] == 1) ++shared;
    ++refs[p];
  }
  void unref(int p) {
    --refs[p];
    if (refs[p] == 1) --shared;
    if (refs[p] == 0) {
      --used;
      free_pages.push(p);
    }
  }
  Seq* get(int s) { return (s >= 0 && s < static_cast<int>(seqs.size()) && seqs[s].open) ? &seqs[s] : nullptr; }
  const Seq* get(int s) const {
    return (s >= 0 && s < static_cast<int>(seqs.size()) && seqs[s].open) ? &seqs[s] : nullptr;
  }
  // Release pages past ceil((committed + reserved) / 16).
  void trim(Seq& q) {
    const long long keep = pages_for(q.committed + q.reserved);
    while (static_cast<long long>(q.pages.size()) > keep) {
      unref(q.pages.back());
      q.pages.pop_back();
    }
  }
};

namespace {
pkv_status bad(const char* msg) { return pkv::record_error(PKV_ERR_INVALID_ARG, msg); }
}  // namespace

extern "C" {

pkv_status pkv_alloc_create(pkv_alloc** out, int num_pages, int max_seqs, int max_pages_per_seq) {
  if (!out) return bad("null output pointer");
  *out = nullptr;
  if (num_pages < 1 || max_seqs < 1 || max_pages_per_seq < 1)
    return bad("num_pages, max_seqs and max_pages_per_seq must be >= 1");
  pkv_alloc* a = new (std::nothrow) pkv_alloc();
  if (!a) return bad("out of host memory");
  try {
    a->num_pages = num_pages;
    a->max_pages_per_seq = max_pages_per_seq;
    a->refs.assign(num_pages, 0);
    std::vector<int> ids(num_pages);
    for (int p = 0; p < num_pages; ++p) ids[p] = p;
    a->free_pages = MinHeap(std::greater<int>(), std::move(ids));
    a->seqs.resize(max_seqs);
    std::vector<int> sids(max_seqs);
    for (int s = 0; s < max_seqs; ++s) sids[s] = s;
    a->closed = MinHeap(std::greater<int>(), std::move(sids));
    a->mark.assign(max_seqs, 0);
  } catch (...) {
    delete a;
    return bad("out of host memory");
  }
  *out = a;
  return PKV_OK;
}

void pkv_alloc_destroy(pkv_alloc* a) { delete a; }

pkv_status pkv_alloc_open(pkv_alloc* a, int* seq) {
  if (!a || !seq) return bad("null allocator or output pointer");
  if (a->closed.empty()) return pkv::record_error(PKV_ERR_CAPACITY, "every sequence id is open");
  const int s = a->closed.top();
  a->closed.pop();
  Seq& q = a->seqs[s];
  q.open = true;
  q.committed = q.reserved = 0;
  q.pages.clear();
  *seq = s;
  return PKV_OK;
}

pkv_status pkv_alloc_reserve(pkv_alloc* a, int seq, int n_tokens) {
  Seq* q = a ? a->get(seq) : nullptr;
  if (!q) return bad("sequence is not open");
  if (n_tokens < 0) return bad("negative token count");
  const long long need = pages_for(q->committed + q->reserved + n_tokens) -
                         static_cast<long long>(q->pages.size());
  if (static_cast<long long>(q->pages.size()) + need > a->max_pages_per_seq)
    return pkv::record_error(PKV_ERR_CAPACITY, "sequence would exceed max_pages_per_seq");
  if (need > static_cast<long long>(a->free_pages.size()))
    return pkv::record_error(PKV_ERR_CAPACITY, "not enough free pages in the pool");
  for (long long k = 0; k < need; ++k) {
    const int p = a->free_pages.top();
    a->free_pages.pop();
    a->ref(p);
    q->pages.push_back(p);
  }
  q->reserved += n_tokens;
  return PKV_OK;
}

pkv_status pkv_alloc_commit(pkv_alloc* a, int seq, int n_tokens) {
  Seq* q = a ? a->get(seq) : nullptr;
  if (!q) return bad("sequence is not open");
  if (n_tokens < 0 || n_tokens > q->reserved) return bad("commit count outside [0, reserved]");
  q->committed += n_tokens;
  q->reserved -= n_tokens;
  return PKV_OK;
}

pkv_status pkv_alloc_unreserve(pkv_alloc* a, int seq, int n_tokens) {
  Seq* q = a ? a->get(seq) : nullptr;
  if (!q) return bad("sequence is not open");
  if (n_tokens < 0 || n_tokens > q->reserved) return bad("unreserve count outside [0, reserved]");
  q->reserved -= n_tokens;
  a->trim(*q);
  return PKV_OK;
}

pkv_status pkv_alloc_fork(pkv_alloc* a, int parent, int* child) {
  if (!a || !child) return bad("null allocator or output pointer");
  const Seq* p = a->get(parent);
  if (!p) return bad("parent sequence is not open");
  if (a->closed.empty()) return pkv::record_error(PKV_ERR_CAPACITY, "every sequence id is open");
  const long long full = p->committed / kPage;  // complete committed pages
  const int c = a->closed.top();
  a->closed.pop();
  Seq& q = a->seqs[c];
  const Seq& par = a->seqs[parent];  // re-read: seqs does not reallocate
  q.open = true;
  q.committed = full * kPage;
  q.reserved = 0;
  q.pages.assign(par.pages.begin(), par.pages.begin() + full);
  for (int32_t pg : q.pages) a->ref(pg);
  *child = c;
  return PKV_OK;
}

pkv_status pkv_alloc_release(pkv_alloc* a, int seq) {
  Seq* q = a ? a->get(seq) : nullptr;
  if (!q) return bad("sequence is not open");
  for (int32_t pg : q->pages) a->unref(pg);
  q->pages.clear();
  q->committed = q->reserved = 0;
  q->open = false;
  a->closed.push(seq);
  return PKV_OK;
}

pkv_status pkv_alloc_reserve_many(pkv_alloc* a, const int* seqs, int num_seqs, int n_tokens) {
  if (!a || (num_seqs > 0 && !seqs)) return bad("null argument");
  if (num_seqs < 0 || n_tokens < 0) return bad("negative count");
  const int gen = ++a->mark_gen;
  for (int r = 0; r < num_seqs; ++r) {
    if (!a->get(seqs[r])) return bad("sequence is not open");
    if (a->mark[seqs[r]] == gen) return bad("a sequence appears twice");
    a->mark[seqs[r]] = gen;
  }
  for (int r = 0; r < num_seqs; ++r) {
    const pkv_status st = pkv_alloc_reserve(a, seqs[r], n_tokens);
    if (st != PKV_OK) {  // give back what the earlier rows took: nothing changes
      for (int u = 0; u < r; ++u) pkv_alloc_unreserve(a, seqs[u], n_tokens);
      return st;
    }
  }
  return PKV_OK;
}

pkv_status pkv_alloc_commit_many(pkv_alloc* a, const int* seqs, int num_seqs, int n_tokens) {
  if (!a || (num_seqs > 0 && !seqs)) return bad("null argument");
  if (num_seqs < 0 || n_tokens < 0) return bad("negative count");
  const int gen = ++a->mark_gen;
  for (int r = 0; r < num_seqs; ++r) {
    const Seq* q = a->get(seqs[r]);
    if (!q) return bad("sequence is not open");
    if (n_tokens > q->reserved) return bad("commit count above a sequence's reserved tokens");
    if (a->mark[seqs[r]] == gen) return bad("a sequence appears twice");
    a->mark[seqs[r]] = gen;
  }
  for (int r = 0; r < num_seqs; ++r) pkv_alloc_commit(a, seqs[r], n_tokens);
  return PKV_OK;
}

pkv_status pkv_alloc_seq_info(const pkv_alloc* a, int seq, int* committed, int* reserved,
                              int* pages) {
  const Seq* q = a ? a->get(seq) : nullptr;
  if (!q) return bad("sequence is not open");
  if (committed) *committed = static_cast<int>(q->committed);
  if (reserved) *reserved = static_cast<int>(q->reserved);
  if (pages) *pages = static_cast<int>(q->pages.size());
  return PKV_OK;
}

pkv_status pkv_alloc_block_table(const pkv_alloc* a, int seq, int32_t* row, int stride) {
  const Seq* q = a ? a->get(seq) : nullptr;
  if (!q) return bad("sequence is not open");
  if (!row) return bad("null block-table row");
  if (stride < static_cast<long long>(q->pages.size())) return bad("stride below the page count");
  const size_t n = q->pages.size();
  if (n) std::memcpy(row, q->pages.data(), n * sizeof(int32_t));
  std::fill(row + n, row + stride, -1);
  return PKV_OK;
}

pkv_status pkv_alloc_batch(const pkv_alloc* a, const int* seqs, int num_rows, int extra,
                           int32_t* block_table, int bt_stride, int32_t* seq_lens) {
  if (!a || (num_rows > 0 && (!seqs || !block_table || !seq_lens))) return bad("null argument");
  if (num_rows < 0 || extra < 0) return bad("negative row count or extra");
  for (int r = 0; r < num_rows; ++r) {  // validate everything before writing
    const Seq* q = a->get(seqs[r]);
    if (!q) return bad("batch names a sequence that is not open");
    if (extra > q->reserved) return bad("extra exceeds a sequence's reserved tokens");
    if (bt_stride < static_cast<long long>(q->pages.size()))
      return bad("bt_stride below a sequence's page count");
  }
  for (int r = 0; r < num_rows; ++r) {
    const Seq* q = a->get(seqs[r]);
    pkv_alloc_block_table(a, seqs[r], block_table + static_cast<long long>(r) * bt_stride,
                          bt_stride);
    seq_lens[r] = static_cast<int32_t>(q->committed + extra);
  }
  return PKV_OK;
}

pkv_status pkv_alloc_stats(const pkv_alloc* a, int* free_pages, int* used_pages,
                           int* shared_pages) {
  if (!a) return bad("null allocator");
  if (free_pages) *free_pages = a->num_pages - a->used;
  if (used_pages) *used_pages = a->used;
  if (shared_pages) *shared_pages = a->shared;
  return PKV_OK;
}

pkv_status pkv_alloc_page_refs(const pkv_alloc* a, int page, int* refs) {
  if (!a || !refs) return bad("null argument");
  if (page < 0 || page >= a->num_pages) return bad("page outside the pool");
  *refs = a->refs[page];
  return PKV_OK;
}

}  // extern "C"

// Host side of the paged KV cache: block tables, lengths, reference counts
// and the free list of a pool of pages ("efficient-attention/flash-2-3",
// section "Paged KV caches, a preview of serving": a new page is taken from
// the free list only when a sequence's last page fills; sequences that share
// a prompt share its pages and copy one only when they would write to it).
//
// The free list is a stack: pages start as n-1, ..., 1, 0 (page 0 is taken
// first) and a released page is pushed on top.  Only a sequence's last page
// is ever written, so only it is copied; the device work of an append (the
// copy, then the token) is fa_paged_append.  A batch of appends is checked
// as a whole first: if the pool cannot hold it, nothing changes.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "fa.h"

struct fa_page_pool {
  int num_pages;
  int page_size;
  int max_seqs;
  int max_blocks;
  std::vector<int> free_list;            // stack of free pages
  std::vector<int> ref;                  // [num_pages] tables that hold the page
  std::vector<std::vector<int>> tables;  // [max_seqs] logical block -> page
  std::vector<int> lens;                 // [max_seqs] tokens
  std::vector<char> live;                // [max_seqs] slot in use
};

namespace {

bool valid_seq(const fa_page_pool* p, int s) { return p && s >= 0 && s < p->max_seqs && p->live[s]; }

int take_page(fa_page_pool* p) {
  const int page = p->free_list.back();
  p->free_list.pop_back();
  p->ref[page] = 1;
  return page;
}

}  // namespace

extern "C" {

fa_page_pool* fa_pool_create(int num_pages, int page_size, int max_seqs, int max_blocks) {
  if (num_pages < 1 || page_size < 1 || max_seqs < 1 || max_blocks < 1) return nullptr;
  fa_page_pool* p = new (std::nothrow) fa_page_pool;
  if (!p) return nullptr;
  try {
    p->num_pages = num_pages;
    p->page_size = page_size;
    p->max_seqs = max_seqs;
    p->max_blocks = max_blocks;
    p->free_list.resize(num_pages);
    for (int i = 0; i < num_pages; ++i) p->free_list[i] = num_pages - 1 - i;
    p->ref.assign(num_pages, 0);
    p->tables.assign(max_seqs, std::vector<int>());
    p->lens.assign(max_seqs, 0);
    p->live.assign(max_seqs, 0);
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void fa_pool_destroy(fa_page_pool* pool) { delete pool; }

int fa_pool_free_pages(const fa_page_pool* pool) { return pool ? (int)pool->free_list.size() : -1; }

int fa_pool_refcount(const fa_page_pool* pool, int page) {
  return (pool && page >= 0 && page < pool->num_pages) ? pool->ref[page] : -1;
}

fa_status fa_pool_add_seq(fa_page_pool* pool, int* seq) {
  if (!pool || !seq) return FA_ERR_INVALID_ARG;
  for (int s = 0; s < pool->max_seqs; ++s) {
    if (!pool->live[s]) {
      pool->live[s] = 1;
      pool->tables[s].clear();
      pool->lens[s] = 0;
      *seq = s;
      return FA_OK;
    }
  }
  return FA_ERR_OUT_OF_PAGES;
}

fa_status fa_pool_fork(fa_page_pool* pool, int parent, int* child) {
  if (!valid_seq(pool, parent) || !child) return FA_ERR_INVALID_ARG;
  int c = -1;
  const fa_status st = fa_pool_add_seq(pool, &c);
  if (st != FA_OK) return st;
  try {
    pool->tables[c] = pool->tables[parent];
  } catch (...) {  // host memory: undo the slot
    pool->live[c] = 0;
    return FA_ERR_OUT_OF_PAGES;
  }
  pool->lens[c] = pool->lens[parent];
  for (int page : pool->tables[c]) ++pool->ref[page];
  *child = c;
  return FA_OK;
}

fa_status fa_pool_release(fa_page_pool* pool, int seq) {
  if (!valid_seq(pool, seq)) return FA_ERR_INVALID_ARG;
  for (int page : pool->tables[seq]) {
    if (--pool->ref[page] == 0) pool->free_list.push_back(page);
  }
  pool->tables[seq].clear();
  pool->lens[seq] = 0;
  pool->live[seq] = 0;
  return FA_OK;
}

static fa_status reserve_append(fa_page_pool* pool, const int* seqs, int n, int* page, int* slot, int* copy_src) {
  // the whole batch first: valid, distinct sequences, room in the tables and in the pool
  std::vector<char> seen(pool->max_seqs, 0);
  std::unordered_map<int, int> writers;  // shared last page -> members of the batch that write it
  long long need = 0;
  for (int i = 0; i < n; ++i) {
    const int s = seqs[i];
    if (!valid_seq(pool, s) || seen[s]) return FA_ERR_INVALID_ARG;
    seen[s] = 1;
    const int L = pool->lens[s];
    if (L % pool->page_size == 0) {
      if ((int)pool->tables[s].size() >= pool->max_blocks) return FA_ERR_INVALID_ARG;
      ++need;
    } else if (pool->ref[pool->tables[s].back()] > 1) {
      ++writers[pool->tables[s].back()];
    }
  }
  // m writers of a page held r times copy it min(m, r - 1) times: the last holder writes in place
  for (const auto& kv : writers) {
    const int r = pool->ref[kv.first];
    need += kv.second < r - 1 ? kv.second : r - 1;
  }
  if (need > (long long)pool->free_list.size()) return FA_ERR_OUT_OF_PAGES;
  for (int i = 0; i < n; ++i) {
    const int s = seqs[i];
    std::vector<int>& t = pool->tables[s];
    const int L = pool->lens[s];
    int src = -1;
    if (L % pool->page_size == 0) {
      t.push_back(take_page(pool));
    } else if (pool->ref[t.back()] > 1) {
      const int fresh = take_page(pool);
      --pool->ref[t.back()];
      src = t.back();
      t.back() = fresh;
    }
    pool->lens[s] = L + 1;
    page[i] = t.back();
    slot[i] = L % pool->page_size;
    copy_src[i] = src;
  }
  return FA_OK;
}

fa_status fa_pool_reserve_append(fa_page_pool* pool, const int* seqs, int n, int* page, int* slot, int* copy_src) {
  if (!pool || n < 0 || (n > 0 && (!seqs || !page || !slot || !copy_src))) return FA_ERR_INVALID_ARG;
  // every table can hold max_blocks pages: reserve that up front so that the
  // commit loop below never allocates (and so never fails half way)
  try {
    for (int i = 0; i < n; ++i)
      if (valid_seq(pool, seqs[i])) pool->tables[seqs[i]].reserve(pool->max_blocks);
    return reserve_append(pool, seqs, n, page, slot, copy_src);
  } catch (...) {
    return FA_ERR_OUT_OF_PAGES;  // host memory for the checks; nothing was changed
  }
}

fa_status fa_pool_export(const fa_page_pool* pool, int* block_table, int* seq_lens) {
  if (!pool || !block_table || !seq_lens) return FA_ERR_INVALID_ARG;
  for (int s = 0; s < pool->max_seqs; ++s) {
    const std::vector<int>& t = pool->tables[s];
    for (int j = 0; j < pool->max_blocks; ++j) block_table[(size_t)s * pool->max_blocks + j] = j < (int)t.size() ? t[j] : 0;
    seq_lens[s] = pool->lens[s];
  }
  return FA_OK;
}

}  // extern "C"

// Host block manager: LIFO free list, per-page reference counts, per-sequence
// page tables, fork and copy-on-write.
//
// "PagedAttention原理" (vLLM long-sequence memory guide, ch. 3):
//   §3.3.2 -- a request starts with one page; a new page is taken from the free
//            list when the current one is full; the pages of a finished request
//            return to the free list.
//   §3.3.4 -- the free list is used as a stack: take from the end, return to the
//            end in page-table order; an empty free list is an out-of-memory error.
//   §3.3.3 and the pitfall note after §3.3.4 -- shared pages carry a reference
//            count and are only returned when it reaches zero.
// "mlx-paged-attention", feature 2 -- a shared page is copied only when one of
// its holders writes to it.
// "PagedAttention MLX：为Apple Silicon打造的高吞吐量LLM推理引擎" (dynamic
// scheduling; physical KV pool) -- the pages of an inactive request can be
// swapped out to CPU memory and back: a whole sequence moves to blocks of a host
// pool (LIFO host free list) and returns to fresh device pages.
//
// The state is plain vectors plus a hash map from sequence id to its record; all
// operations are O(1) except fork and free (O(pages of the sequence)).
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Sequence {
  std::vector<int32_t> pages;       // device pages, or host blocks while swapped
  int64_t length = 0;
  bool swapped = false;
};

}  // namespace

struct pa_bm {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_list;   // top of the stack is the back
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, Sequence> seqs;
  int32_t num_host_blocks = 0;      // 0: swapping not enabled
  std::vector<int32_t> host_free;   // top of the stack is the back
};

namespace {

// Reserve one token slot for `s`.  Returns PA_ERR_OUT_OF_BLOCKS (state
// untouched) when a page is needed and none is free.
int append_one(pa_bm* bm, Sequence& s, int64_t* slot, int64_t* cow_src, int64_t* cow_dst) {
  const int64_t index = s.length / bm->block_size;
  const int64_t offset = s.length % bm->block_size;
  int64_t src = -1, dst = -1;
  int32_t page;
  if (index == static_cast<int64_t>(s.pages.size())) {
    if (bm->free_list.empty()) return PA_ERR_OUT_OF_BLOCKS;
    page = bm->free_list.back();
    bm->free_list.pop_back();
    bm->refcount[page] = 1;
    s.pages.push_back(page);
  } else {
    page = s.pages[static_cast<size_t>(index)];
    if (bm->refcount[page] > 1) {
      if (bm->free_list.empty()) return PA_ERR_OUT_OF_BLOCKS;
      const int32_t fresh = bm->free_list.back();
      bm->free_list.pop_back();
      bm->refcount[fresh] = 1;
      bm->refcount[page] -= 1;
      s.pages[static_cast<size_t>(index)] = fresh;
      src = page;
      dst = fresh;
      page = fresh;
    }
  }
  s.length += 1;
  *slot = static_cast<int64_t>(page) * bm->block_size + offset;
  *cow_src = src;
  *cow_dst = dst;
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_bm_create(int num_blocks, int block_size, const int32_t* initial_free_order, pa_bm** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  pa_bm* bm = new (std::nothrow) pa_bm;
  if (!bm) return PA_ERR_INVALID_ARG;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
  bm->free_list.resize(static_cast<size_t>(num_blocks));
  if (initial_free_order) {
    std::vector<uint8_t> seen(static_cast<size_t>(num_blocks), 0);
    for (int i = 0; i < num_blocks; ++i) {
      const int32_t p = initial_free_order[i];
      if (p < 0 || p >= num_blocks || seen[static_cast<size_t>(p)]) {
        delete bm;
        return PA_ERR_INVALID_ARG;  // not a permutation of the pool
      }
      seen[static_cast<size_t>(p)] = 1;
      bm->free_list[static_cast<size_t>(i)] = p;
    }
  } else {
    for (int i = 0; i < num_blocks; ++i) bm->free_list[static_cast<size_t>(i)] = i;
  }
  *out = bm;
  return PA_OK;
}

void pa_bm_destroy(pa_bm* bm) { delete bm; }

int pa_bm_add_seq(pa_bm* bm, int64_t seq_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  if (bm->seqs.count(seq_id)) return PA_ERR_EXISTS;
  if (bm->free_list.empty()) return PA_ERR_OUT_OF_BLOCKS;
  const int32_t page = bm->free_list.back();
  bm->free_list.pop_back();
  bm->refcount[page] = 1;
  Sequence& s = bm->seqs[seq_id];
  s.pages.push_back(page);
  s.length = 0;
  return PA_OK;
}

int pa_bm_append_slot(pa_bm* bm, int64_t seq_id, int64_t* slot, int64_t* cow_src,
                      int64_t* cow_dst) {
  if (!bm || !slot || !cow_src || !cow_dst) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  if (it->second.swapped) return PA_ERR_SWAPPED;
  return append_one(bm, it->second, slot, cow_src, cow_dst);
}

int pa_bm_fork(pa_bm* bm, int64_t parent, int64_t child) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  if (it->second.swapped) return PA_ERR_SWAPPED;
  if (bm->seqs.count(child)) return PA_ERR_EXISTS;
  Sequence copy = it->second;
  for (int32_t p : copy.pages) bm->refcount[p] += 1;
  bm->seqs.emplace(child, std::move(copy));
  return PA_OK;
}

int pa_bm_free(pa_bm* bm, int64_t seq_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  if (it->second.swapped) {                  // its host blocks go back
    for (int32_t h : it->second.pages) bm->host_free.push_back(h);
  } else {
    for (int32_t p : it->second.pages) {
      bm->refcount[p] -= 1;
      if (bm->refcount[p] == 0) bm->free_list.push_back(p);
    }
  }
  bm->seqs.erase(it);
  return PA_OK;
}

int pa_bm_enable_swap(pa_bm* bm, int num_host_blocks, const int32_t* initial_host_order) {
  if (!bm || num_host_blocks <= 0 || bm->num_host_blocks != 0) return PA_ERR_INVALID_ARG;
  std::vector<int32_t> order(static_cast<size_t>(num_host_blocks));
  if (initial_host_order) {
    std::vector<uint8_t> seen(static_cast<size_t>(num_host_blocks), 0);
    for (int i = 0; i < num_host_blocks; ++i) {
      const int32_t h = initial_host_order[i];
      if (h < 0 || h >= num_host_blocks || seen[static_cast<size_t>(h)])
        return PA_ERR_INVALID_ARG;                 // not a permutation of the host pool
      seen[static_cast<size_t>(h)] = 1;
      order[static_cast<size_t>(i)] = h;
    }
  } else {
    for (int i = 0; i < num_host_blocks; ++i) order[static_cast<size_t>(i)] = i;
  }
  bm->host_free = std::move(order);
  bm->num_host_blocks = num_host_blocks;
  return PA_OK;
}

int pa_bm_swap_out(pa_bm* bm, int64_t seq_id, int64_t* pairs, int cap, int* num_pairs) {
  if (!bm || !num_pairs || cap < 0 || (cap > 0 && !pairs)) return PA_ERR_INVALID_ARG;
  if (bm->num_host_blocks == 0) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  Sequence& s = it->second;
  if (s.swapped) return PA_ERR_SWAPPED;
  const size_t n = s.pages.size();
  if (cap < static_cast<int>(n)) return PA_ERR_INVALID_ARG;
  if (bm->host_free.size() < n) return PA_ERR_OUT_OF_BLOCKS;
  for (size_t i = 0; i < n; ++i) {
    const int32_t h = bm->host_free.back();
    bm->host_free.pop_back();
    pairs[2 * i] = s.pages[i];
    pairs[2 * i + 1] = h;
  }
  for (size_t i = 0; i < n; ++i) {          // drop the device references, table order
    const int32_t p = s.pages[i];
    bm->refcount[p] -= 1;
    if (bm->refcount[p] == 0) bm->free_list.push_back(p);
    s.pages[i] = static_cast<int32_t>(pairs[2 * i + 1]);
  }
  s.swapped = true;
  *num_pairs = static_cast<int>(n);
  return PA_OK;
}

int pa_bm_swap_in(pa_bm* bm, int64_t seq_id, int64_t* pairs, int cap, int* num_pairs) {
  if (!bm || !num_pairs || cap < 0 || (cap > 0 && !pairs)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  Sequence& s = it->second;
  if (!s.swapped) return PA_ERR_INVALID_ARG;
  const size_t n = s.pages.size();
  if (cap < static_cast<int>(n)) return PA_ERR_INVALID_ARG;
  if (bm->free_list.size() < n) return PA_ERR_OUT_OF_BLOCKS;
  for (size_t i = 0; i < n; ++i) {
    const int32_t p = bm->free_list.back();
    bm->free_list.pop_back();
    bm->refcount[p] = 1;
    pairs[2 * i] = s.pages[i];
    pairs[2 * i + 1] = p;
  }
  for (size_t i = 0; i < n; ++i) {          // host blocks back, table order
    bm->host_free.push_back(s.pages[i]);
    s.pages[i] = static_cast<int32_t>(pairs[2 * i + 1]);
  }
  s.swapped = false;
  *num_pairs = static_cast<int>(n);
  return PA_OK;
}

int pa_bm_num_free_host(const pa_bm* bm) {
  if (!bm) return PA_ERR_INVALID_ARG;
  return static_cast<int>(bm->host_free.size());
}

int pa_bm_host_free_list(const pa_bm* bm, int32_t* out, int cap) {
  if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  const int n = static_cast<int>(bm->host_free.size());
  for (int i = 0; i < n && i < cap; ++i) out[i] = bm->host_free[static_cast<size_t>(i)];
  return n;
}

int pa_bm_block_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int cap, int* num_pages,
                      int* length) {
  if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  const Sequence& s = it->second;
  if (s.swapped) return PA_ERR_SWAPPED;
  const int n = static_cast<int>(s.pages.size());
  for (int i = 0; i < n && i < cap; ++i) out[i] = s.pages[static_cast<size_t>(i)];
  if (num_pages) *num_pages = n;
  if (length) *length = static_cast<int>(s.length);
  return PA_OK;
}

int pa_bm_refcount(const pa_bm* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return PA_ERR_INVALID_ARG;
  return bm->refcount[static_cast<size_t>(block)];
}

int pa_bm_num_free(const pa_bm* bm) {
  if (!bm) return PA_ERR_INVALID_ARG;
  return static_cast<int>(bm->free_list.size());
}

int pa_bm_free_list(const pa_bm* bm, int32_t* out, int cap) {
  if (!bm || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  const int n = static_cast<int>(bm->free_list.size());
  for (int i = 0; i < n && i < cap; ++i) out[i] = bm->free_list[static_cast<size_t>(i)];
  return n;
}

int pa_bm_stats(const pa_bm* bm, int64_t* out4) {
  if (!bm || !out4) return PA_ERR_INVALID_ARG;
  int64_t used = 0, shared = 0, waste = 0;
  for (int32_t r : bm->refcount) {
    used += r > 0;
    shared += r > 1;
  }
  for (const auto& kv : bm->seqs)
    if (!kv.second.swapped)
      waste += static_cast<int64_t>(kv.second.pages.size()) * bm->block_size - kv.second.length;
  out4[0] = used;
  out4[1] = static_cast<int64_t>(bm->free_list.size());
  out4[2] = shared;
  out4[3] = waste;
  return PA_OK;
}

int pa_bm_append_slots(pa_bm* bm, const int64_t* seq_ids, int n, int64_t* slots,
                       int64_t* cow_pairs, int* num_cow, int* num_done) {
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots || !cow_pairs)) || !num_cow)
    return PA_ERR_INVALID_ARG;
  *num_cow = 0;
  if (num_done) *num_done = 0;
  for (int j = 0; j < n; ++j) {
    auto it = bm->seqs.find(seq_ids[j]);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    if (it->second.swapped) return PA_ERR_SWAPPED;
    int64_t src, dst;
    const int rc = append_one(bm, it->second, &slots[j], &src, &dst);
    if (rc != PA_OK) return rc;
    if (src >= 0) {
      cow_pairs[2 * *num_cow] = src;
      cow_pairs[2 * *num_cow + 1] = dst;
      *num_cow += 1;
    }
    if (num_done) *num_done = j + 1;
  }
  return PA_OK;
}

int pa_bm_build_block_tables(const pa_bm* bm, const int64_t* seq_ids, int n, int32_t* tables,
                             int max_blocks, int32_t* context_lens) {
  if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !tables || !context_lens)))
    return PA_ERR_INVALID_ARG;
  for (int j = 0; j < n; ++j) {
    auto it = bm->seqs.find(seq_ids[j]);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    const Sequence& s = it->second;
    if (s.swapped) return PA_ERR_SWAPPED;
    if (static_cast<int>(s.pages.size()) > max_blocks) return PA_ERR_INVALID_ARG;
    int32_t* row = tables + static_cast<size_t>(j) * max_blocks;
    int i = 0;
    for (; i < static_cast<int>(s.pages.size()); ++i) row[i] = s.pages[static_cast<size_t>(i)];
    for (; i < max_blocks; ++i) row[i] = -1;
    context_lens[j] = static_cast<int32_t>(s.length);
  }
  return PA_OK;
}

}  // extern "C"

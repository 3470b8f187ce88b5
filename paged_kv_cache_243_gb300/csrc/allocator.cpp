// Host page allocator [HBM-layout page, section 三: allocate_blocks takes
// ceil(tokens / block_size) blocks from a free list and fails (None) when the
// list is short; free_sequence returns a sequence's blocks to the list].
// Pages leave the free list from the front and return to its back, so the
// allocation order is deterministic.
#include <deque>
#include <unordered_map>
#include <vector>

#include "pkv.h"

struct pkv_allocator {
  int32_t num_pages = 0;
  std::deque<int32_t> free_list;
  std::unordered_map<int64_t, std::vector<int32_t>> owned;
};

extern "C" {

pkv_status pkv_alloc_create(int32_t num_pages, pkv_allocator** out) {
  if (!out || num_pages < 0) return PKV_ERR_INVALID_ARG;
  pkv_allocator* a = new pkv_allocator();
  a->num_pages = num_pages;
  for (int32_t i = 0; i < num_pages; ++i) a->free_list.push_back(i);
  *out = a;
  return PKV_OK;
}

void pkv_alloc_destroy(pkv_allocator* a) { delete a; }

pkv_status pkv_alloc_reserve(pkv_allocator* a, int64_t seq_id, int32_t total_tokens,
                             int32_t page_size, int32_t* block_table_row, int32_t max_pages) {
  if (!a || total_tokens < 0 || page_size <= 0 || max_pages < 0) return PKV_ERR_INVALID_ARG;
  if (max_pages > 0 && !block_table_row) return PKV_ERR_INVALID_ARG;
  const int64_t need = ((int64_t)total_tokens + page_size - 1) / page_size;
  if (need > max_pages) return PKV_ERR_INVALID_ARG;
  auto it = a->owned.find(seq_id);
  const int64_t have = it == a->owned.end() ? 0 : (int64_t)it->second.size();
  const int64_t extra = need > have ? need - have : 0;
  if (extra > (int64_t)a->free_list.size()) return PKV_ERR_OUT_OF_PAGES;
  std::vector<int32_t>& pages = a->owned[seq_id];
  for (int64_t i = 0; i < extra; ++i) {
    pages.push_back(a->free_list.front());
    a->free_list.pop_front();
  }
  for (int32_t i = 0; i < max_pages; ++i)
    block_table_row[i] = i < (int32_t)pages.size() ? pages[i] : -1;
  return PKV_OK;
}

pkv_status pkv_alloc_free(pkv_allocator* a, int64_t seq_id) {
  if (!a) return PKV_ERR_INVALID_ARG;
  auto it = a->owned.find(seq_id);
  if (it == a->owned.end()) return PKV_ERR_INVALID_ARG;
  for (int32_t pg : it->second) a->free_list.push_back(pg);
  a->owned.erase(it);
  return PKV_OK;
}

int32_t pkv_alloc_num_free(const pkv_allocator* a) { return a ? (int32_t)a->free_list.size() : 0; }

int32_t pkv_alloc_seq_pages(const pkv_allocator* a, int64_t seq_id) {
  if (!a) return 0;
  auto it = a->owned.find(seq_id);
  return it == a->owned.end() ? 0 : (int32_t)it->second.size();
}

int32_t pkv_alloc_check(const pkv_allocator* a) {
  if (!a) return 0;
  std::vector<int32_t> refs(a->num_pages, 0);
  int32_t bad = 0;
  auto mark = [&](int32_t pg) {
    if (pg < 0 || pg >= a->num_pages) ++bad;
    else ++refs[pg];
  };
  for (int32_t pg : a->free_list) mark(pg);
  for (const auto& kv : a->owned)
    for (int32_t pg : kv.second) mark(pg);
  for (int32_t r : refs) bad += r != 1;
  return bad;
}

}  // extern "C"

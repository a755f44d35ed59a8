// Host page pool of the paged KV cache ("Build a Speculative Decoding Engine
// to Cut LLM Latency by 3x", Rollback Protocol: rollback is a page-table
// update; the pages of rejected positions go back to the free list, nothing
// is zeroed).  Host code only: a LIFO free list of page ids and the host copy
// of the page table [batch][max_pages] (-1 = unmapped).
#include <new>
#include <vector>

#include "internal.h"

struct spec_page_pool {
  int n_pages, batch, max_pages;
  std::vector<int32_t> table;  // [batch][max_pages]
  std::vector<int32_t> mapped; // pages mapped per sequence (a prefix of its row)
  std::vector<int32_t> free;   // free page ids; the back is taken first
};

namespace {
int pages_for(int slots) { return (slots + SPEC_PAGE_SLOTS - 1) / SPEC_PAGE_SLOTS; }
}  // namespace

extern "C" {

int spec_page_pool_create(int n_pages, int batch, int max_pages, spec_page_pool** out) {
  if (!out) return SPEC_EINVAL;
  *out = nullptr;
  if (n_pages <= 0 || batch <= 0 || max_pages <= 0) return SPEC_EINVAL;
  if (static_cast<long long>(batch) * max_pages > (1ll << 28)) return SPEC_ESIZE;
  spec_page_pool* p = new (std::nothrow) spec_page_pool();
  if (!p) return SPEC_ESIZE;
  p->n_pages = n_pages;
  p->batch = batch;
  p->max_pages = max_pages;
  try {
    p->table.assign(static_cast<size_t>(batch) * max_pages, -1);
    p->mapped.assign(batch, 0);
    p->free.resize(n_pages);
  } catch (...) {
    delete p;
    return SPEC_ESIZE;
  }
  for (int i = 0; i < n_pages; ++i) p->free[i] = n_pages - 1 - i;  // page 0 is taken first
  *out = p;
  return SPEC_OK;
}

int spec_page_pool_destroy(spec_page_pool* p) {
  delete p;
  return SPEC_OK;
}

int spec_page_pool_reserve(spec_page_pool* p, int b, int slots) {
  if (!p || b < 0 || b >= p->batch || slots < 0) return SPEC_EINVAL;
  const int need = pages_for(slots);
  if (need > p->max_pages) return SPEC_ESIZE;
  const int add = need - p->mapped[b];
  if (add <= 0) return SPEC_OK;
  if (add > static_cast<int>(p->free.size())) return SPEC_ESIZE;
  int32_t* row = p->table.data() + static_cast<size_t>(b) * p->max_pages;
  for (int j = p->mapped[b]; j < need; ++j) {
    row[j] = p->free.back();
    p->free.pop_back();
  }
  p->mapped[b] = need;
  return SPEC_OK;
}

int spec_page_pool_release(spec_page_pool* p, int b, int slots) {
  if (!p || b < 0 || b >= p->batch || slots < 0) return SPEC_EINVAL;
  const int keep = pages_for(slots);
  int32_t* row = p->table.data() + static_cast<size_t>(b) * p->max_pages;
  for (int j = p->mapped[b] - 1; j >= keep; --j) {  // the last page goes back first
    p->free.push_back(row[j]);
    row[j] = -1;
  }
  if (keep < p->mapped[b]) p->mapped[b] = keep;
  return SPEC_OK;
}

const int32_t* spec_page_pool_table(const spec_page_pool* p) { return p ? p->table.data() : nullptr; }

int spec_page_pool_free_pages(const spec_page_pool* p) {
  return p ? static_cast<int>(p->free.size()) : SPEC_EINVAL;
}

}  // extern "C"

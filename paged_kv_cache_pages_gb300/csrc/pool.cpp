// Host-side page pool: the per-sequence page mapping of the UA-PagedAttention
// page (section 作品简介) and the fixed-size blocks with reference-counted
// sharing of the CacheFlow page (section 核心架构 2).  Pure host code.
#include <cstdint>
#include <new>
#include <set>
#include <vector>

#include "../../include/paged_attn.h"

struct pa_page_pool {
  std::vector<int32_t> refcount;
  std::set<int32_t> free_pages;  // lowest id first
};

extern "C" {

pa_page_pool *pa_pool_create(int num_pages) {
  if (num_pages <= 0) return nullptr;
  pa_page_pool *p = new (std::nothrow) pa_page_pool;
  if (!p) return nullptr;
  try {
    p->refcount.assign(num_pages, 0);
    for (int i = 0; i < num_pages; ++i) p->free_pages.insert(p->free_pages.end(), i);
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void pa_pool_destroy(pa_page_pool *pool) { delete pool; }

int pa_pool_num_free(const pa_page_pool *pool) {
  return pool ? static_cast<int>(pool->free_pages.size()) : PA_EINVAL;
}

int pa_pool_alloc(pa_page_pool *pool, int n, int32_t *out_pages) {
  if (!pool || n < 0 || (n > 0 && !out_pages)) return PA_EINVAL;
  if (static_cast<size_t>(n) > pool->free_pages.size()) return PA_ENOSPACE;
  for (int i = 0; i < n; ++i) {
    auto it = pool->free_pages.begin();
    out_pages[i] = *it;
    pool->refcount[*it] = 1;
    pool->free_pages.erase(it);
  }
  return n;
}

static bool valid_busy(const pa_page_pool *pool, const int32_t *pages, int n) {
  for (int i = 0; i < n; ++i) {
    int32_t pg = pages[i];
    if (pg < 0 || pg >= static_cast<int32_t>(pool->refcount.size())) return false;
    if (pool->refcount[pg] <= 0) return false;
  }
  return true;
}

int pa_pool_share(pa_page_pool *pool, const int32_t *pages, int n) {
  if (!pool || n < 0 || (n > 0 && !pages)) return PA_EINVAL;
  if (!valid_busy(pool, pages, n)) return PA_EINVAL;
  for (int i = 0; i < n; ++i) ++pool->refcount[pages[i]];
  return PA_OK;
}

int pa_pool_release(pa_page_pool *pool, const int32_t *pages, int n) {
  if (!pool || n < 0 || (n > 0 && !pages)) return PA_EINVAL;
  // a page listed k times must hold at least k references
  std::vector<int32_t> need(pool->refcount.size(), 0);
  for (int i = 0; i < n; ++i) {
    int32_t pg = pages[i];
    if (pg < 0 || pg >= static_cast<int32_t>(pool->refcount.size())) return PA_EINVAL;
    if (++need[pg] > pool->refcount[pg]) return PA_EINVAL;
  }
  for (int i = 0; i < n; ++i) {
    if (--pool->refcount[pages[i]] == 0) pool->free_pages.insert(pages[i]);
  }
  return PA_OK;
}

int pa_pool_fork(pa_page_pool *pool, const int32_t *pages, int n_tokens, int P,
                 int32_t *out_pages, int32_t *copy_src, int32_t *copy_dst) {
  if (!pool || n_tokens < 0 || P <= 0 || !copy_src || !copy_dst) return PA_EINVAL;
  const int n_pages = (n_tokens + P - 1) / P;
  if (n_pages > 0 && (!pages || !out_pages)) return PA_EINVAL;
  if (!valid_busy(pool, pages, n_pages)) return PA_EINVAL;
  const int full = n_tokens / P;  // pages the child may share as they are
  const bool partial = full < n_pages;
  if (partial && pool->free_pages.empty()) return PA_ENOSPACE;
  for (int i = 0; i < full; ++i) {
    ++pool->refcount[pages[i]];
    out_pages[i] = pages[i];
  }
  if (!partial) return 0;
  auto it = pool->free_pages.begin();
  const int32_t fresh = *it;
  pool->free_pages.erase(it);
  pool->refcount[fresh] = 1;
  out_pages[full] = fresh;
  *copy_src = pages[full];
  *copy_dst = fresh;
  return 1;
}

int pa_pool_refcount(const pa_page_pool *pool, int32_t page) {
  if (!pool || page < 0 || page >= static_cast<int32_t>(pool->refcount.size())) return PA_EINVAL;
  return pool->refcount[page];
}

}  // extern "C"

// Page pool admission ledger (host only, no CUDA call): the pages' memory
// admission (PR #2011 review, "Memory admission") -- a request claims its
// pages up front when it is seated, waits with LaneMemory while the pool
// cannot hold it, and is turned away by fits() when it never could.
//
// Pages need not be contiguous, so a claim depends only on the free count.
// It is all or nothing and takes the lowest free ids (a std::set keeps the
// free ids ordered); a claimed bitmap catches releases of pages that are not
// claimed.  One mutex per pool.
#include <algorithm>
#include <mutex>
#include <set>
#include <vector>

#include "tfpa.h"

struct tfpa_pool {
  std::mutex mu;
  int32_t n = 0;
  std::set<int32_t> free_ids;
  std::vector<uint8_t> claimed;
};

extern "C" tfpa_pool* tfpa_pool_create(int32_t num_pages) {
  if (num_pages < 1) return nullptr;
  tfpa_pool* p = new (std::nothrow) tfpa_pool;
  if (!p) return nullptr;
  p->n = num_pages;
  p->claimed.assign(num_pages, 0);
  for (int32_t i = 0; i < num_pages; ++i) p->free_ids.insert(p->free_ids.end(), i);
  return p;
}

extern "C" void tfpa_pool_destroy(tfpa_pool* pool) { delete pool; }

extern "C" int32_t tfpa_pool_free(const tfpa_pool* pool) {
  if (!pool) return 0;
  std::lock_guard<std::mutex> lock(const_cast<tfpa_pool*>(pool)->mu);
  return (int32_t)pool->free_ids.size();
}

extern "C" int tfpa_pool_fits(const tfpa_pool* pool, int32_t npages) {
  return pool && npages >= 0 && npages <= pool->n ? 1 : 0;
}

extern "C" int tfpa_pool_claim(tfpa_pool* pool, int32_t npages, int32_t* pages_out) {
  if (!pool || npages < 0 || (npages > 0 && !pages_out)) return TFPA_EINVAL;
  if (npages > pool->n) return TFPA_ECAPACITY;
  std::lock_guard<std::mutex> lock(pool->mu);
  if ((int32_t)pool->free_ids.size() < npages) return TFPA_ELANEMEM;
  auto it = pool->free_ids.begin();
  for (int32_t i = 0; i < npages; ++i) {
    pages_out[i] = *it;
    pool->claimed[*it] = 1;
    it = pool->free_ids.erase(it);
  }
  return TFPA_OK;
}

extern "C" int tfpa_pool_release(tfpa_pool* pool, const int32_t* pages, int32_t n) {
  if (!pool || n < 0 || (n > 0 && !pages)) return TFPA_EINVAL;
  std::lock_guard<std::mutex> lock(pool->mu);
  std::vector<int32_t> v(pages, pages + n);
  std::sort(v.begin(), v.end());
  for (int32_t i = 0; i < n; ++i) {
    if (v[i] < 0 || v[i] >= pool->n || !pool->claimed[v[i]]) return TFPA_EINVAL;
    if (i > 0 && v[i] == v[i - 1]) return TFPA_EINVAL;
  }
  for (int32_t id : v) {
    pool->claimed[id] = 0;
    pool->free_ids.insert(id);
  }
  return TFPA_OK;
}

// Page pool of the paged KV cache (host code) and the cache's page ledger.
//
// "SGLang x Qwen x NVIDIA Collaboration: NVFP4 KV Cache ...", sections "The
// Core of the Ledger" (16 values take 9 bytes in NVFP4 against 16 in FP8)
// and the equal-capacity comparison (more sequences fit in the same KV
// memory): every layer's cache is indexed by the same page ids, so the KV
// budget buys floor(budget / sum over layers of one page's bytes) pages, and a
// sequence of L tokens holds ceil(L / page_size) of them.
#include <cstdint>
#include <new>
#include <vector>

#include "nvfp4kv.h"

struct nvkv_page_pool {
  std::vector<int32_t> free_stack;  // free page ids, the next one on top
  std::vector<uint8_t> held;        // 1 while a page is handed out
};

extern "C" {

size_t nvkv_cache_page_bytes(int32_t prec, int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 16 != 0) return 0;
  const int64_t per_token = prec == NVKV_PREC_NVFP4 ? 2 * (head_dim / 2 + head_dim / 16)
                            : prec == NVKV_PREC_FP8_E4M3 ? 2 * head_dim
                                                         : 0;
  return static_cast<size_t>(per_token * page_size * num_kv_heads);
}

int32_t nvkv_pool_pages_for_budget(size_t budget_bytes, const int32_t *layer_prec, int32_t num_layers,
                                   int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (!layer_prec || num_layers <= 0) return -1;
  size_t per_page = 0;  // one page id across every layer's cache
  for (int32_t l = 0; l < num_layers; ++l) {
    const size_t b = nvkv_cache_page_bytes(layer_prec[l], page_size, num_kv_heads, head_dim);
    if (b == 0) return -1;
    per_page += b;
  }
  const size_t pages = budget_bytes / per_page;
  return pages > 0x7fffffffu ? 0x7fffffff : static_cast<int32_t>(pages);
}

nvkv_page_pool *nvkv_pool_create(int32_t num_pages) {
  if (num_pages < 0) return nullptr;
  nvkv_page_pool *p = new (std::nothrow) nvkv_page_pool;
  if (!p) return nullptr;
  try {
    p->free_stack.resize(num_pages);
    for (int32_t i = 0; i < num_pages; ++i) p->free_stack[i] = num_pages - 1 - i;  // page 0 comes out first
    p->held.assign(num_pages, 0);
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void nvkv_pool_destroy(nvkv_page_pool *p) { delete p; }

int32_t nvkv_pool_num_free(const nvkv_page_pool *p) {
  return p ? static_cast<int32_t>(p->free_stack.size()) : -1;
}

int32_t nvkv_pool_alloc(nvkv_page_pool *p, int32_t n, int32_t *out) {
  if (!p || n < 0 || (n > 0 && !out)) return -1;
  if (static_cast<size_t>(n) > p->free_stack.size()) return -1;  // all or nothing
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = p->free_stack.back();
    p->free_stack.pop_back();
    p->held[id] = 1;
    out[i] = id;
  }
  return n;
}

nvkv_status nvkv_pool_release(nvkv_page_pool *p, const int32_t *pages, int32_t n) {
  if (!p || n < 0 || (n > 0 && !pages)) return NVKV_ERR_INVALID_ARG;
  const int32_t total = static_cast<int32_t>(p->held.size());
  for (int32_t i = 0; i < n; ++i) {  // check everything first: a bad list releases nothing
    if (pages[i] < 0 || pages[i] >= total || !p->held[pages[i]]) return NVKV_ERR_INVALID_ARG;
    for (int32_t j = 0; j < i; ++j)
      if (pages[j] == pages[i]) return NVKV_ERR_INVALID_ARG;
  }
  for (int32_t i = n - 1; i >= 0; --i) {
    p->held[pages[i]] = 0;
    p->free_stack.push_back(pages[i]);
  }
  return NVKV_OK;
}

}  // extern "C"

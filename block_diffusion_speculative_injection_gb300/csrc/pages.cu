// Paged KV cache: the host-side page allocator and the context calls that
// map and unmap a sequence's pages.
//
// The allocator keeps the free pages in an ordered set (the lowest id goes
// out first, so a run of reservations is reproducible) and, per sequence
// slot, the list of pages in table order.  The device page table is only
// written here, with one host-to-device copy of the entries a call adds (or
// one fill of -1 for a release), on the caller's stream.
#include <cstdio>
#include <set>

#include "internal.cuh"

namespace dflash {

struct PagePool {
  int n_pages = 0, max_seqs = 0, max_pages = 0;
  std::set<int32_t> free_ids;
  std::vector<std::vector<int32_t>> owned;  // [seq] page ids in table order
};

static PagePool* pool_new(int n_pages, int max_seqs, int max_pages) {
  if (n_pages < 0 || max_seqs < 1 || max_pages < 1) return nullptr;
  PagePool* p = new PagePool;
  p->n_pages = n_pages;
  p->max_seqs = max_seqs;
  p->max_pages = max_pages;
  for (int i = 0; i < n_pages; ++i) p->free_ids.insert(p->free_ids.end(), i);
  p->owned.resize(max_seqs);
  return p;
}

// pages needed for n_slots cache slots
static int64_t pages_for(int64_t n_slots) { return (n_slots + kPageSlots - 1) / kPageSlots; }

static dflash_status pool_reserve(PagePool* p, int seq, int64_t n_slots, int* first_new,
                                  int* n_new) {
  if (first_new) *first_new = 0;
  if (n_new) *n_new = 0;
  if (!p || seq < 0 || seq >= p->max_seqs || n_slots < 0) return DFLASH_E_INVALID_ARG;
  std::vector<int32_t>& mine = p->owned[seq];
  const int64_t need = pages_for(n_slots);
  if (first_new) *first_new = (int)mine.size();
  if (need <= (int64_t)mine.size()) return DFLASH_OK;
  const int64_t add = need - (int64_t)mine.size();
  if (need > p->max_pages || add > (int64_t)p->free_ids.size()) return DFLASH_E_CAPACITY;
  for (int64_t i = 0; i < add; ++i) {
    mine.push_back(*p->free_ids.begin());
    p->free_ids.erase(p->free_ids.begin());
  }
  if (n_new) *n_new = (int)add;
  return DFLASH_OK;
}

static int pool_release(PagePool* p, int seq) {
  if (!p || seq < 0 || seq >= p->max_seqs) return -1;
  std::vector<int32_t>& mine = p->owned[seq];
  const int n = (int)mine.size();
  for (int32_t id : mine) p->free_ids.insert(id);
  mine.clear();
  return n;
}

// context side --------------------------------------------------------------

dflash_status pages_init(dflash_ctx* ctx) {
  const dflash_config& c = ctx->cfg;
  ctx->pps = (int)pages_for(c.max_ctx);
  ctx->paged = c.kv_pages > 0;
  ctx->n_pages = ctx->paged ? c.kv_pages : c.max_batch * ctx->pps;
  if (ctx->paged) {
    ctx->pool = pool_new(ctx->n_pages, c.max_batch, ctx->pps);
    if (!ctx->pool) return DFLASH_E_INVALID_ARG;
  }
  return DFLASH_OK;
}

// The table at create: every slot's own pages in order (kv_pages = 0), or
// nothing mapped.
dflash_status pages_fill_table(dflash_ctx* ctx) {
  const dflash_config& c = ctx->cfg;
  std::vector<int32_t> tab((size_t)c.max_batch * ctx->pps, -1);
  if (!ctx->paged)
    for (size_t i = 0; i < tab.size(); ++i) tab[i] = (int32_t)i;
  return cudaMemcpy(ctx->page_tab, tab.data(), tab.size() * sizeof(int32_t),
                    cudaMemcpyHostToDevice) == cudaSuccess
             ? DFLASH_OK
             : DFLASH_E_CUDA;
}

// Keys any sequence of a pass can have: the slots its mapped pages cover
// (paged), else max_ctx.  The attention planner sizes its split for this.
int64_t pages_key_bound(const dflash_ctx* ctx) {
  const int64_t cap = ctx->cfg.max_ctx;
  if (!ctx->paged) return cap;
  size_t most = 0;
  for (const std::vector<int32_t>& v : ctx->pool->owned) most = std::max(most, v.size());
  return std::max<int64_t>(1, std::min<int64_t>(cap, (int64_t)most * kPageSlots));
}

void pages_destroy(dflash_ctx* ctx) {
  delete ctx->pool;
  ctx->pool = nullptr;
}

}  // namespace dflash

using namespace dflash;

struct dflash_kv_pool {
  PagePool p;
};

extern "C" {

dflash_kv_pool* dflash_kv_pool_create(int32_t n_pages, int32_t max_seqs, int32_t max_pages) {
  PagePool* p = pool_new(n_pages, max_seqs, max_pages);
  if (!p) return nullptr;
  dflash_kv_pool* out = new dflash_kv_pool;
  out->p = std::move(*p);
  delete p;
  return out;
}

void dflash_kv_pool_destroy(dflash_kv_pool* pool) { delete pool; }

dflash_status dflash_kv_pool_reserve(dflash_kv_pool* pool, int32_t seq, int32_t n_slots,
                                     int32_t* first_new, int32_t* n_new) {
  if (!pool) return DFLASH_E_INVALID_ARG;
  int f = 0, n = 0;
  const dflash_status s = pool_reserve(&pool->p, seq, n_slots, &f, &n);
  if (first_new) *first_new = f;
  if (n_new) *n_new = n;
  return s;
}

int32_t dflash_kv_pool_release(dflash_kv_pool* pool, int32_t seq) {
  return pool ? pool_release(&pool->p, seq) : -1;
}

int32_t dflash_kv_pool_pages(const dflash_kv_pool* pool, int32_t seq, int32_t* out,
                             int32_t max_out) {
  if (!pool || seq < 0 || seq >= pool->p.max_seqs) return -1;
  const std::vector<int32_t>& mine = pool->p.owned[seq];
  for (int i = 0; out && i < max_out && i < (int)mine.size(); ++i) out[i] = mine[i];
  return (int32_t)mine.size();
}

int32_t dflash_kv_pool_free(const dflash_kv_pool* pool) {
  return pool ? (int32_t)pool->p.free_ids.size() : -1;
}

dflash_status dflash_kv_reserve(dflash_ctx* ctx, int32_t seq_id, int32_t n_slots,
                                dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  if (!ctx_on_current_device(ctx)) {
    ctx->last_error = "called with another device current than the context's";
    return DFLASH_E_STATE;
  }
  const dflash_config& c = ctx->cfg;
  if (seq_id < 0 || seq_id >= c.max_batch || n_slots < 0) {
    ctx->last_error = "dflash_kv_reserve: bad slot or slot count";
    return DFLASH_E_INVALID_ARG;
  }
  if (n_slots > c.max_ctx) {
    ctx->last_error = "dflash_kv_reserve: more slots than max_ctx";
    return DFLASH_E_CAPACITY;
  }
  if (!ctx->paged) return DFLASH_OK;
  int first = 0, n = 0;
  const dflash_status s = pool_reserve(ctx->pool, seq_id, n_slots, &first, &n);
  if (s != DFLASH_OK) {
    ctx->last_error = "dflash_kv_reserve: not enough free pages";
    return s;
  }
  if (n == 0) return DFLASH_OK;
  // pageable source: the copy is staged before this call returns
  const int32_t* ids = ctx->pool->owned[seq_id].data() + first;
  if (cudaMemcpyAsync(ctx->page_tab + (size_t)seq_id * ctx->pps + first, ids,
                      (size_t)n * sizeof(int32_t), cudaMemcpyHostToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    ctx->last_error = "dflash_kv_reserve: page table copy failed";
    return DFLASH_E_CUDA;
  }
  return DFLASH_OK;
}

dflash_status dflash_kv_release(dflash_ctx* ctx, int32_t seq_id, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  if (!ctx_on_current_device(ctx)) {
    ctx->last_error = "called with another device current than the context's";
    return DFLASH_E_STATE;
  }
  if (seq_id < 0 || seq_id >= ctx->cfg.max_batch) {
    ctx->last_error = "dflash_kv_release: bad slot";
    return DFLASH_E_INVALID_ARG;
  }
  if (!ctx->paged) return DFLASH_OK;
  const int n = pool_release(ctx->pool, seq_id);
  if (n > 0 && cudaMemsetAsync(ctx->page_tab + (size_t)seq_id * ctx->pps, 0xFF,
                               (size_t)n * sizeof(int32_t),
                               static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    ctx->last_error = "dflash_kv_release: page table fill failed";
    return DFLASH_E_CUDA;
  }
  return DFLASH_OK;
}

int32_t dflash_kv_free_pages(const dflash_ctx* ctx) {
  if (!ctx) return -1;
  if (!ctx->paged) return 0;
  return (int32_t)ctx->pool->free_ids.size();
}

}  // extern "C"

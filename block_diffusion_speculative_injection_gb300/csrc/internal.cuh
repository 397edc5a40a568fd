// Internal declarations of the DFlash GB300 library: context layout,
// kernel launchers and small PTX wrappers (mbarrier, TMA, tcgen05).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <utility>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/dflash.h"

namespace dflash {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// device status word (sticky; read by dflash_check)
// ---------------------------------------------------------------------------
enum DevStatus { kDevOk = 0, kDevCapacity = 1, kDevTimeout = 2, kDevCheck = 3 };

__device__ __forceinline__ void set_dev_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Iteration bound of every spin-wait on an mbarrier.  try_wait suspends the
// thread for a hardware-defined interval per call, so this is seconds at most.
constexpr uint32_t kSpinLimit = 1u << 26;

// ---------------------------------------------------------------------------
// weights and context
// ---------------------------------------------------------------------------
struct WeightRef {
  const void* ptr = nullptr;
  int64_t shape[2] = {0, 0};
  int ndim = 0;
};

enum PassKind { kPassNone = 0, kPassLinear = 1, kPassTree = 2, kPassDraft = 3 };

// ---------------------------------------------------------------------------
// KV cache addressing.  A layer's cache is a pool of pages
// [page][n_kv][kPageSlots][hd]; slot s of sequence q is row s % kPageSlots of
// page tab[q * pps + s / kPageSlots].  With tab == nullptr the cache is one
// contiguous region per sequence, [seq][n_kv][ctx_cap][hd] (the op-level
// attention over caller tensors).
// ---------------------------------------------------------------------------
constexpr int kPageSlots = DFLASH_PAGE_SLOTS;
static_assert((kPageSlots & (kPageSlots - 1)) == 0, "page slots: a power of two");

struct KvPages {
  const int32_t* tab;  // [max_batch][pps] page ids, -1 unmapped (nullptr: contiguous)
  int pps;             // table entries per sequence
  int n_pages;         // pool size (bounds of a page id)
  int ctx_cap;         // contiguous layout: slots per (sequence, head)
};

// Row (in units of head_dim elements) of cache slot `slot` of sequence `seq`,
// KV head `head`, within one layer; -1 when its page is not mapped.
__device__ __forceinline__ long long kv_row(const KvPages& kp, int Hkv, int seq, int head,
                                            int slot) {
  if (!kp.tab) return ((long long)seq * Hkv + head) * kp.ctx_cap + slot;
  const int pg = kp.tab[seq * kp.pps + slot / kPageSlots];
  if (pg < 0 || pg >= kp.n_pages) return -1;
  return ((long long)pg * Hkv + head) * kPageSlots + (slot & (kPageSlots - 1));
}

// host-side page allocator (csrc/pages.cu)
struct PagePool;

struct LayerW {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
};

}  // namespace dflash

namespace dflash {
enum ProfKind { kProfGemm = 0, kProfAttn = 1, kProfRow = 2, kProfVocab = 3, kProfSpec = 4,
                kProfKinds = 5 };
struct ProfRec {
  int kind;
  int ev;  // index of the start event; the end event is ev + 1
  double bytes, flops;
};
}  // namespace dflash

struct dflash_ctx {
  dflash_config cfg;
  int device = 0;
  int sm_count = 0;
  int esize = 2;  // bytes per stored element (2 bf16, 4 f32)

  std::map<std::string, dflash::WeightRef> weights;
  std::vector<dflash::LayerW> tl, dl;  // resolved target / draft layer pointers
  const void *tok_emb = nullptr, *lm_head = nullptr, *final_norm = nullptr;
  const void *fuse = nullptr, *mask_emb = nullptr, *draft_final_norm = nullptr;
  bool resolved = false;
  int active_block = 0;  // block size of the next draft passes (<= cfg.block_size)

  // per-sequence state
  int32_t* seq_len = nullptr;        // [max_batch] committed length
  int32_t* gen_count = nullptr;      // [max_batch] tokens emitted since reset
  int32_t* dev_status = nullptr;     // [1]

  // caches: [layers][pages][n_kv][kPageSlots][hd], one page table for all
  void *kc = nullptr, *vc = nullptr, *dkc = nullptr, *dvc = nullptr;
  size_t layer_cache_elems = 0;
  int32_t* page_tab = nullptr;     // [max_batch][pps]
  int pps = 0, n_pages = 0;        // table entries per sequence, pool pages
  bool paged = false;              // kv_pages > 0: pages come from the pool on demand
  dflash::PagePool* pool = nullptr;

  // activations (rows = max_rows)
  void* capture = nullptr;  // [max_rows][n_inject][d]
  float* resid = nullptr;   // [max_rows][d]
  void* xn = nullptr;       // [max_rows][d]  normalised GEMM input
  void* qb = nullptr;       // [max_rows][H*hd]
  void* ao = nullptr;       // [max_rows][H*hd] attention output
  void* act = nullptr;      // [max_rows][F] SwiGLU product
  void* fb = nullptr;       // [max_rows][d] fused injection feature F
  void* lm_in = nullptr;    // [max_rows][d] gathered lm_head input
  float* ws = nullptr;      // GEMM fp32 output / split-K partials
  size_t ws_elems = 0;
  // stream-K remainder of the persistent GEMM: one fp32 128 x 256 partial
  // tile per CTA, then the launch ticket (uint64) and one arrival count
  // per remainder tile
  float* sk_part = nullptr;
  void* sk_sync = nullptr;
  float* part_o = nullptr;  // split-KV partial outputs
  float* part_ml = nullptr;
  size_t part_rows_cap = 0;  // capacity in (split*row*head) units
  int32_t* vk_part = nullptr;  // vocab reduction partial ids
  float* vv_part = nullptr;    // vocab reduction partial values / lse
  size_t vpart_cap = 0;

  // pass metadata
  int32_t* pass_seq = nullptr;   // [max_batch]
  int32_t* pass_ctx = nullptr;   // [max_batch] committed length at pass start
  int32_t* pass_blk = nullptr;   // [max_batch] block rows of the sequence
  int32_t* row_pos = nullptr;    // [max_rows] rope position (-1 inactive)
  int32_t* row_slot = nullptr;   // [max_rows] cache slot
  int32_t* row_seq = nullptr;    // [max_rows] sequence slot (-1 inactive)
  int32_t* lm_rows = nullptr;    // [max_rows] rows fed to the lm_head
  int32_t* inj_seq = nullptr;    // [max_rows] pending injection: slot (-1 none)
  int32_t* inj_pos = nullptr;    // [max_rows] pending injection: position
  int32_t* path = nullptr;       // [max_batch][32] accepted tree path (+ old length)
  float* rope_cos = nullptr;     // [rope_len][hd/2]
  float* rope_sin = nullptr;
  int rope_len = 0;

  int last_kind = dflash::kPassNone;
  int last_batch = 0, last_q = 0;
  int pending_rows = 0;  // rows of the injection queue (capture rows)


  float* trace = nullptr;  // debug: residual after every target layer [L][max_rows][d]
  float* dtrace = nullptr; // debug: residual after every draft layer [L_d][max_rows][d]
  void* dtrace_q = nullptr;  // debug: roped Q of every draft layer [L_d][max_rows][H*hd]
  void* dtrace_ao = nullptr; // debug: attention output of every draft layer, same layout
  bool pdl = true;  // programmatic dependent launch between this context's kernels
  int64_t launches = 0;
  std::string last_error;
  // optional per-launch timing (dflash_profile): a pool of CUDA events
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_ev;
  std::vector<dflash::ProfRec> prof_recs;
  size_t prof_next = 0;
  std::map<std::tuple<const void*, int64_t, int64_t, int>, CUtensorMap> tmaps;
};

namespace dflash {

// ---------------------------------------------------------------------------
// launchers (each increments ctx->launches per kernel launched)
// ---------------------------------------------------------------------------
struct GemmSegs {
  const void* w[12];
  int rows[12];
  int n;
};

// paged KV cache (csrc/pages.cu): sizes from the config, the initial table,
// teardown of the host allocator
dflash_status pages_init(dflash_ctx* ctx);
dflash_status pages_fill_table(dflash_ctx* ctx);
void pages_destroy(dflash_ctx* ctx);
int64_t pages_key_bound(const dflash_ctx* ctx);

// A context's calls launch on the current device: it must be the device the
// context was created on (a context on another GPU would be handed foreign
// pointers).  Entry points that launch refuse the call otherwise.
inline bool ctx_on_current_device(const dflash_ctx* ctx) {
  int d = -1;
  return cudaGetDevice(&d) == cudaSuccess && d == ctx->device;
}

inline KvPages ctx_pages(const dflash_ctx* ctx) {
  return KvPages{ctx->page_tab, ctx->pps, ctx->n_pages, 0};
}

struct EpiArgs;
// bytes of ctx->sk_sync for a GPU of sm_count SMs: the launch ticket, then
// one arrival count per stream-K tile (fewer than the persistent CTAs)
inline size_t sk_sync_bytes(int sm_count) { return 8 + 4 * (size_t)std::max(sm_count, 1); }
// X[M][K] . W^T with W the vertical stack of the segments, then the fused
// epilogue described by `epi` (see epilogue.cuh).  The fp32 result / K-split
// slabs live in ctx->ws; *splits_used reports the split count.
dflash_status gemm(dflash_ctx* ctx, const void* x, int M, int K, const GemmSegs& segs,
                   const EpiArgs& epi, int max_splits, int* splits_used, cudaStream_t st);

enum MaskKind { kMaskNone = 0, kMaskCausal = 1, kMaskTree = 2 };

struct AttnArgs {
  const void* q;      // [rows][H][hd]
  void* out;          // [rows][H*hd]
  const void* kc;     // layer cache base [max_batch][Hkv][max_ctx][hd]
  const void* vc;
  int batch, q_stride;  // rows of sequence b: b*q_stride + j, j < pass_blk[b]
  int mask;
  const uint64_t* anc;  // tree: [batch][q_stride][anc_words]
  int anc_words;
  int64_t max_keys_ub;  // host upper bound on ctx+blk keys of any sequence
};
dflash_status attention(dflash_ctx* ctx, const AttnArgs& a, cudaStream_t st);

// row operations
dflash_status launch_pass_setup_full(dflash_ctx* ctx, int batch, const int32_t* seq_ids, int q,
                                     const int32_t* q_lens, const int32_t* depth,
                                     const int32_t* n_nodes, int kind, int last_only,
                                     const int32_t* anchor, int32_t* block_out, int32_t* pseq,
                                     int32_t* pctx, int32_t* pblk, cudaStream_t st);
dflash_status launch_embed(dflash_ctx* ctx, const int32_t* tokens, int rows, int draft_block,
                           int block, cudaStream_t st);
// out[i] = RMSNorm(resid[rows_in ? rows_in[i] : i]) * gain, i < n_out
dflash_status launch_norm(dflash_ctx* ctx, int n_out, const int32_t* rows_in, const void* gain,
                          void* out, cudaStream_t st);
// fp32 logits slab (ctx->ws) -> chunk candidates -> per-row results
dflash_status launch_vocab_reduce(dflash_ctx* ctx, int rows, int vocab, const int32_t* row_out,
                                  int topk, int32_t* argmax, float* margin, int32_t* topk_ids,
                                  float* topk_logp, float* logits_copy, cudaStream_t st);
// per-row results from K candidates of each of n_chunks chunks already in
// ctx->vk_part / ctx->vv_part (the lm_head epilogue's); row_out = [arg_idx |
// vec_idx] (vec_idx at + max_rows)
dflash_status launch_vocab_merge(dflash_ctx* ctx, int rows, int n_chunks, int K,
                                 const int32_t* row_out, int topk, int32_t* argmax, float* margin,
                                 int32_t* topk_ids, float* topk_logp, cudaStream_t st);

// speculation control
dflash_status launch_accept_linear(dflash_ctx* ctx, int batch, const int32_t* seq_ids,
                                   const int32_t* block, const int32_t* argmax, int q, int mode,
                                   int32_t* accept_len, int32_t* next_anchor, int32_t* emitted,
                                   cudaStream_t st);
dflash_status launch_advance_lengths(dflash_ctx* ctx, int batch, const int32_t* seq_ids,
                                     const int32_t* counts, cudaStream_t st);
dflash_status launch_tree_build(dflash_ctx* ctx, int batch, const int32_t* anchor,
                                const int32_t* ids, const float* logp, int topk, int depth,
                                int budget, const dtree_buffers* t, cudaStream_t st);
dflash_status launch_tree_accept(dflash_ctx* ctx, int batch, const int32_t* seq_ids,
                                 const dtree_buffers* t, const int32_t* argmax,
                                 int32_t* accept_len, int32_t* next_anchor, int32_t* emitted,
                                 cudaStream_t st);

void set_error(dflash_ctx* ctx, const char* fmt, ...);

// Per-device one-time host state.  Kernel attributes set with
// cudaFuncSetAttribute and SM counts belong to one device, so they are kept
// per device index (slots are atomics: two host threads may race on a first
// call; both store the same value).
constexpr int kMaxDevices = 64;
// current device index in [0, kMaxDevices), or -1
inline int current_device_slot() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
// raises a kernel's dynamic shared-memory limit once per device
template <typename K>
inline cudaError_t ensure_smem_attr(std::atomic<bool>* done, K kernel, int bytes) {
  const int dev = current_device_slot();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_relaxed);
  return e;
}

// Brackets the launches of one launcher with CUDA events when profiling is
// on; `bytes` / `flops` are the algorithmic traffic and work of the launch.
struct ProfScope {
  dflash_ctx* ctx;
  cudaStream_t st;
  int idx = -1;
  ProfScope(dflash_ctx* c, int kind, cudaStream_t s, double bytes = 0, double flops = 0)
      : ctx(c), st(s) {
    if (!c->prof_on || c->prof_next + 2 > c->prof_ev.size()) return;
    idx = (int)c->prof_next;
    c->prof_next += 2;
    cudaEventRecord(c->prof_ev[idx], s);
    c->prof_recs.push_back(ProfRec{kind, idx, bytes, flops});
  }
  ~ProfScope() {
    if (idx >= 0) cudaEventRecord(ctx->prof_ev[idx + 1], st);
  }
};

// Tensor maps (gemm.cu).  tmap_2d: bf16 [rows][cols] row-major, box [box_rows][64],
// 128-byte swizzle, cached in the context.  encode_tmap_bf16: any rank <= 3
// bf16 tensor (dims innermost first, byte strides of dims 1..rank-1), box
// dims innermost first, 128-byte swizzle, zero fill out of bounds.
dflash_status tmap_2d(dflash_ctx* ctx, const void* ptr, int64_t rows, int64_t cols, int box_rows,
                      const CUtensorMap** out);
bool encode_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box);

int64_t block_attention_workspace(int batch, int H, int Hkv, int hd, int ctx_len, int block);
dflash_status plan_attention(int sm_count, int batch, int H, int Hkv, int q_per_seq,
                             int64_t max_keys, int min_splits, int32_t* out);
dflash_status plan_gemm(int sm_count, int M, int N, int K, int kind, int max_splits, int32_t* out);
dflash_status block_attention(int batch, int H, int Hkv, int hd, int ctx_len, int block, int causal,
                              const void* q, const void* k, const void* v, void* out,
                              void* workspace, int64_t workspace_bytes, cudaStream_t st);

#define DF_CUDA_TRY(ctx, expr)                                                    \
  do {                                                                            \
    cudaError_t e__ = (expr);                                                     \
    if (e__ != cudaSuccess) {                                                     \
      ::dflash::set_error((ctx), "%s: %s", #expr, cudaGetErrorString(e__));       \
      return DFLASH_E_CUDA;                                                       \
    }                                                                             \
  } while (0)

#define DF_LAUNCHED(ctx)                                                          \
  do {                                                                            \
    (ctx)->launches++;                                                            \
    cudaError_t e__ = cudaGetLastError();                                         \
    if (e__ != cudaSuccess) {                                                     \
      ::dflash::set_error((ctx), "launch at %s:%d: %s", __FILE__, __LINE__,       \
                          cudaGetErrorString(e__));                               \
      return DFLASH_E_CUDA;                                                       \
    }                                                                             \
  } while (0)

#define DF_TRY(expr)                  \
  do {                                \
    dflash_status s__ = (expr);       \
    if (s__ != DFLASH_OK) return s__; \
  } while (0)

// ---------------------------------------------------------------------------
// element load/store helpers for the two storage types
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<bf16>(const bf16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void st_f(T* p, float v);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_f<bf16>(bf16* p, float v) { *p = __float2bfloat16_rn(v); }
// four consecutive elements (address aligned to four elements)
template <typename T>
__device__ __forceinline__ void st_f4(T* p, float4 v);
template <>
__device__ __forceinline__ void st_f4<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <>
__device__ __forceinline__ void st_f4<bf16>(bf16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel may start while its predecessor
// drains; it must call pdl_wait() before touching any memory an earlier
// kernel writes or reads-then-rewrites.  Kernels signal their dependents
// (pdl_trigger) before they wait, so a launch can be resident two or three
// kernels ahead of the one that is running; what it does before its wait
// (the GEMM's weight prefetch) reads only memory no kernel writes.  A kernel
// is released only once every CTA of its predecessor has started, so the
// CTAs that wait never hold back one that is still to be scheduled.  Both
// are no-ops without the launch attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                            size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// same, as thread-block clusters of `cluster` CTAs
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_cluster(bool pdl, dim3 cluster, void (*kernel)(KArgs...), dim3 grid,
                                    dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster.x;
  attr[0].val.clusterDim.y = cluster.y;
  attr[0].val.clusterDim.z = cluster.z;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// thread-block clusters and distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster arrives, then waits
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// address of the same shared-memory offset in cluster CTA `rank`
__device__ __forceinline__ uint32_t map_peer(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// four consecutive fp32 (16-byte aligned address)
__device__ __forceinline__ float4 ld_peer_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// cp.async (16-byte global -> shared copies; src_bytes 0 zero-fills)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: gives up after ~2 s of wall time (or kSpinLimit polls),
// records a timeout in the status word and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023u) == 0 && global_ns() - t0 > 2000000000ull) break;
  }
  set_dev_status(status, kDevTimeout);
  return false;
}

// Same bound, for waiters that have nothing else to do (epilogue warps):
// back off between polls so the issuing warps keep their issue slots.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    __nanosleep(128);
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > 2000000000ull) break;
  }
  set_dev_status(status, kDevTimeout);
  return false;
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// the same copy with an L2 eviction-priority hint (a createpolicy value)
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// 3-D tiled copy (box {x, y, z} of the tensor map), same completion mechanism
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// one plain arrival (the barrier's count tells how many complete a phase)
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// generic-proxy shared-memory writes become visible to the async proxy (TMA,
// tensor cores) once a barrier orders them after this fence
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// data read once per pass: first in line for eviction from L2
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D(tmem) (+)= A(smem desc) * B(smem desc)^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns per warp.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 consecutive 32-bit columns per warp, without the wait (the
// caller issues tmem_wait_ld() once after a batch of loads).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Half-warp form: threads 0..15 read lanes 0..15 of the warp's lane quarter at
// columns c .. c+31, threads 16..31 the SAME lanes at columns c+kOff .. (kOff
// is an immediate), so two threads can share the columns of one row.
template <int kOff>
__device__ __forceinline__ void tmem_ld_half32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], %33;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "n"(kOff));
}
template <int kOff>
__device__ __forceinline__ void tmem_st_half32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};" ::"r"(
          taddr),
      "n"(kOff), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
      "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns per warp (the store form of tmem_ld16).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
// a 32-bit load with acquire semantics at GPU scope (a flag set by another CTA)
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 64 elements (128 B), 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFF);  // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused with swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                      // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                      // swizzle mode: 128 B
  return d;
}

// Descriptor of an MN-major bf16 operand with 128-byte swizzling: rows of 128 B
// hold 64 consecutive MN elements at one K index, 8-row groups (8 K values)
// sit 1024 B apart, and the next 64 MN elements start `mn_stride` bytes
// further (the leading byte offset in this mode).
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t smem_addr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFF);
  d |= (uint64_t)((mn_stride >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor: kind::f16, D f32, A/B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
// bit 16 of the instruction descriptor: the B operand is MN-major
constexpr uint32_t kIdescBMajorMN = 1u << 16;

}  // namespace dflash

// Acceptance, commit/rollback and the DDTree builder.
//
// Linear block (glossary "DFlash: architecture and workflow", stage 4): the
// longest prefix of draft tokens equal to the target's argmax at the
// previous position is accepted, the target's token at the first mismatch
// is emitted after it, and the committed length grows by a + 1.  Rows past
// the accepted prefix are rolled back by length alone: their cache slots
// are simply overwritten by the next pass.
//
// DDTree (ludicrous-speed story, DDTree paragraph): best-first heap over
// prefixes of the per-slot top-k lists; the accepted path found by walking
// from the root is compacted to consecutive cache slots in every target
// layer.
#include <climits>

#include "internal.cuh"

namespace dflash {

// ---------------------------------------------------------------------------
// linear accept / commit (one thread per sequence)
// ---------------------------------------------------------------------------
__global__ void accept_linear_kernel(int batch, int q, int mode, const int32_t* __restrict__ block,
                                     const int32_t* __restrict__ argmax,
                                     const int32_t* __restrict__ pass_seq,
                                     const int32_t* __restrict__ pass_ctx,
                                     const int32_t* __restrict__ pass_blk,
                                     int32_t* __restrict__ seq_len, int32_t* __restrict__ gen_count,
                                     int32_t* __restrict__ accept_len,
                                     int32_t* __restrict__ next_anchor,
                                     int32_t* __restrict__ emitted, int32_t* __restrict__ inj_seq,
                                     int32_t* __restrict__ inj_pos) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int seq = pass_seq[b], ctx = pass_ctx[b], n = pass_blk[b];
  const size_t base = (size_t)b * q;
  int commit = 0;
  if (n <= 0) {
    accept_len[b] = -1;
    next_anchor[b] = -1;
    for (int j = 0; j < q; ++j) emitted[base + j] = -1;
  } else if (mode == DFLASH_ACCEPT_ALL) {
    commit = n;
    const int y = argmax[base + n - 1];
    accept_len[b] = n;
    next_anchor[b] = y;
    emitted[base] = y;
    for (int j = 1; j < q; ++j) emitted[base + j] = -1;
  } else {
    int a = 0, y;
    if (mode == DFLASH_ACCEPT_GIVEN) {  // decided by the caller's sampling step
      a = min(max(accept_len[b], 0), n - 1);
      y = next_anchor[b];
    } else {
      while (a < n - 1 && block[base + 1 + a] == argmax[base + a]) ++a;
      y = argmax[base + a];
    }
    for (int j = 0; j < a; ++j) emitted[base + j] = block[base + 1 + j];
    emitted[base + a] = y;
    for (int j = a + 1; j < q; ++j) emitted[base + j] = -1;
    accept_len[b] = a;
    next_anchor[b] = y;
    commit = a + 1;
  }
  if (n > 0) {
    seq_len[seq] = ctx + commit;
    gen_count[seq] += mode == DFLASH_ACCEPT_ALL ? 1 : commit;
  }
  for (int j = 0; j < q; ++j) {
    inj_seq[base + j] = j < commit ? seq : -1;
    inj_pos[base + j] = ctx + j;
  }
}

dflash_status launch_accept_linear(dflash_ctx* ctx, int batch, const int32_t* seq_ids,
                                   const int32_t* block, const int32_t* argmax, int q, int mode,
                                   int32_t* accept_len, int32_t* next_anchor, int32_t* emitted,
                                   cudaStream_t st) {
  ProfScope prof__(ctx, kProfSpec, st);
  (void)seq_ids;
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, accept_linear_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, 
      batch, q, mode, block, argmax, ctx->pass_seq, ctx->pass_ctx, ctx->pass_blk, ctx->seq_len,
      ctx->gen_count, accept_len, next_anchor, emitted, ctx->inj_seq, ctx->inj_pos));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

// Committed lengths moved on by counts decided elsewhere (a drafter-side
// context mirroring the commits of a verifier-side one).  A count that would
// pass max_ctx leaves the length and flags the capacity status.
__global__ void advance_lengths_kernel(int batch, const int32_t* __restrict__ seq_ids,
                                       const int32_t* __restrict__ counts,
                                       int32_t* __restrict__ seq_len, int max_batch, int max_ctx,
                                       int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int seq = seq_ids[b], n = counts[b];
  if (seq < 0 || seq >= max_batch) {
    set_dev_status(status, kDevCheck);
    return;
  }
  if (n <= 0) return;
  if (seq_len[seq] + n > max_ctx) {
    set_dev_status(status, kDevCapacity);
    return;
  }
  seq_len[seq] += n;
}

dflash_status launch_advance_lengths(dflash_ctx* ctx, int batch, const int32_t* seq_ids,
                                     const int32_t* counts, cudaStream_t st) {
  ProfScope prof__(ctx, kProfSpec, st);
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, advance_lengths_kernel, dim3((batch + 127) / 128), dim3(128),
                            0, st, batch, seq_ids, counts, ctx->seq_len, ctx->cfg.max_batch,
                            ctx->cfg.max_ctx, ctx->dev_status));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// DDTree best-first builder (one CTA per sequence; thread 0 runs the heap)
// ---------------------------------------------------------------------------
struct HeapEnt {
  float score;
  int depth;
  unsigned long long rk;  // rank vector: 4 bits per level, level 1 in the top bits
  int parent;             // node id of the prefix without the last rank
  int rank;
};

__device__ __forceinline__ bool heap_before(const HeapEnt& a, const HeapEnt& b) {
  if (a.score != b.score) return a.score > b.score;
  if (a.depth != b.depth) return a.depth < b.depth;
  return a.rk < b.rk;
}

constexpr int kMaxTreeNodes = 128;

__global__ void tree_build_kernel(int depth_max, int topk, int budget,
                                  const int32_t* __restrict__ anchor,
                                  const int32_t* __restrict__ ids, const float* __restrict__ logp,
                                  dtree_buffers t) {
  pdl_wait();
  pdl_trigger();
  __shared__ HeapEnt heap[kMaxTreeNodes + 2];
  __shared__ float node_score[kMaxTreeNodes];
  __shared__ int n_nodes_s;
  const int b = blockIdx.x;
  const size_t nb = (size_t)b * t.max_nodes;
  const int32_t* id_b = ids + (size_t)b * depth_max * topk;
  const float* lp_b = logp + (size_t)b * depth_max * topk;
  if (threadIdx.x == 0) {
    int hn = 0;
    auto push = [&](const HeapEnt& e) {
      int i = hn++;
      heap[i] = e;
      while (i > 0) {
        const int p = (i - 1) / 2;
        if (!heap_before(heap[i], heap[p])) break;
        const HeapEnt tmp = heap[p];
        heap[p] = heap[i];
        heap[i] = tmp;
        i = p;
      }
    };
    auto pop = [&]() {
      const HeapEnt top = heap[0];
      heap[0] = heap[--hn];
      int i = 0;
      for (;;) {
        const int l = 2 * i + 1, r = l + 1;
        int m = i;
        if (l < hn && heap_before(heap[l], heap[m])) m = l;
        if (r < hn && heap_before(heap[r], heap[m])) m = r;
        if (m == i) break;
        const HeapEnt tmp = heap[m];
        heap[m] = heap[i];
        heap[i] = tmp;
        i = m;
      }
      return top;
    };
    // root
    t.tok[nb] = anchor[b];
    t.parent[nb] = -1;
    t.depth[nb] = 0;
    for (int w = 0; w < t.anc_words; ++w) t.anc[nb * t.anc_words + w] = w == 0 ? 1ull : 0ull;
    node_score[0] = 0.f;
    int n = 1;
    if (depth_max >= 1 && topk >= 1 && budget > 0) {
      HeapEnt e;
      e.score = __fadd_rn(0.f, lp_b[0]);
      e.depth = 1;
      e.rk = 0ull;
      e.parent = 0;
      e.rank = 0;
      push(e);
    }
    while (hn > 0 && n - 1 < budget) {
      const HeapEnt e = pop();
      const int me = n++;
      t.tok[nb + me] = id_b[(size_t)(e.depth - 1) * topk + e.rank];
      t.parent[nb + me] = e.parent;
      t.depth[nb + me] = e.depth;
      for (int w = 0; w < t.anc_words; ++w) {
        unsigned long long a = t.anc[(nb + e.parent) * t.anc_words + w];
        if (w == (me >> 6)) a |= 1ull << (me & 63);
        t.anc[(nb + me) * t.anc_words + w] = a;
      }
      node_score[me] = e.score;
      if (e.depth < depth_max) {  // first child: rank 0 one level deeper
        HeapEnt c;
        c.score = __fadd_rn(e.score, lp_b[(size_t)e.depth * topk]);
        c.depth = e.depth + 1;
        c.rk = e.rk;
        c.parent = me;
        c.rank = 0;
        push(c);
      }
      if (e.rank + 1 < topk) {  // next sibling
        HeapEnt s;
        s.score = __fadd_rn(node_score[e.parent], lp_b[(size_t)(e.depth - 1) * topk + e.rank + 1]);
        s.depth = e.depth;
        s.rk = e.rk + (1ull << (4 * (15 - e.depth)));
        s.parent = e.parent;
        s.rank = e.rank + 1;
        push(s);
      }
    }
    n_nodes_s = n;
    t.n_nodes[b] = n;
  }
  __syncthreads();
  // clear the unused node rows
  const int n = n_nodes_s;
  for (int i = n + threadIdx.x; i < t.max_nodes; i += blockDim.x) {
    t.tok[nb + i] = -1;
    t.parent[nb + i] = -1;
    t.depth[nb + i] = 0;
    for (int w = 0; w < t.anc_words; ++w) t.anc[(nb + i) * t.anc_words + w] = 0ull;
  }
}

dflash_status launch_tree_build(dflash_ctx* ctx, int batch, const int32_t* anchor,
                                const int32_t* ids, const float* logp, int topk, int depth,
                                int budget, const dtree_buffers* t, cudaStream_t st) {
  ProfScope prof__(ctx, kProfSpec, st);
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, tree_build_kernel, dim3(batch), dim3(32), 0, st, depth, topk, budget, anchor, ids, logp, *t));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// tree accept walk (one thread per sequence) + KV compaction
// ---------------------------------------------------------------------------
constexpr int kPathStride = 34;  // [a, ctx, node_0 .. node_a]

__global__ void tree_accept_kernel(int batch, dtree_buffers t, const int32_t* __restrict__ argmax,
                                   const int32_t* __restrict__ pass_seq,
                                   const int32_t* __restrict__ pass_ctx,
                                   const int32_t* __restrict__ pass_blk,
                                   int32_t* __restrict__ seq_len, int32_t* __restrict__ gen_count,
                                   int32_t* __restrict__ accept_len,
                                   int32_t* __restrict__ next_anchor, int32_t* __restrict__ emitted,
                                   int32_t* __restrict__ inj_seq, int32_t* __restrict__ inj_pos,
                                   int32_t* __restrict__ path, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int q = t.max_nodes;
  const size_t base = (size_t)b * q;
  const int seq = pass_seq[b], ctx = pass_ctx[b], n = pass_blk[b];
  int32_t* pb = path + (size_t)b * kPathStride;
  for (int j = 0; j < q; ++j) {
    inj_seq[base + j] = -1;
    inj_pos[base + j] = -1;
    emitted[base + j] = -1;
  }
  if (n <= 0) {
    accept_len[b] = -1;
    next_anchor[b] = -1;
    pb[0] = 0;
    pb[1] = ctx;
    pb[2] = 0;
    return;
  }
  int cur = 0, a = 0;
  pb[2] = 0;
  for (;;) {
    const int y = argmax[base + cur];
    int nxt = -1;
    for (int c = cur + 1; c < n; ++c)
      if (t.parent[base + c] == cur && t.tok[base + c] == y) {
        nxt = c;
        break;
      }
    if (nxt < 0) break;
    if (a + 1 > kPathStride - 3) {
      set_dev_status(status, kDevCheck);
      break;
    }
    cur = nxt;
    ++a;
    pb[2 + a] = cur;
    emitted[base + a - 1] = t.tok[base + cur];
  }
  const int y = argmax[base + cur];
  emitted[base + a] = y;
  accept_len[b] = a;
  next_anchor[b] = y;
  pb[0] = a;
  pb[1] = ctx;
  for (int i = 0; i <= a; ++i) {
    inj_seq[base + pb[2 + i]] = seq;
    inj_pos[base + pb[2 + i]] = ctx + i;
  }
  seq_len[seq] = ctx + a + 1;
  gen_count[seq] += a + 1;
}

// One CTA per (layer, sequence, KV head): gather every accepted row first,
// then write them to their final slots (a source slot may be another row's
// destination).
template <typename T>
__global__ void tree_compact_kernel(const int32_t* __restrict__ path,
                                    const int32_t* __restrict__ pass_seq,
                                    const int32_t* __restrict__ pass_blk, T* kc, T* vc,
                                    size_t layer_elems, int batch, int Hkv, int hd,
                                    const KvPages kp, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t buf[];
  const int l = blockIdx.x / batch, b = blockIdx.x % batch, kh = blockIdx.y;
  if (pass_blk[b] <= 0) return;
  const int32_t* pb = path + (size_t)b * kPathStride;
  const int a = pb[0], ctx = pb[1];
  const int seq = pass_seq[b];
  if (a <= 0) return;
  T* ks = reinterpret_cast<T*>(buf);
  T* vs = ks + (size_t)a * hd;
  const size_t layer = (size_t)l * layer_elems;
  // the pages of every slot of the pass were checked at pass setup; an
  // unmapped one is flagged and its row skipped
  for (int i = threadIdx.x; i < a * hd; i += blockDim.x) {
    const int r = i / hd + 1, e = i % hd;
    const long long row = kv_row(kp, Hkv, seq, kh, ctx + pb[2 + r]);
    if (row < 0) {
      set_dev_status(status, kDevCapacity);
      continue;
    }
    const size_t src = layer + (size_t)row * hd + e;
    ks[i] = kc[src];
    vs[i] = vc[src];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a * hd; i += blockDim.x) {
    const int r = i / hd + 1, e = i % hd;
    const long long row = kv_row(kp, Hkv, seq, kh, ctx + r);
    if (row < 0) continue;
    const size_t dst = layer + (size_t)row * hd + e;
    kc[dst] = ks[i];
    vc[dst] = vs[i];
  }
}

dflash_status launch_tree_accept(dflash_ctx* ctx, int batch, const int32_t* seq_ids,
                                 const dtree_buffers* t, const int32_t* argmax,
                                 int32_t* accept_len, int32_t* next_anchor, int32_t* emitted,
                                 cudaStream_t st) {
  ProfScope prof__(ctx, kProfSpec, st);
  (void)seq_ids;
  const dflash_config& c = ctx->cfg;
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, tree_accept_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, 
      batch, *t, argmax, ctx->pass_seq, ctx->pass_ctx, ctx->pass_blk, ctx->seq_len, ctx->gen_count,
      accept_len,
      next_anchor, emitted, ctx->inj_seq, ctx->inj_pos, ctx->path, ctx->dev_status));
  DF_LAUNCHED(ctx);
  dim3 grid(c.n_target_layers * batch, c.n_kv_heads);
  const size_t smem = 2 * 16 * (size_t)c.head_dim * ctx->esize;
  if (c.dtype == DFLASH_BF16)
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, tree_compact_kernel<bf16>, dim3(grid), dim3(128), smem, st, 
        ctx->path, ctx->pass_seq, ctx->pass_blk, static_cast<bf16*>(ctx->kc),
        static_cast<bf16*>(ctx->vc), ctx->layer_cache_elems, batch, c.n_kv_heads, c.head_dim,
        ctx_pages(ctx), ctx->dev_status));
  else
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, tree_compact_kernel<float>, dim3(grid), dim3(128), smem, st, 
        ctx->path, ctx->pass_seq, ctx->pass_blk, static_cast<float*>(ctx->kc),
        static_cast<float*>(ctx->vc), ctx->layer_cache_elems, batch, c.n_kv_heads, c.head_dim,
        ctx_pages(ctx), ctx->dev_status));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

}  // namespace dflash

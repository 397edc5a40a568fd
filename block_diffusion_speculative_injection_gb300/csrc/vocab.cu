// Reductions over the vocabulary of one lm_head pass.
//
// Pass 1 gives, per row and chunk of the vocabulary, the chunk's best K
// candidates (value descending, id ascending) plus its (max, sum exp(x -
// max)).  With bf16 storage the lm_head GEMM's epilogue produces them per
// 128-feature tile (the logits never reach memory); the fp32 model's slab
// is scanned here in chunks of 4096 (vocab_pass1_kernel).  Pass 2 (one CTA
// per row) merges the chunks: argmax, top-1 minus top-2 margin, top-k ids
// and log-softmax values (logit - logsumexp, temperature 1).
#include <cfloat>
#include <climits>

#include "internal.cuh"

namespace dflash {

constexpr int kVocabChunk = 4096;
constexpr int kVocabThreads = 256;
constexpr int kMaxK = 16;

struct Cand {
  float v;
  int id;
};

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// K rounds of a block-wide arg-best over per-thread sorted lists.
// Thread lists: lv/li[0..n) sorted best-first.  Winners go to out[0..K).
__device__ void block_select(const float* lv, const int* li, int n, int K, Cand* out,
                             Cand* red) {
  int head = 0;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int k = 0; k < K; ++k) {
    float v = head < n ? lv[head] : -INFINITY;
    int id = head < n ? li[head] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, id, o);
      if (better(v2, i2, v, id)) {
        v = v2;
        id = i2;
      }
    }
    if (lane == 0) red[w] = Cand{v, id};
    __syncthreads();
    if (threadIdx.x == 0) {
      Cand best = red[0];
      for (int i = 1; i < nw; ++i)
        if (better(red[i].v, red[i].id, best.v, best.id)) best = red[i];
      out[k] = best;
    }
    __syncthreads();
    if (head < n && li[head] == out[k].id && lv[head] == out[k].v) ++head;
    __syncthreads();
  }
}

// block-wide sum (kSum) or max, result in every thread; red holds 32 floats
template <bool kSum>
__device__ float block_reduce(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = kSum ? v + w : fmaxf(v, w);
  }
  __syncthreads();  // red may still be read from an earlier call
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) v = kSum ? v + red[i] : fmaxf(v, red[i]);
  return v;
}

__global__ void __launch_bounds__(kVocabThreads)
    vocab_pass1_kernel(const float* __restrict__ logits, int vocab, int K,
                       const int32_t* __restrict__ vec_idx, float* __restrict__ logits_copy,
                       int32_t* __restrict__ part_id, float* __restrict__ part_v,
                       float* __restrict__ part_lse, int n_chunks) {
  pdl_wait();
  pdl_trigger();
  __shared__ Cand red[32];
  __shared__ Cand best[kMaxK];
  __shared__ float mred[32];
  const int row = blockIdx.x, chunk = blockIdx.y;
  const float* x = logits + (size_t)row * vocab;
  const int c0 = chunk * kVocabChunk, c1 = min(vocab, c0 + kVocabChunk);
  float lv[kMaxK];
  int li[kMaxK];
  int n = 0;
  float m = -INFINITY;
  const int vi = vec_idx[row];
  for (int i = c0 + threadIdx.x; i < c1; i += kVocabThreads) {
    const float v = x[i];
    if (logits_copy && vi >= 0) logits_copy[(size_t)vi * vocab + i] = v;
    m = fmaxf(m, v);
    // insertion into the sorted list (ids arrive ascending, so ties keep order)
    if (n < K || v > lv[n - 1]) {
      int p = n < K ? n : K - 1;
      while (p > 0 && v > lv[p - 1]) {
        lv[p] = lv[p - 1];
        li[p] = li[p - 1];
        --p;
      }
      lv[p] = v;
      li[p] = i;
      if (n < K) ++n;
    }
  }
  // chunk max and sum of exp
  float bm = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
  if ((threadIdx.x & 31) == 0) mred[threadIdx.x >> 5] = bm;
  __syncthreads();
  float cm = -INFINITY;
  for (int i = 0; i < kVocabThreads / 32; ++i) cm = fmaxf(cm, mred[i]);
  float se = 0.f;
  for (int i = c0 + threadIdx.x; i < c1; i += kVocabThreads) se += __expf(x[i] - cm);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) mred[threadIdx.x >> 5] = se;
  __syncthreads();
  block_select(lv, li, n, K, best, red);
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < kVocabThreads / 32; ++i) s += mred[i];
    const size_t pb = (size_t)row * n_chunks + chunk;
    part_lse[pb * 2] = cm;
    part_lse[pb * 2 + 1] = s;
  }
  if (threadIdx.x < K) {
    const size_t pb = ((size_t)row * n_chunks + chunk) * K + threadIdx.x;
    part_id[pb] = best[threadIdx.x].id;
    part_v[pb] = best[threadIdx.x].v;
  }
}

__global__ void __launch_bounds__(kVocabThreads)
    vocab_pass2_kernel(int K, int topk, int n_chunks, const int32_t* __restrict__ part_id,
                       const float* __restrict__ part_v, const float* __restrict__ part_lse,
                       const int32_t* __restrict__ arg_idx, const int32_t* __restrict__ vec_idx,
                       int32_t* __restrict__ argmax, float* __restrict__ margin,
                       int32_t* __restrict__ topk_ids, float* __restrict__ topk_logp) {
  pdl_wait();
  pdl_trigger();
  __shared__ Cand red[32];
  __shared__ Cand best[kMaxK];
  __shared__ float lse_s;
  const int row = blockIdx.x;
  // each thread takes whole chunk lists (already sorted best-first)
  // and merges them into a private sorted list of length K
  float lv[kMaxK];
  int li[kMaxK];
  int n = 0;
  for (int c = threadIdx.x; c < n_chunks; c += kVocabThreads) {
    const size_t pb = ((size_t)row * n_chunks + c) * K;
    for (int k = 0; k < K; ++k) {
      const float v = part_v[pb + k];
      const int id = part_id[pb + k];
      if (id == INT_MAX) continue;
      if (n < K || better(v, id, lv[n - 1], li[n - 1])) {
        int p = n < K ? n : K - 1;
        while (p > 0 && better(v, id, lv[p - 1], li[p - 1])) {
          lv[p] = lv[p - 1];
          li[p] = li[p - 1];
          --p;
        }
        lv[p] = v;
        li[p] = id;
        if (n < K) ++n;
      }
    }
  }
  block_select(lv, li, n, K, best, red);
  if (topk > 0) {  // log-sum-exp over the chunks (only the top-k log-probs use it)
    __shared__ float lred[32];
    const float2* pl = reinterpret_cast<const float2*>(part_lse) + (size_t)row * n_chunks;
    float M = -INFINITY;
    for (int c = threadIdx.x; c < n_chunks; c += kVocabThreads) M = fmaxf(M, pl[c].x);
    M = block_reduce<false>(M, lred);
    float S = 0.f;
    for (int c = threadIdx.x; c < n_chunks; c += kVocabThreads) {
      const float2 ms = pl[c];
      S += ms.y * __expf(ms.x - M);
    }
    S = block_reduce<true>(S, lred);
    if (threadIdx.x == 0) lse_s = M + logf(S);
  }
  if (threadIdx.x == 0) {
    const int ai = arg_idx[row];
    if (ai >= 0) {
      if (argmax) argmax[ai] = best[0].id;
      if (margin) margin[ai] = K > 1 ? best[0].v - best[1].v : INFINITY;
    }
  }
  __syncthreads();
  const int vi = vec_idx[row];
  if (topk > 0 && vi >= 0 && threadIdx.x < topk) {
    topk_ids[(size_t)vi * topk + threadIdx.x] = best[threadIdx.x].id;
    topk_logp[(size_t)vi * topk + threadIdx.x] = best[threadIdx.x].v - lse_s;
  }
}

dflash_status launch_vocab_merge(dflash_ctx* ctx, int rows, int n_chunks, int K,
                                 const int32_t* row_out, int topk, int32_t* argmax, float* margin,
                                 int32_t* topk_ids, float* topk_logp, cudaStream_t st) {
  ProfScope prof__(ctx, kProfVocab, st);
  if (rows <= 0) return DFLASH_OK;
  if ((size_t)rows * n_chunks * K > ctx->vpart_cap || K < 2 || K > kMaxK || topk > K) {
    set_error(ctx, "vocab partial buffer too small");
    return DFLASH_E_CAPACITY;
  }
  // row_out = [arg_idx | vec_idx] for these rows
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, vocab_pass2_kernel, dim3(rows), dim3(kVocabThreads), 0, st,
                            K, topk, n_chunks, ctx->vk_part, ctx->vv_part,
                            ctx->vv_part + ctx->vpart_cap, row_out, row_out + ctx->cfg.max_rows,
                            argmax, margin, topk_ids, topk_logp));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

dflash_status launch_vocab_reduce(dflash_ctx* ctx, int rows, int vocab, const int32_t* row_out,
                                  int topk, int32_t* argmax, float* margin, int32_t* topk_ids,
                                  float* topk_logp, float* logits_copy, cudaStream_t st) {
  if (rows <= 0) return DFLASH_OK;
  const int K = topk > 2 ? topk : 2;
  const int n_chunks = (vocab + kVocabChunk - 1) / kVocabChunk;
  if ((size_t)rows * n_chunks * K > ctx->vpart_cap) {
    set_error(ctx, "vocab partial buffer too small");
    return DFLASH_E_CAPACITY;
  }
  {
    ProfScope prof__(ctx, kProfVocab, st);
    dim3 g1(rows, n_chunks);
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, vocab_pass1_kernel, dim3(g1), dim3(kVocabThreads), 0, st,
                              ctx->ws, vocab, K, row_out + ctx->cfg.max_rows, logits_copy,
                              ctx->vk_part, ctx->vv_part, ctx->vv_part + ctx->vpart_cap,
                              n_chunks));
    DF_LAUNCHED(ctx);
  }
  return launch_vocab_merge(ctx, rows, n_chunks, K, row_out, topk, argmax, margin, topk_ids,
                            topk_logp, st);
}

}  // namespace dflash

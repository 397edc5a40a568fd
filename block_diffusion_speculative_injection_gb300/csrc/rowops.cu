// Row-wise kernels of the target / draft passes: the pass setup (per-sequence
// and per-row metadata), the token / mask embedding into the fp32 residual
// stream, and RMSNorm of residual rows into the next GEMM's input (optionally
// gathering rows).  What follows each projection (RoPE + cache scatter,
// SwiGLU, residual add + capture, injection) is fused into the GEMM's
// epilogue instead.
#include "internal.cuh"

namespace dflash {

// ---------------------------------------------------------------------------
// pass setup: per-sequence and per-row metadata of one pass
// ---------------------------------------------------------------------------
struct PassSetupArgs {
  const int32_t* seq_ids;
  const int32_t* q_lens;
  const int32_t* depth;    // tree: [batch][q]
  const int32_t* n_nodes;  // tree: [batch]
  const int32_t* anchor;   // draft: [batch] (slot 0 of the block)
  int32_t* block_out;      // draft: [batch][q]
  const int32_t* seq_len;
  int32_t *pass_seq, *pass_ctx, *pass_blk;
  int32_t *row_pos, *row_slot, *row_seq;
  int32_t *lm_in, *lm_arg, *lm_vec;
  int batch, q, kind, last_only, max_batch, max_ctx;
  KvPages kp;  // every slot a pass touches must sit in a mapped page
  int32_t* status;
};

__global__ void pass_setup_kernel(PassSetupArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_blk[1024];
  __shared__ int s_ctx[1024];
  for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
    const int seq = a.seq_ids[b];
    int blk = 0, ctx = 0;
    if (seq < 0 || seq >= a.max_batch) {
      set_dev_status(a.status, kDevCheck);
    } else {
      ctx = a.seq_len[seq];
      if (a.kind == kPassTree) blk = a.n_nodes[b];
      else if (a.kind == kPassDraft) blk = a.q;
      else blk = a.q_lens ? a.q_lens[b] : a.q;
      if (blk < 0 || blk > a.q) {
        set_dev_status(a.status, kDevCheck);
        blk = 0;
      }
      if (ctx + blk > a.max_ctx) {
        set_dev_status(a.status, kDevCapacity);
        blk = 0;
      }
      // the pass reads slots 0 .. ctx + blk - 1 (keys) and writes ctx ..
      // ctx + blk - 1: all of their pages must be mapped
      for (int pg = 0; blk > 0 && pg * kPageSlots < ctx + blk; ++pg) {
        const int id = a.kp.tab[seq * a.kp.pps + pg];
        if (id < 0 || id >= a.kp.n_pages) {
          set_dev_status(a.status, kDevCapacity);
          blk = 0;
        }
      }
    }
    a.pass_seq[b] = seq < 0 || seq >= a.max_batch ? 0 : seq;
    a.pass_ctx[b] = ctx;
    a.pass_blk[b] = blk;
    s_blk[b] = blk;
    s_ctx[b] = ctx;
    if (a.kind == kPassDraft && a.block_out) a.block_out[(size_t)b * a.q] = a.anchor[b];
  }
  __syncthreads();
  const int rows = a.batch * a.q;
  for (int r = threadIdx.x; r < rows; r += blockDim.x) {
    const int b = r / a.q, j = r % a.q;
    const int blk = s_blk[b], ctx = s_ctx[b];
    const bool live = j < blk;
    int pos = ctx + j;
    if (a.kind == kPassTree && live) {
      const int d = a.depth[r];
      if (d < 0 || d > j) set_dev_status(a.status, kDevCheck);
      pos = ctx + (d < 0 ? 0 : (d > j ? j : d));
    }
    a.row_pos[r] = live ? pos : -1;
    a.row_slot[r] = live ? ctx + j : -1;
    a.row_seq[r] = live ? a.seq_ids[b] : -1;
  }
  // lm_head row maps
  if (a.kind == kPassDraft) {
    const int per = a.q - 1;
    for (int i = threadIdx.x; i < a.batch * per; i += blockDim.x) {
      const int b = i / per, j = i % per;
      const int r = b * a.q + 1 + j;
      a.lm_in[i] = r;
      a.lm_arg[i] = s_blk[b] > 0 ? r : -1;
      a.lm_vec[i] = s_blk[b] > 0 ? i : -1;
    }
  } else if (a.last_only) {
    for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
      const int r = b * a.q + (s_blk[b] > 0 ? s_blk[b] - 1 : 0);
      a.lm_in[b] = r;
      a.lm_arg[b] = s_blk[b] > 0 ? r : -1;
      a.lm_vec[b] = s_blk[b] > 0 ? r : -1;
    }
  } else {
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
      const bool live = (r % a.q) < s_blk[r / a.q];
      a.lm_in[r] = r;
      a.lm_arg[r] = live ? r : -1;
      a.lm_vec[r] = live ? r : -1;
    }
  }
}

dflash_status launch_pass_setup_full(dflash_ctx* ctx, int batch, const int32_t* seq_ids, int q,
                                     const int32_t* q_lens, const int32_t* depth,
                                     const int32_t* n_nodes, int kind, int last_only,
                                     const int32_t* anchor, int32_t* block_out, int32_t* pseq,
                                     int32_t* pctx, int32_t* pblk, cudaStream_t st) {
  ProfScope prof__(ctx, kProfRow, st);
  PassSetupArgs a;
  a.seq_ids = seq_ids;
  a.q_lens = q_lens;
  a.depth = depth;
  a.n_nodes = n_nodes;
  a.anchor = anchor;
  a.block_out = block_out;
  a.seq_len = ctx->seq_len;
  a.pass_seq = pseq;
  a.pass_ctx = pctx;
  a.pass_blk = pblk;
  a.row_pos = ctx->row_pos;
  a.row_slot = ctx->row_slot;
  a.row_seq = ctx->row_seq;
  a.lm_in = ctx->lm_rows;
  a.lm_arg = ctx->lm_rows + ctx->cfg.max_rows;
  a.lm_vec = ctx->lm_rows + 2 * (size_t)ctx->cfg.max_rows;
  a.batch = batch;
  a.q = q;
  a.kind = kind;
  a.last_only = last_only;
  a.max_batch = ctx->cfg.max_batch;
  a.max_ctx = ctx->cfg.max_ctx;
  a.kp = ctx_pages(ctx);
  a.status = ctx->dev_status;
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, pass_setup_kernel, dim3(1), dim3(1024), 0, st, a));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// embedding: resid[r] = tok_emb[token] (target rows) or, for a draft block,
// slot 0 = tok_emb[anchor], slots 1..B-1 = mask embedding.  Dead rows = 0.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void embed_kernel(const int32_t* __restrict__ tokens, const T* __restrict__ emb,
                             const T* __restrict__ mask_emb, const int32_t* __restrict__ row_pos,
                             float* __restrict__ resid, int d, int vocab, int draft_block,
                             int block, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  float* out = resid + (size_t)r * d;
  const T* src = nullptr;
  // the row's position and token are independent loads (both in flight)
  const int pos = row_pos[r];
  int tok;
  if (draft_block) {
    const int b = r / block, j = r % block;
    tok = j == 0 ? tokens[b] : -2;
  } else {
    tok = tokens[r];
  }
  if (pos >= 0) {
    if (tok == -2) src = mask_emb;
    else if (tok >= 0 && tok < vocab) src = emb + (size_t)tok * d;
    else set_dev_status(status, kDevCheck);
  }
  // 16-byte loads and stores when the row and the (borrowed) tables allow
  constexpr int V = 16 / (int)sizeof(T);
  const bool aligned = ((reinterpret_cast<uintptr_t>(emb) | reinterpret_cast<uintptr_t>(mask_emb)) &
                        15u) == 0;
  if (aligned && d % V == 0 && d % 4 == 0) {
    for (int i = threadIdx.x * V; i < d; i += blockDim.x * V) {
      float x[V];
      if (src) {
        const uint4 u = *reinterpret_cast<const uint4*>(src + i);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int k = 0; k < V; ++k) x[k] = ld_f(e + k);
      } else {
#pragma unroll
        for (int k = 0; k < V; ++k) x[k] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < V; k += 4)
        *reinterpret_cast<float4*>(out + i + k) = make_float4(x[k], x[k + 1], x[k + 2], x[k + 3]);
    }
    return;
  }
  for (int i = threadIdx.x; i < d; i += blockDim.x) out[i] = src ? ld_f(src + i) : 0.f;
}

dflash_status launch_embed(dflash_ctx* ctx, const int32_t* tokens, int rows, int draft_block,
                           int block, cudaStream_t st) {
  ProfScope prof__(ctx, kProfRow, st);
  const int d = ctx->cfg.d_model;
  if (ctx->cfg.dtype == DFLASH_BF16)
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, embed_kernel<bf16>, dim3(rows), dim3(256), 0, st, tokens, static_cast<const bf16*>(ctx->tok_emb),
                                             static_cast<const bf16*>(ctx->mask_emb), ctx->row_pos,
                                             ctx->resid, d, ctx->cfg.vocab, draft_block, block,
                                             ctx->dev_status));
  else
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, embed_kernel<float>, dim3(rows), dim3(256), 0, st, tokens, static_cast<const float*>(ctx->tok_emb),
                                              static_cast<const float*>(ctx->mask_emb),
                                              ctx->row_pos, ctx->resid, d, ctx->cfg.vocab,
                                              draft_block, block, ctx->dev_status));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// RMSNorm of residual rows into the next GEMM's input (optionally gathered)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  const int nw = blockDim.x >> 5;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

constexpr int kNormThreads = 256;
constexpr int kNormMaxPer = 32;  // d_model <= 8192

template <typename T>
__global__ void __launch_bounds__(kNormThreads)
    norm_kernel(const float* __restrict__ resid, const int32_t* __restrict__ rows_in, int d,
                const T* __restrict__ gain, T* __restrict__ out, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int i_out = blockIdx.x;
  const int r = rows_in ? rows_in[i_out] : i_out;
  float x[kNormMaxPer];
  float ss = 0.f;
  const int per = (d + kNormThreads - 1) / kNormThreads;
#pragma unroll
  for (int k = 0; k < kNormMaxPer; ++k) {
    if (k >= per) break;
    const int i = threadIdx.x + k * kNormThreads;
    const float v = (i < d && r >= 0) ? resid[(size_t)r * d + i] : 0.f;
    x[k] = v;
    ss += v * v;
  }
  const float tot = block_sum(ss, red);
  const float inv = rsqrtf(tot / (float)d + eps);
#pragma unroll
  for (int k = 0; k < kNormMaxPer; ++k) {
    if (k >= per) break;
    const int i = threadIdx.x + k * kNormThreads;
    if (i < d) st_f(out + (size_t)i_out * d + i, x[k] * inv * ld_f(gain + i));
  }
}

// Vectorised variant for d_model % 1024 == 0: VPT float4 groups per thread,
// all loads issued before the reduction.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

template <typename T, int VPT>
__global__ void __launch_bounds__(kNormThreads)
    norm_vec_kernel(const float* __restrict__ resid, const int32_t* __restrict__ rows_in, int d,
                    const T* __restrict__ gain, T* __restrict__ out, float eps) {
  pdl_trigger();
  __shared__ float red[32];
  float4 x[VPT], g[VPT];
  // the gains are weights (no kernel writes them): load them before waiting
  // on the preceding kernel
#pragma unroll
  for (int v = 0; v < VPT; ++v) g[v] = ld4(gain + (threadIdx.x + v * kNormThreads) * 4);
  pdl_wait();
  const int i_out = blockIdx.x;
  const int r = rows_in ? rows_in[i_out] : i_out;
  float ss = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int i = (threadIdx.x + v * kNormThreads) * 4;
    x[v] = r >= 0 ? ld4(resid + (size_t)r * d + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int v = 0; v < VPT; ++v) ss += x[v].x * x[v].x + x[v].y * x[v].y + x[v].z * x[v].z + x[v].w * x[v].w;
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + eps);
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int i = (threadIdx.x + v * kNormThreads) * 4;
    st4(out + (size_t)i_out * d + i, make_float4(x[v].x * inv * g[v].x, x[v].y * inv * g[v].y,
                                                 x[v].z * inv * g[v].z, x[v].w * inv * g[v].w));
  }
}

template <typename T>
static cudaError_t launch_norm_t(dflash_ctx* ctx, int n_out, const int32_t* rows_in,
                                 const void* gain, void* out, cudaStream_t st) {
  const int d = ctx->cfg.d_model;
  const float eps = ctx->cfg.rms_eps;
  const T* g = static_cast<const T*>(gain);
  T* o = static_cast<T*>(out);
  const int vpt = d % 1024 == 0 ? d / 1024 : 0;
  switch (vpt) {
    case 1: return launch_k(ctx->pdl, norm_vec_kernel<T, 1>, dim3(n_out), dim3(kNormThreads), 0, st, ctx->resid, rows_in, d, g, o, eps);
    case 2: return launch_k(ctx->pdl, norm_vec_kernel<T, 2>, dim3(n_out), dim3(kNormThreads), 0, st, ctx->resid, rows_in, d, g, o, eps);
    case 4: return launch_k(ctx->pdl, norm_vec_kernel<T, 4>, dim3(n_out), dim3(kNormThreads), 0, st, ctx->resid, rows_in, d, g, o, eps);
    case 8: return launch_k(ctx->pdl, norm_vec_kernel<T, 8>, dim3(n_out), dim3(kNormThreads), 0, st, ctx->resid, rows_in, d, g, o, eps);
    default: return launch_k(ctx->pdl, norm_kernel<T>, dim3(n_out), dim3(kNormThreads), 0, st, ctx->resid, rows_in, d, g, o, eps);
  }
}

dflash_status launch_norm(dflash_ctx* ctx, int n_out, const int32_t* rows_in, const void* gain,
                          void* out, cudaStream_t st) {
  ProfScope prof__(ctx, kProfRow, st);
  if (n_out <= 0) return DFLASH_OK;
  if (ctx->cfg.dtype == DFLASH_BF16)
    DF_CUDA_TRY(ctx, (launch_norm_t<bf16>(ctx, n_out, rows_in, gain, out, st)));
  else
    DF_CUDA_TRY(ctx, (launch_norm_t<float>(ctx, n_out, rows_in, gain, out, st)));
  DF_LAUNCHED(ctx);
  return DFLASH_OK;
}

}  // namespace dflash

// Temperature-1 drafting and acceptance (speculative rejection sampling).
//
// The pages run DFlash at temperature 1 (report "DFlash benchmark results")
// and describe sampled draft tokens and an acceptance criterion (glossary
// "DFlash: architecture and workflow", stages 2 and 3) without stating the
// rule; the standard speculative rejection rule is taken:
//   d_j ~ p_j = softmax(drafter logits at slot j), 1 <= j < B;
//   d_j passes when u_j * p_j(d_j) < q_{j-1}(d_j), q_i = softmax(target
//   logits at block row i); at the first failure one token is drawn from
//   max(0, q_{j-1} - p_j) normalised; if all pass, from q_{B-1};
//   a draw with uniform u is the smallest token id whose cumulative weight
//   (in id order) exceeds u times the total.
//
// fp32 logits [rows][V].  Everything is split into chunks of kChunk token ids:
//   samp_stats_kernel   per (row, chunk): max m and sum exp(x - m), merged in
//                       a fixed tree order (deterministic)
//   samp_pick_kernel    per row: the chunk where the cumulative mass crosses
//                       u * total (chunks in id order), then a block-wide scan
//                       inside it -- draws from softmax(row)
//   samp_accept_kernel  per sequence: one lane per block slot runs its accept
//                       test; the first failure fixes the accept length and
//                       the rows of the final draw
//   samp_final_kernel   per (sequence, chunk): mass of the final draw's weights
//                       (residual or bonus row), then the same pick
// Every sum runs in a fixed order, so equal inputs give equal outputs.
#include <cfloat>
#include <cmath>
#include <cstdio>

#include "internal.cuh"

namespace dflash {

constexpr int kChunk = 4096;
constexpr int kSampThreads = 256;
constexpr int kPerThread = kChunk / kSampThreads;  // 16 consecutive ids per thread
constexpr int kMaxBlock = 32;    // block slots tested by one warp
constexpr int kMaxChunks = 128;  // vocabulary up to 524,288 ids

struct MS {
  float m, s;
};

// (m, s) of x merged into (m, s): s = sum exp(x_i - m)
__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  const float m = fmaxf(a.m, b.m);
  return {m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}

// block-wide merge in a fixed order (warp butterflies, then warp 0 over warps)
__device__ MS block_merge(MS v) {
  __shared__ MS warp_part[kSampThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MS o;
    o.m = __shfl_xor_sync(0xffffffffu, v.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, v.s, off);
    v = ms_merge(v, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) warp_part[warp] = v;
  __syncthreads();
  MS r = {-INFINITY, 0.f};
  if (threadIdx.x == 0)
    for (int w = 0; w < kSampThreads / 32; ++w) r = ms_merge(r, warp_part[w]);
  __syncthreads();
  return r;  // valid in thread 0
}

// rows x chunks of (max, sum exp) ----------------------------------------
__global__ void __launch_bounds__(kSampThreads) samp_stats_kernel(const float* __restrict__ logits,
                                                                  int V, int n_chunks,
                                                                  float2* __restrict__ stats) {
  pdl_wait();
  pdl_trigger();
  const int k = blockIdx.x, row = blockIdx.y;
  const float* x = logits + (size_t)row * V;
  const int x0 = k * kChunk, x1 = min(V, x0 + kChunk);
  // this thread's ids x0 + e * kSampThreads + tid: all loads first, then the
  // max, then one exponential per id, summed in e order
  float xs[kPerThread];
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < kPerThread; ++e) {
    const int i = x0 + e * kSampThreads + (int)threadIdx.x;
    xs[e] = i < x1 ? x[i] : -INFINITY;
    m = fmaxf(m, xs[e]);
  }
  // exp(x - m) = 2^((x - m) log2 e)
  constexpr float kLog2e = 1.4426950408889634f;
  float sum = 0.f;
  if (m != -INFINITY) {
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) sum += exp2f((xs[e] - m) * kLog2e);
  }
  const MS v = {m, sum};
  const MS r = block_merge(v);
  if (threadIdx.x == 0) stats[(size_t)row * n_chunks + k] = make_float2(r.m, r.s);
}

// log-sum-exp of a row from its chunk stats, chunks in id order
__device__ __forceinline__ float row_lse(const float2* st, int n_chunks) {
  float M = -INFINITY;
  for (int k = 0; k < n_chunks; ++k) M = fmaxf(M, st[k].x);
  if (M == -INFINITY) return -INFINITY;
  float T = 0.f;
  for (int k = 0; k < n_chunks; ++k)
    if (st[k].x != -INFINITY) T += st[k].y * expf(st[k].x - M);
  return M + logf(T);
}

// Weight of token id i in a draw: plain softmax (mode 0: exp(t - lse_t)) or
// residual (mode 1: max(0, exp(t - lse_t) - exp(d - lse_d))).
struct DrawRow {
  const float* t;
  const float* d;
  float lse_t, lse_d;
  int mode;
};

__device__ __forceinline__ float draw_w(const DrawRow& r, int i) {
  const float q = expf(r.t[i] - r.lse_t);
  if (r.mode == 0) return q;
  return fmaxf(0.f, q - expf(r.d[i] - r.lse_d));
}

// Mass of one chunk of a draw, summed in a fixed order (thread-contiguous
// runs of kPerThread ids, then threads in order).
__device__ float chunk_mass(const DrawRow& r, int x0, int x1, float* thread_sum_out) {
  __shared__ float part[kSampThreads];
  const int a = x0 + (int)threadIdx.x * kPerThread;
  float s = 0.f;
  for (int i = a; i < min(x1, a + kPerThread); ++i) s += draw_w(r, i);
  part[threadIdx.x] = s;
  if (thread_sum_out) *thread_sum_out = s;
  __syncthreads();
  float tot = 0.f;
  if (threadIdx.x == 0)
    for (int t = 0; t < kSampThreads; ++t) tot += part[t];
  __syncthreads();
  return tot;  // valid in thread 0
}

// Inside chunk [x0, x1): the first id whose cumulative weight, starting at
// `before`, exceeds `target` (block-wide; every thread gets the result).
// Rounding can leave the crossing past the chunk end: then the last id of
// the chunk with positive weight.
__device__ int pick_in_chunk(const DrawRow& r, int x0, int x1, float before, float target) {
  __shared__ float tsum[kSampThreads];
  __shared__ int s_pick;
  const int a = x0 + (int)threadIdx.x * kPerThread;
  float s = 0.f;
  for (int i = a; i < min(x1, a + kPerThread); ++i) s += draw_w(r, i);
  tsum[threadIdx.x] = s;
  if (threadIdx.x == 0) s_pick = -1;
  __syncthreads();
  if (threadIdx.x == 0) {
    float acc = before;
    int t = 0;
    for (; t < kSampThreads; ++t) {
      if (acc + tsum[t] > target) break;
      acc += tsum[t];
    }
    if (t < kSampThreads) {
      const int b = x0 + t * kPerThread;
      for (int i = b; i < min(x1, b + kPerThread); ++i) {
        acc += draw_w(r, i);
        if (acc > target) {
          s_pick = i;
          break;
        }
      }
    }
    if (s_pick < 0)
      for (int i = x1 - 1; i >= x0; --i)
        if (draw_w(r, i) > 0.f) {
          s_pick = i;
          break;
        }
  }
  __syncthreads();
  return s_pick;
}

// One draw from softmax(row) per row ----------------------------------------
__global__ void __launch_bounds__(kSampThreads)
    samp_pick_kernel(const float* __restrict__ logits, int V, int n_chunks,
                     const float2* __restrict__ stats, const float* __restrict__ u,
                     int32_t* __restrict__ tokens) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const float2* st = stats + (size_t)row * n_chunks;
  __shared__ float s_before, s_target;
  __shared__ int s_chunk;
  __shared__ float s_lse;
  if (threadIdx.x == 0) {
    const float lse = row_lse(st, n_chunks);
    // chunk masses exp(m_k - lse) * s_k, in id order
    float T = 0.f;
    for (int k = 0; k < n_chunks; ++k)
      if (st[k].x != -INFINITY) T += st[k].y * expf(st[k].x - lse);
    const float target = u[row] * T;
    float acc = 0.f;
    int k = 0, last = 0;
    for (; k < n_chunks; ++k) {
      if (st[k].x == -INFINITY) continue;
      last = k;
      const float c = st[k].y * expf(st[k].x - lse);
      if (acc + c > target) break;
      acc += c;
    }
    if (k == n_chunks) k = last;  // rounding: the last chunk with mass
    s_chunk = k;
    s_before = acc;
    s_target = target;
    s_lse = lse;
  }
  __syncthreads();
  const DrawRow r{logits + (size_t)row * V, nullptr, s_lse, 0.f, 0};
  const int x0 = s_chunk * kChunk, x1 = min(V, x0 + kChunk);
  const int tok = pick_in_chunk(r, x0, x1, s_before, s_target);
  if (threadIdx.x == 0) tokens[row] = tok;
}

// Accept tests: one warp per sequence, lane j tests slot j ------------------
struct SeqDraw {
  int mode, trow, drow, pad;
  float lse_t, lse_d, pad2, pad3;
};

__global__ void __launch_bounds__(32)
    samp_accept_kernel(const float* __restrict__ dl, const float* __restrict__ tl, int B, int V,
                       int n_chunks, const float2* __restrict__ dstats,
                       const float2* __restrict__ tstats, const int32_t* __restrict__ tokens,
                       const float* __restrict__ u_accept, int32_t* __restrict__ accept_len,
                       SeqDraw* __restrict__ draw) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, j = threadIdx.x;
  bool pass = true;
  float lse_t = 0.f, lse_d = 0.f;
  if (j >= 1 && j < B) {
    const int d = tokens[b * B + j];
    const size_t drow = (size_t)b * (B - 1) + j - 1, trow = (size_t)b * B + j - 1;
    lse_d = row_lse(dstats + drow * n_chunks, n_chunks);
    lse_t = row_lse(tstats + trow * n_chunks, n_chunks);
    if (d >= 0 && d < V) {
      const float p = expf(dl[drow * V + d] - lse_d);
      const float q = expf(tl[trow * V + d] - lse_t);
      pass = u_accept[b * B + j] * p < q;
    } else {
      pass = false;
    }
  }
  const unsigned fail = __ballot_sync(0xffffffffu, !pass);
  const int jf = fail ? __ffs(fail) - 1 : B;  // first failing slot (lanes >= B pass)
  const float lt = __shfl_sync(0xffffffffu, lse_t, jf < B ? jf : 0);
  const float ld = __shfl_sync(0xffffffffu, lse_d, jf < B ? jf : 0);
  if (j == 0) {
    SeqDraw s;
    s.pad = 0;
    s.pad2 = s.pad3 = 0.f;
    if (jf < B) {  // residual of q_{jf-1} against p_jf
      accept_len[b] = jf - 1;
      s.mode = 1;
      s.trow = b * B + jf - 1;
      s.drow = b * (B - 1) + jf - 1;
      s.lse_t = lt;
      s.lse_d = ld;
    } else {  // all passed: bonus from q_{B-1}
      accept_len[b] = B - 1;
      s.mode = 0;
      s.trow = b * B + B - 1;
      s.drow = 0;
      s.lse_t = row_lse(tstats + (size_t)(b * B + B - 1) * n_chunks, n_chunks);
      s.lse_d = 0.f;
    }
    draw[b] = s;
  }
}

// chunk masses of each sequence's final draw
__global__ void __launch_bounds__(kSampThreads)
    samp_final_mass_kernel(const float* __restrict__ dl, const float* __restrict__ tl, int V,
                           int n_chunks, const SeqDraw* __restrict__ draw,
                           float* __restrict__ mass) {
  pdl_wait();
  pdl_trigger();
  const int k = blockIdx.x, b = blockIdx.y;
  const SeqDraw s = draw[b];
  const DrawRow r{tl + (size_t)s.trow * V, dl + (size_t)s.drow * V, s.lse_t, s.lse_d, s.mode};
  const int x0 = k * kChunk, x1 = min(V, x0 + kChunk);
  const float m = chunk_mass(r, x0, x1, nullptr);
  if (threadIdx.x == 0) mass[(size_t)b * n_chunks + k] = m;
}

__global__ void __launch_bounds__(kSampThreads)
    samp_final_pick_kernel(const float* __restrict__ dl, const float* __restrict__ tl, int V,
                           int n_chunks, const SeqDraw* __restrict__ draw,
                           const float* __restrict__ mass, const float* __restrict__ u_resample,
                           int32_t* __restrict__ emitted) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const SeqDraw s = draw[b];
  __shared__ float s_mass[kMaxChunks];
  __shared__ float s_before, s_target;
  __shared__ int s_chunk, s_fallback;
  if (threadIdx.x == 0) {
    float T = 0.f;
    for (int k = 0; k < n_chunks; ++k) T += mass[(size_t)b * n_chunks + k];
    // a residual without mass (q and p equal up to rounding) draws from q
    s_fallback = (s.mode == 1 && !(T > 0.f)) ? 1 : 0;
  }
  __syncthreads();
  const DrawRow r{tl + (size_t)s.trow * V, dl + (size_t)s.drow * V, s.lse_t, s.lse_d,
                  s_fallback ? 0 : s.mode};
  for (int k = 0; k < n_chunks; ++k) {
    float m;
    if (s_fallback) m = chunk_mass(r, k * kChunk, min(V, (k + 1) * kChunk), nullptr);
    else m = mass[(size_t)b * n_chunks + k];
    if (threadIdx.x == 0) s_mass[k] = m;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float T = 0.f;
    for (int k = 0; k < n_chunks; ++k) T += s_mass[k];
    const float target = u_resample[b] * T;
    float acc = 0.f;
    int k = 0, last = 0;
    for (; k < n_chunks; ++k) {
      if (!(s_mass[k] > 0.f)) continue;
      last = k;
      if (acc + s_mass[k] > target) break;
      acc += s_mass[k];
    }
    if (k == n_chunks) k = last;  // rounding: the last chunk with mass
    s_chunk = k;
    s_before = acc;
    s_target = target;
  }
  __syncthreads();
  const int x0 = s_chunk * kChunk, x1 = min(V, x0 + kChunk);
  const int tok = pick_in_chunk(r, x0, x1, s_before, s_target);
  if (threadIdx.x == 0) emitted[b] = tok;
}

static int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

static int sample_chunks(int vocab) { return (vocab + kChunk - 1) / kChunk; }

}  // namespace dflash

using namespace dflash;

extern "C" {

int64_t dflash_sample_workspace(int32_t rows, int32_t vocab) {
  if (rows < 1 || rows > 65535 || vocab < 1 || sample_chunks(vocab) > kMaxChunks) return -1;
  return align256((int64_t)rows * sample_chunks(vocab) * (int64_t)sizeof(float2));
}

dflash_status dflash_sample_rows(int32_t rows, int32_t vocab, const float* logits, const float* u,
                                 int32_t* tokens, void* workspace, int64_t workspace_bytes,
                                 dflash_stream_t stream) {
  const int64_t need = dflash_sample_workspace(rows, vocab);
  if (need < 0 || !logits || !u || !tokens || !workspace) return DFLASH_E_INVALID_ARG;
  if (workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return DFLASH_E_INVALID_ARG;
  const int nc = sample_chunks(vocab);
  float2* stats = static_cast<float2*>(workspace);
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_k(true, samp_stats_kernel, dim3(nc, rows), dim3(kSampThreads), 0, st, logits, vocab,
               nc, stats) != cudaSuccess)
    return DFLASH_E_CUDA;
  if (launch_k(true, samp_pick_kernel, dim3(rows), dim3(kSampThreads), 0, st, logits, vocab, nc,
               (const float2*)stats, u, tokens) != cudaSuccess)
    return DFLASH_E_CUDA;
  return DFLASH_OK;
}

int64_t dflash_spec_accept_workspace(int32_t batch, int32_t block, int32_t vocab) {
  if (batch < 1 || block < 1 || block > kMaxBlock || (int64_t)batch * block > 65535 || vocab < 1 ||
      sample_chunks(vocab) > kMaxChunks)
    return -1;
  const int64_t nc = sample_chunks(vocab);
  const int64_t stats = align256((int64_t)batch * block * nc * (int64_t)sizeof(float2));
  return 2 * stats + align256((int64_t)batch * (int64_t)sizeof(SeqDraw)) +
         align256((int64_t)batch * nc * (int64_t)sizeof(float));  // draft stats fit in `stats`
}

dflash_status dflash_spec_accept_sampled(int32_t batch, int32_t block, int32_t vocab,
                                         const float* draft_logits, const float* target_logits,
                                         const int32_t* tokens, const float* u_accept,
                                         const float* u_resample, int32_t* accept_len,
                                         int32_t* emitted, void* workspace,
                                         int64_t workspace_bytes, dflash_stream_t stream) {
  const int64_t need = dflash_spec_accept_workspace(batch, block, vocab);
  if (need < 0 || (block > 1 && !draft_logits) || !target_logits || !tokens || !u_accept ||
      !u_resample || !accept_len || !emitted || !workspace)
    return DFLASH_E_INVALID_ARG;
  if (workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return DFLASH_E_INVALID_ARG;
  const int nc = sample_chunks(vocab);
  const int rows = batch * block;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const int64_t stats_bytes = align256((int64_t)rows * nc * (int64_t)sizeof(float2));
  float2* dstats = reinterpret_cast<float2*>(w);
  float2* tstats = reinterpret_cast<float2*>(w + stats_bytes);
  SeqDraw* draw = reinterpret_cast<SeqDraw*>(w + 2 * stats_bytes);
  float* mass = reinterpret_cast<float*>(w + 2 * stats_bytes +
                                         align256((int64_t)batch * (int64_t)sizeof(SeqDraw)));
  cudaStream_t st = (cudaStream_t)stream;
  if ((block > 1 &&
       launch_k(true, samp_stats_kernel, dim3(nc, batch * (block - 1)), dim3(kSampThreads), 0, st,
                draft_logits, vocab, nc, dstats) != cudaSuccess) ||
      launch_k(true, samp_stats_kernel, dim3(nc, rows), dim3(kSampThreads), 0, st, target_logits,
               vocab, nc, tstats) != cudaSuccess ||
      launch_k(true, samp_accept_kernel, dim3(batch), dim3(32), 0, st, draft_logits,
               target_logits, (int)block, vocab, nc, (const float2*)dstats,
               (const float2*)tstats, tokens, u_accept, accept_len, draw) != cudaSuccess ||
      launch_k(true, samp_final_mass_kernel, dim3(nc, batch), dim3(kSampThreads), 0, st,
               draft_logits, target_logits, vocab, nc, (const SeqDraw*)draw, mass) !=
          cudaSuccess ||
      launch_k(true, samp_final_pick_kernel, dim3(batch), dim3(kSampThreads), 0, st, draft_logits,
               target_logits, vocab, nc, (const SeqDraw*)draw, (const float*)mass, u_resample,
               emitted) != cudaSuccess)
    return DFLASH_E_CUDA;
  return DFLASH_OK;
}

}  // extern "C"

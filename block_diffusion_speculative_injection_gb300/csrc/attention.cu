// Attention of the block-draft, verify, tree-verify and prefill passes.
//
// Every query row belongs to one sequence of the pass and sits at block
// index j.  Keys are cache slots of that sequence: slots < ctx_len (the
// committed / injected context) are visible to every row; block slot
// ctx_len + i is visible according to the pass's mask:
//   none   (block draft: bidirectional inside the block) -> every i < blk
//   causal (verify, prefill)                             -> i <= j
//   tree   (DDTree verify: ancestors and self)           -> bit i of anc[j]
//
// bf16, head_dim 128: one CTA takes 64 query rows = (64/G) block positions x
// the G query heads that share one KV head, so each K/V tile streamed from
// HBM feeds G heads at once.  K/V tiles of 64 slots are staged in shared
// memory with cp.async (16-byte chunks, XOR-swizzled rows) in a two-deep
// ring; QK^T and PV run on mma.sync m16n8k16 with an online softmax in
// registers (exp2 domain).  Long contexts are split across CTAs; a combine
// kernel merges the partial (m, l, O).
#include <cfloat>
#include <cmath>
#include <cstring>

#include "internal.cuh"

namespace dflash {

struct AttnK {
  const void* q;
  void* out;
  const void* kc;
  const void* vc;
  const int32_t* pass_seq;
  const int32_t* pass_ctx;
  const int32_t* pass_blk;
  int q_stride, H, Hkv, G, hd, max_ctx;
  int mask;
  const uint64_t* anc;
  int anc_words;
  int n_splits, keys_per_split;
  float* part_o;
  float* part_ml;
  int rows_total;
  float scale_log2;
  int uni_ctx, uni_blk;  // used when pass_seq == nullptr: seq = b, same lengths
};

__device__ __forceinline__ void seq_meta(const AttnK& p, int b, int& seq, int& ctx, int& blk) {
  if (p.pass_seq) {
    seq = p.pass_seq[b];
    ctx = p.pass_ctx[b];
    blk = p.pass_blk[b];
  } else {
    seq = b;
    ctx = p.uni_ctx;
    blk = p.uni_blk;
  }
}

// ---------------------------------------------------------------------------
// small PTX wrappers (legacy warp-level MMA path)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (x0, x1) -> packed bf16 high parts and packed bf16 residuals x - hi
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l =
      __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// byte offset of 16-byte chunk c (0..15) of row r in a [rows][256 B] tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ bool key_visible(int mask, int kidx, int ctx_len, int blk, int j,
                                            const uint64_t* anc_row) {
  if (kidx < ctx_len) return true;
  const int i = kidx - ctx_len;
  if (i >= blk) return false;
  if (mask == kMaskNone) return true;
  if (mask == kMaskCausal) return i <= j;
  return (anc_row[i >> 6] >> (i & 63)) & 1ull;
}

constexpr int kTileKeys = 64;
constexpr int kHd = 128;
constexpr int kAttnSmem = 3 * 64 * 256 * 2 - 64 * 256;  // Q + 2 x (K, V) = 80 KB

__global__ void __launch_bounds__(128) attn_mma_kernel(const AttnK p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* qs = sm;                   // 64 x 256 B
  uint8_t* ks0 = sm + 64 * 256;       // 2 stages x (K 16 KB, V 16 KB)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G, POS = 64 / G;
  const int b = blockIdx.z / p.n_splits, split = blockIdx.z % p.n_splits;
  const int kvh = blockIdx.y;
  int seq, ctx_len, blk;
  seq_meta(p, b, seq, ctx_len, blk);
  const int j0 = blockIdx.x * POS;
  if (j0 >= blk) return;
  const int jmax = min(j0 + POS, blk);  // exclusive
  int key_end = (p.mask == kMaskCausal) ? ctx_len + jmax : ctx_len + blk;
  // causal and draft passes: this sequence's keys in equal whole-tile
  // shares over the splits (the launch is sized for the longest context;
  // shorter ones must not leave the later splits idle).  Tree verify keeps
  // the plan's fixed share, which measured faster there.
  const int kps =
      p.mask == kMaskTree
          ? p.keys_per_split
          : min(p.keys_per_split,
                max(kTileKeys, (key_end + p.n_splits * kTileKeys - 1) / (p.n_splits * kTileKeys) *
                                   kTileKeys));
  const int k_begin = split * kps;
  const int k_stop = min(key_end, k_begin + kps);

  // this thread's two query rows (within the CTA tile) and their block index
  const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
  const int jr0 = j0 + r0 / G, jr1 = j0 + r1 / G;
  const int hr0 = kvh * G + r0 % G, hr1 = kvh * G + r1 % G;
  const bool live0 = jr0 < blk, live1 = jr1 < blk;
  const size_t grow0 = (size_t)b * p.q_stride + jr0, grow1 = (size_t)b * p.q_stride + jr1;

  if (k_begin >= k_stop) {  // empty split: neutral partial
    if (p.n_splits > 1 && (lane & 3) == 0) {
      if (live0) {
        float* ml = p.part_ml + (((size_t)split * p.rows_total + grow0) * p.H + hr0) * 2;
        ml[0] = -INFINITY;
        ml[1] = 0.f;
      }
      if (live1) {
        float* ml = p.part_ml + (((size_t)split * p.rows_total + grow1) * p.H + hr1) * 2;
        ml[0] = -INFINITY;
        ml[1] = 0.f;
      }
    }
    if (p.n_splits > 1) {
      // zero the partial outputs of this thread's columns
      for (int nt = 0; nt < 16; ++nt) {
        const int d = nt * 8 + (lane & 3) * 2;
        if (live0) {
          float* o = p.part_o + (((size_t)split * p.rows_total + grow0) * p.H + hr0) * kHd + d;
          o[0] = 0.f;
          o[1] = 0.f;
        }
        if (live1) {
          float* o = p.part_o + (((size_t)split * p.rows_total + grow1) * p.H + hr1) * kHd + d;
          o[0] = 0.f;
          o[1] = 0.f;
        }
      }
    }
    return;
  }

  const bf16* qg = static_cast<const bf16*>(p.q);
  const size_t head_base = ((size_t)seq * p.Hkv + kvh) * (size_t)p.max_ctx;
  const bf16* kg = static_cast<const bf16*>(p.kc) + head_base * kHd;
  const bf16* vg = static_cast<const bf16*>(p.vc) + head_base * kHd;

  // ---- Q tile -> shared (rows past blk are zero)
  for (int i = threadIdx.x; i < 64 * 16; i += 128) {
    const int r = i >> 4, c = i & 15;
    const int j = j0 + r / G, h = kvh * G + r % G;
    const bf16* src = qg + (((size_t)b * p.q_stride + (j < blk ? j : 0)) * p.H + h) * kHd + c * 8;
    cp_async16(smem_u32(qs + swz(r, c)), src, j < blk ? 16u : 0u);
  }
  cp_async_commit();

  auto load_kv = [&](int tile_start, int stage) {
    uint8_t* ks = ks0 + stage * (2 * 64 * 256);
    uint8_t* vs = ks + 64 * 256;
    for (int i = threadIdx.x; i < 64 * 16; i += 128) {
      const int r = i >> 4, c = i & 15;
      const int slot = tile_start + r;
      const bool in = slot < k_stop;
      const size_t off = (size_t)(in ? slot : 0) * kHd + c * 8;
      cp_async16(smem_u32(ks + swz(r, c)), kg + off, in ? 16u : 0u);
      cp_async16(smem_u32(vs + swz(r, c)), vg + off, in ? 16u : 0u);
    }
    cp_async_commit();
  };

  const int n_tiles = (k_stop - k_begin + kTileKeys - 1) / kTileKeys;
  load_kv(k_begin, 0);

  // anc words of this thread's rows (tree mask)
  const uint64_t* anc0 = nullptr;
  const uint64_t* anc1 = nullptr;
  if (p.mask == kMaskTree) {
    anc0 = p.anc + ((size_t)b * p.q_stride + (live0 ? jr0 : 0)) * p.anc_words;
    anc1 = p.anc + ((size_t)b * p.q_stride + (live1 ? jr1 : 0)) * p.anc_words;
  }
  const int mask_from = (p.mask == kMaskNone) ? ctx_len + blk
                        : (p.mask == kMaskCausal) ? ctx_len + j0 + 1
                                                  : ctx_len;

  cp_async_wait<1>();
  __syncthreads();
  uint32_t qf[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int mi = lane >> 3;
    const int r = warp * 16 + (mi & 1) * 8 + (lane & 7);
    const int c = 2 * kk + (mi >> 1);
    ldsm_x4(smem_u32(qs + swz(r, c)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int t = 0; t < n_tiles; ++t) {
    const int tile_start = k_begin + t * kTileKeys;
    if (t + 1 < n_tiles) {
      load_kv(tile_start + kTileKeys, (t + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t* ks = ks0 + (t & 1) * (2 * 64 * 256);
    const uint8_t* vs = ks + 64 * 256;

    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int mi = lane >> 3;
        const int r = np * 16 + (mi >> 1) * 8 + (lane & 7);
        const int c = 2 * kk + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(ks + swz(r, c)), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qf[kk], b0, b1);
        mma_bf16(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // scale, mask, row max
    const bool need_mask = tile_start + kTileKeys > mask_from || tile_start + kTileKeys > k_stop;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[nt][e] * p.scale_log2;
        if (need_mask) {
          const int kidx = tile_start + nt * 8 + (lane & 3) * 2 + (e & 1);
          const bool row1 = e >= 2;
          const bool vis = kidx < k_stop &&
                           key_visible(p.mask, kidx, ctx_len, blk, row1 ? jr1 : jr0,
                                       row1 ? anc1 : anc0);
          if (!vis) v = -INFINITY;
        }
        s[nt][e] = v;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - base0);
      s[nt][1] = exp2f(s[nt][1] - base0);
      s[nt][2] = exp2f(s[nt][2] - base1);
      s[nt][3] = exp2f(s[nt][3] - base1);
      rs0 += s[nt][0] + s[nt][1];
      rs1 += s[nt][2] + s[nt][3];
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= al0;
      o[nt][1] *= al0;
      o[nt][2] *= al1;
      o[nt][3] *= al1;
    }
    // O += P V.  P is split into a bf16 high part and a bf16 residual
    // (P = P_hi + P_lo, ~16 significant bits) and both halves go through the
    // tensor cores, so the probabilities keep fp32-like precision; the extra
    // MMAs are free in this HBM-bound loop.
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t a[4], alo[4];
      split_bf16(s[2 * c][0], s[2 * c][1], a[0], alo[0]);
      split_bf16(s[2 * c][2], s[2 * c][3], a[1], alo[1]);
      split_bf16(s[2 * c + 1][0], s[2 * c + 1][1], a[2], alo[2]);
      split_bf16(s[2 * c + 1][2], s[2 * c + 1][3], a[3], alo[3]);
      // two column pairs at a time: the four high-part MMAs, then the four
      // residual MMAs into the same accumulators, four MMAs apart
#pragma unroll
      for (int np = 0; np < 8; np += 2) {
        const int mi = lane >> 3;
        const int r = c * 16 + (mi & 1) * 8 + (lane & 7);
        uint32_t b[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          ldsm_x4_t(smem_u32(vs + swz(r, 2 * (np + h) + (mi >> 1))), b[h][0], b[h][1], b[h][2],
                    b[h][3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mma_bf16(o[2 * (np + h)], a, b[h][0], b[h][1]);
          mma_bf16(o[2 * (np + h) + 1], a, b[h][2], b[h][3]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mma_bf16(o[2 * (np + h)], alo, b[h][0], b[h][1]);
          mma_bf16(o[2 * (np + h) + 1], alo, b[h][2], b[h][3]);
        }
      }
    }
    __syncthreads();
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  if (p.n_splits == 1) {
    bf16* og = static_cast<bf16*>(p.out);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int d = nt * 8 + (lane & 3) * 2;
      if (live0)
        *reinterpret_cast<__nv_bfloat162*>(og + (grow0 * p.H + hr0) * kHd + d) =
            __floats2bfloat162_rn(o[nt][0] * inv0, o[nt][1] * inv0);
      if (live1)
        *reinterpret_cast<__nv_bfloat162*>(og + (grow1 * p.H + hr1) * kHd + d) =
            __floats2bfloat162_rn(o[nt][2] * inv1, o[nt][3] * inv1);
    }
  } else {
    const size_t base0 = ((size_t)split * p.rows_total + grow0) * p.H + hr0;
    const size_t base1 = ((size_t)split * p.rows_total + grow1) * p.H + hr1;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int d = nt * 8 + (lane & 3) * 2;
      if (live0)
        *reinterpret_cast<float2*>(p.part_o + base0 * kHd + d) = make_float2(o[nt][0], o[nt][1]);
      if (live1)
        *reinterpret_cast<float2*>(p.part_o + base1 * kHd + d) = make_float2(o[nt][2], o[nt][3]);
    }
    if ((lane & 3) == 0) {
      if (live0) *reinterpret_cast<float2*>(p.part_ml + base0 * 2) = make_float2(m0, l0);
      if (live1) *reinterpret_cast<float2*>(p.part_ml + base1 * 2) = make_float2(m1, l1);
    }
  }
}

constexpr int kMaxSplits = 256;

// merge split partials: one warp per (row, head), lane l holds head dims
// 4l..4l+3.  Up to kB splits, every load of the merge (row metadata, each
// split's (m, l) and partial output) is issued before any is used, so the
// kernel costs one memory round trip after its predecessor ends; more
// splits go in batches of kB.  The sums run in split order either way.
template <int kB>
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnK p) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sw[4][kMaxSplits];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x, h = blockIdx.y * 4 + warp;
  if (h >= p.H) return;
  const int b = row / p.q_stride, j = row % p.q_stride;
  int seq_, ctx_, blk_;
  seq_meta(p, b, seq_, ctx_, blk_);
  const int S = p.n_splits;
  const size_t stride = (size_t)p.rows_total * p.H;  // (row, head) units between splits
  const size_t base = (size_t)row * p.H + h;
  // partials of rows past the sequence's block were not written this pass:
  // they are read (in bounds) and then dropped with the row
  const float4* po = reinterpret_cast<const float4*>(p.part_o + base * kHd) + lane;
  const size_t ostride = stride * (kHd / 4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fma4 = [](float4& a, float w, const float4& o) {
    a.x += w * o.x;
    a.y += w * o.y;
    a.z += w * o.z;
    a.w += w * o.w;
  };
  float l = 0.f;
  if (S <= kB) {
    const float2 ml = lane < S
                          ? *reinterpret_cast<const float2*>(p.part_ml + (base + lane * stride) * 2)
                          : make_float2(-INFINITY, 0.f);
    float4 o[kB];
#pragma unroll
    for (int s = 0; s < kB; ++s)
      if (s < S) o[s] = po[s * ostride];
    float mx = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (mx == -INFINITY) mx = 0.f;
    const float w = lane < S ? exp2f(ml.x - mx) : 0.f;
    l = w * ml.y;
#pragma unroll
    for (int s = 0; s < kB; ++s)
      if (s < S) fma4(acc, __shfl_sync(0xffffffffu, w, s), o[s]);
  } else {
    // lane l takes splits l, l + 32, ...: maximum, then weights (kept in
    // shared memory for the output sum) and the weighted sum of l
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, p.part_ml[(base + s * stride) * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (mx == -INFINITY) mx = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (base + s * stride) * 2);
      const float w = exp2f(ml.x - mx);
      sw[warp][s] = w;
      l += w * ml.y;
    }
    __syncwarp();
    for (int s0 = 0; s0 < S; s0 += kB) {
      float4 o[kB];
#pragma unroll
      for (int s = 0; s < kB; ++s)
        if (s0 + s < S) o[s] = po[(s0 + s) * ostride];
#pragma unroll
      for (int s = 0; s < kB; ++s)
        if (s0 + s < S) fma4(acc, sw[warp][s0 + s], o[s]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (j >= blk_) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(static_cast<bf16*>(p.out) + base * kHd + lane * 4) = pk;
}

// few splits: a small batch keeps the registers (and so the resident warps
// that hide the loads) of the common batched case
static void (*combine_for(int splits))(const AttnK) {
  return splits <= 8 ? attn_combine_kernel<8> : attn_combine_kernel<32>;
}

// ---------------------------------------------------------------------------
// fp32 storage: one warp per (row, query head), keys visited in order
// ---------------------------------------------------------------------------
__global__ void attn_simt_f32_kernel(const AttnK p) {
  pdl_trigger();
  pdl_wait();
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= p.rows_total * p.H) return;
  const int row = wid / p.H, h = wid % p.H;
  const int b = row / p.q_stride, j = row % p.q_stride;
  int seq, ctx_len, blk;
  seq_meta(p, b, seq, ctx_len, blk);
  if (j >= blk) return;
  const int kvh = h / p.G;
  const int per = p.hd / 32;  // head_dim <= 128
  const float* qv = static_cast<const float*>(p.q) + ((size_t)row * p.H + h) * p.hd;
  float qr[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i = 0; i < per; ++i) qr[i] = qv[lane + 32 * i];
  const size_t head_base = ((size_t)seq * p.Hkv + kvh) * (size_t)p.max_ctx;
  const float* kg = static_cast<const float*>(p.kc) + head_base * p.hd;
  const float* vg = static_cast<const float*>(p.vc) + head_base * p.hd;
  const uint64_t* anc = p.mask == kMaskTree ? p.anc + (size_t)row * p.anc_words : nullptr;
  const int key_end = (p.mask == kMaskCausal) ? ctx_len + j + 1 : ctx_len + blk;
  const float scale = p.scale_log2;  // log2 domain
  float m = -INFINITY, l = 0.f;
  for (int k = 0; k < key_end; ++k) {
    if (!key_visible(p.mask, k, ctx_len, blk, j, anc)) continue;
    float dot = 0.f;
    for (int i = 0; i < per; ++i) dot += qr[i] * kg[(size_t)k * p.hd + lane + 32 * i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float sc = dot * scale;
    const float mn = fmaxf(m, sc);
    const float corr = exp2f(m - mn), pk = exp2f(sc - mn);
    l = l * corr + pk;
    for (int i = 0; i < per; ++i)
      acc[i] = acc[i] * corr + pk * vg[(size_t)k * p.hd + lane + 32 * i];
    m = mn;
  }
  float* og = static_cast<float*>(p.out) + ((size_t)row * p.H + h) * p.hd;
  for (int i = 0; i < per; ++i) og[lane + 32 * i] = acc[i] / l;
}

// number of KV splits and keys per split for a launch of `ctas` CTAs.  The
// split count minimises the estimated makespan: waves of resident CTAs (2 per
// SM) x (key tiles per split + a fixed cost of about two tiles for the Q
// load, the partial write and the combine), so that a launch never ends with
// a nearly empty extra wave of full-length splits.
static void plan_splits(int sm_count, int ctas, int64_t max_keys, size_t part_cap, int rows_heads,
                        int* n_splits, int* keys_per_split, int min_splits = 1) {
  const int64_t key_tiles = std::max<int64_t>(1, (max_keys + kTileKeys - 1) / kTileKeys);
  const int64_t slots = 2 * (int64_t)sm_count;
  int best = 1;
  int64_t best_cost = INT64_MAX;
  const int64_t s_max = std::min<int64_t>(kMaxSplits, key_tiles);
  for (int64_t sp = std::min<int64_t>(min_splits, s_max); sp <= s_max; ++sp) {
    if (sp > 1 && (size_t)sp * rows_heads > part_cap) break;
    const int64_t tiles_per = (key_tiles + sp - 1) / sp;
    if (sp > 1 && (key_tiles + tiles_per - 1) / tiles_per < sp) continue;  // same as a smaller split
    const int64_t waves = (ctas * sp + slots - 1) / slots;
    const int64_t cost = waves * (tiles_per + 2) + (sp > 1 ? 1 : 0);
    if (cost < best_cost) {
      best_cost = cost;
      best = (int)sp;
    }
  }
  *keys_per_split = 1 << 30;
  if (best > 1) {
    const int64_t tiles_per = (key_tiles + best - 1) / best;
    *keys_per_split = (int)(tiles_per * kTileKeys);
    best = (int)((key_tiles + tiles_per - 1) / tiles_per);
  }
  *n_splits = best;
}

dflash_status plan_attention(int sm_count, int batch, int H, int Hkv, int q_per_seq,
                             int64_t max_keys, int min_splits, int32_t* out) {
  if (!out || sm_count < 1 || batch < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 ||
      64 % (H / Hkv) != 0 || q_per_seq < 1 || max_keys < 1 || max_keys >= (1 << 30) ||
      min_splits < 1)
    return DFLASH_E_INVALID_ARG;
  const int POS = 64 / (H / Hkv);
  const int64_t ctas = (int64_t)((q_per_seq + POS - 1) / POS) * Hkv * batch;
  if (ctas * kMaxSplits >= (1 << 30)) return DFLASH_E_INVALID_ARG;
  int splits = 1, kps = 0;
  plan_splits(sm_count, (int)ctas, max_keys, (size_t)1 << 40, batch * q_per_seq * H, &splits, &kps,
              min_splits);
  out[0] = splits;
  out[1] = splits > 1 ? kps : (int32_t)max_keys;
  out[2] = (int32_t)(ctas * splits);
  return DFLASH_OK;
}

// SM count of the current device (cached per device)
static int device_sms() {
  static std::atomic<int> sms[kMaxDevices];
  const int dev = current_device_slot();
  if (dev < 0) return 1;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static cudaError_t ensure_attn_smem() {
  static std::atomic<bool> done[kMaxDevices];
  return ensure_smem_attr(done, attn_mma_kernel, kAttnSmem);
}

dflash_status attention(dflash_ctx* ctx, const AttnArgs& a, cudaStream_t st) {
  ProfScope prof(ctx, kProfAttn, st);
  const dflash_config& c = ctx->cfg;
  AttnK p;
  p.q = a.q;
  p.out = a.out;
  p.kc = a.kc;
  p.vc = a.vc;
  p.pass_seq = ctx->pass_seq;
  p.pass_ctx = ctx->pass_ctx;
  p.pass_blk = ctx->pass_blk;
  p.q_stride = a.q_stride;
  p.H = c.n_heads;
  p.Hkv = c.n_kv_heads;
  p.G = c.n_heads / c.n_kv_heads;
  p.hd = c.head_dim;
  p.max_ctx = c.max_ctx;
  p.mask = a.mask;
  p.anc = a.anc;
  p.anc_words = a.anc_words;
  p.rows_total = a.batch * a.q_stride;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
  p.part_o = ctx->part_o;
  p.part_ml = ctx->part_ml;
  p.n_splits = 1;
  p.keys_per_split = 1 << 30;
  p.uni_ctx = p.uni_blk = 0;

  if (c.dtype == DFLASH_F32) {
    const int warps = p.rows_total * p.H;
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, attn_simt_f32_kernel, dim3((warps + 3) / 4), dim3(128), 0, st, p));
    DF_LAUNCHED(ctx);
    return DFLASH_OK;
  }
  if (c.head_dim != kHd || 64 % p.G != 0) {
    set_error(ctx, "bf16 attention needs head_dim 128 and a GQA group dividing 64");
    return DFLASH_E_UNSUPPORTED;
  }
  const int POS = 64 / p.G;
  const int q_tiles = (a.q_stride + POS - 1) / POS;
  const int ctas = q_tiles * c.n_kv_heads * a.batch;
  // a batch's sequences differ in length: with one split the longest ones
  // set the time while the rest idle, so batched passes take two or more
  int splits = 1;
  plan_splits(ctx->sm_count, ctas, a.max_keys_ub, ctx->part_rows_cap, p.rows_total * p.H, &splits,
              &p.keys_per_split, a.batch > 1 ? 2 : 1);
  p.n_splits = splits;
  DF_CUDA_TRY(ctx, ensure_attn_smem());
  dim3 grid(q_tiles, c.n_kv_heads, a.batch * splits);
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, attn_mma_kernel, dim3(grid), dim3(128), kAttnSmem, st, p));
  DF_LAUNCHED(ctx);
  if (splits > 1) {
    dim3 g2(p.rows_total, (c.n_heads + 3) / 4);
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, combine_for(splits), dim3(g2), dim3(128), 0, st, p));
    DF_LAUNCHED(ctx);
  }
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// op-level entry: block attention over caller-provided K/V
// ---------------------------------------------------------------------------
static bool op_shape_ok(int batch, int H, int Hkv, int hd, int ctx_len, int block) {
  return batch >= 1 && H >= 1 && Hkv >= 1 && H % Hkv == 0 && hd == kHd && 64 % (H / Hkv) == 0 &&
         ctx_len >= 0 && block >= 1 && block <= 64 && (int64_t)ctx_len + block < (1 << 30);
}

int64_t block_attention_workspace(int batch, int H, int Hkv, int hd, int ctx_len, int block) {
  if (!op_shape_ok(batch, H, Hkv, hd, ctx_len, block)) return -1;
  const int G = H / Hkv, POS = 64 / G;
  const int ctas = ((block + POS - 1) / POS) * Hkv * batch;
  int splits = 1, kps = 0;
  plan_splits(device_sms(), ctas, ctx_len + block, (size_t)1 << 40, batch * block * H, &splits,
              &kps);
  if (splits == 1) return 0;
  return (int64_t)splits * batch * block * H * (kHd + 2) * (int64_t)sizeof(float);
}

dflash_status block_attention(int batch, int H, int Hkv, int hd, int ctx_len, int block, int causal,
                              const void* q, const void* k, const void* v, void* out,
                              void* workspace, int64_t workspace_bytes, cudaStream_t st) {
  if (!op_shape_ok(batch, H, Hkv, hd, ctx_len, block)) return DFLASH_E_INVALID_ARG;
  if (!q || !k || !v || !out) return DFLASH_E_INVALID_ARG;
  // 16-byte copies of Q/K/V rows and partials, 8-byte stores of the output
  auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(out) || (workspace && !a16(workspace)))
    return DFLASH_E_INVALID_ARG;
  AttnK p;
  memset(&p, 0, sizeof(p));
  p.q = q;
  p.out = out;
  p.kc = k;
  p.vc = v;
  p.q_stride = block;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.hd = hd;
  p.max_ctx = ctx_len + block;
  p.mask = causal ? kMaskCausal : kMaskNone;
  p.rows_total = batch * block;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)hd));
  p.uni_ctx = ctx_len;
  p.uni_blk = block;
  const int POS = 64 / p.G;
  const int q_tiles = (block + POS - 1) / POS;
  const int ctas = q_tiles * Hkv * batch;
  // splits limited by the caller's workspace
  const size_t per_split = (size_t)p.rows_total * H * (kHd + 2) * sizeof(float);
  const size_t cap_units = workspace ? (size_t)workspace_bytes / per_split * p.rows_total * H : 0;
  int splits = 1;
  plan_splits(device_sms(), ctas, p.max_ctx, cap_units, p.rows_total * H, &splits,
              &p.keys_per_split);
  if (splits > 1) {
    p.part_o = static_cast<float*>(workspace);
    p.part_ml = p.part_o + (size_t)splits * p.rows_total * H * kHd;
  }
  p.n_splits = splits;
  if (ensure_attn_smem() != cudaSuccess) return DFLASH_E_CUDA;
  dim3 grid(q_tiles, Hkv, batch * splits);
  if (launch_k(true, attn_mma_kernel, dim3(grid), dim3(128), kAttnSmem, st, p) != cudaSuccess)
    return DFLASH_E_CUDA;
  if (splits > 1) {
    dim3 g2(p.rows_total, (H + 3) / 4);
    if (launch_k(true, combine_for(splits), dim3(g2), dim3(128), 0, st, p) != cudaSuccess)
      return DFLASH_E_CUDA;
  }
  return DFLASH_OK;
}

}  // namespace dflash

// Dense projections of the target and of the drafter: out = X . W^T.
//
// bf16 storage: tcgen05 tensor-core kernel.  The weight matrix is always the
// 128-row MMA operand (A) and the token rows are the N operand (B, 16..256
// wide), so one kernel covers the weight-streaming regime of a 16-row block
// and the compute-bound regime of a 512-row batch.  Operands are staged in
// shared memory by TMA (128-byte swizzle) through an mbarrier ring; one
// thread issues the MMAs, accumulators live in tensor memory and are read
// back by every warp of the CTA (4, or 8 on tiles of more than 32 token
// rows).  The projection's epilogue (RoPE + cache scatter, SwiGLU, residual
// add, store) is fused: straight from tensor memory when the tile takes the
// whole K range, else the K splits of the tile form a thread-block cluster
// and sum their partial tiles through distributed shared memory in split
// order.  The lm_head's epilogue reduces each 128-feature vocabulary tile to
// per-row candidates (best logits, max and sum of exp) instead of writing the
// logits; the plain fp32 result remains for the small fp32 model.
//
// f32 storage: a tiled SIMT kernel (fp32 FMA) writes per-split fp32 slabs
// and an epilogue kernel sums them in a fixed order (the small fp32 model).
#include <climits>
#include <cstdio>
#include <cstring>

#include "epilogue.cuh"
#include "internal.cuh"

namespace dflash {

constexpr int kMaxSeg = 12;

struct TmapSet {
  CUtensorMap m[kMaxSeg];
};

struct TcParams {
  int M, N, K;
  int n_seg;
  int seg_begin[kMaxSeg + 1];
  int BN, stages, kb_per_split, n_kb;
  int m_tiles, n_tiles;  // the persistent form walks m_tiles * n_tiles tiles
  int sk_tiles;          // ... the last sk_tiles of them split along K (stream-K)
  float* sk_part;        // [CTA][BN columns][128 lanes] fp32 partial tiles
  unsigned long long* sk_ticket;
  int32_t* sk_cnt;       // [sk_tiles] partials arrived
  float* out;
  long long split_stride;
  int32_t* status;
  EpiArgs epi;
};

// lm_head tile reduction: the CTA's 128 x BN logits sit feature-major in
// shared memory (row pitch BN + 1 floats, so the TMEM-order writes and the
// reads below are free of bank conflicts).  Ties go to the lower id.
//   K = 2 (argmax and margin): one thread per token row scans the tile's
//   features in id order (a strict "greater" keeps the lower id ahead).
//   K > 2 (top-k): one warp per token row, lane l holding features l + 32 i;
//   K rounds of a warp arg-max, the winner's lane retiring that feature.
// With vr_lse the tile's (max, sum exp(x - max)) goes alongside.
__device__ __forceinline__ void vocab_tile_reduce(const EpiArgs& e, const float* tile, int pitch,
                                                  int nf, int n0, int m0, int BN, int M) {
  const int K = e.vr_k;
  if (K == 2) {
    for (int u = threadIdx.x; u < BN; u += blockDim.x) {
      const int t = m0 + u;
      if (t >= M) break;
      const size_t pb = (size_t)t * gridDim.y + blockIdx.y;
      const float* col = tile + u;
      float v1 = -INFINITY, v2 = -INFINITY;
      int i1 = INT_MAX, i2 = INT_MAX;
      for (int f = 0; f < nf; ++f) {
        const float x = col[f * pitch];
        if (x > v2) {
          if (x > v1) {
            v2 = v1;
            i2 = i1;
            v1 = x;
            i1 = n0 + f;
          } else {
            v2 = x;
            i2 = n0 + f;
          }
        }
      }
      e.vr_id[pb * 2] = i1;
      e.vr_id[pb * 2 + 1] = i2;
      e.vr_v[pb * 2] = v1;
      e.vr_v[pb * 2 + 1] = v2;
      if (e.vr_lse) {
        float se = 0.f;
        for (int f = 0; f < nf; ++f) se += __expf(col[f * pitch] - v1);
        *reinterpret_cast<float2*>(e.vr_lse + pb * 2) = make_float2(v1, se);
      }
    }
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int u = warp; u < BN; u += nw) {
    const int t = m0 + u;
    if (t >= M) break;
    const size_t pb = (size_t)t * gridDim.y + blockIdx.y;
    float x[4], v[4];
    int id[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int f = lane + 32 * i;
      x[i] = f < nf ? tile[f * pitch + u] : -INFINITY;
      v[i] = x[i];
      id[i] = f < nf ? n0 + f : INT_MAX;
    }
    float top = -INFINITY;
    for (int k = 0; k < K; ++k) {
      // this lane's best remaining feature (its ids ascend with i)
      float bv = v[0];
      int bi = id[0];
#pragma unroll
      for (int i = 1; i < 4; ++i)
        if (v[i] > bv) {
          bv = v[i];
          bi = id[i];
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (k == 0) top = bv;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (id[i] == bi && bi != INT_MAX) {
          v[i] = -INFINITY;
          id[i] = INT_MAX;
        }
      if (lane == k) {
        e.vr_id[pb * K + k] = bi;
        e.vr_v[pb * K + k] = bv;
      }
    }
    if (e.vr_lse) {
      float se = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) se += x[i] == -INFINITY ? 0.f : __expf(x[i] - top);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
      if (lane == 0) *reinterpret_cast<float2*>(e.vr_lse + pb * 2) = make_float2(top, se);
    }
  }
}

__global__ void __launch_bounds__(384, 1)
    gemm_tc_kernel(const __grid_constant__ TmapSet wmaps, const __grid_constant__ CUtensorMap xmap,
                   const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int BN = p.BN, S = p.stages;
  const uint32_t a_bytes = 128 * 64 * 2;
  const uint32_t b_bytes = (uint32_t)BN * 64 * 2;
  uint8_t* a_s = smem;
  uint8_t* b_s = smem + S * a_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(b_s + S * b_bytes);
  uint64_t* empty = full + S;
  uint64_t* accum = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // SwiGLU: CTA x takes features f0 = 64 x of both the gate and the up
  // segment; its 128-row weight tile is gate rows f0..f0+63 over up rows
  // f0..f0+63 (two 64-row TMA boxes), so SiLU(gate) * up forms in one CTA
  const bool swiglu = p.epi.kind == kEpiSwiGLU;
  // grid: x = token tile, y = weight tile, z = K split.  The token tiles of
  // one weight tile are neighbours in launch order, so they run together and
  // the second reads the weight tile from L2 (weights carry an evict-first
  // hint: a token tile a wave later would find them gone from L2 and fetch
  // them from HBM again)
  const int n0 = swiglu ? (int)blockIdx.y * 64 : (int)blockIdx.y * 128, m0 = blockIdx.x * BN;
  const int kb0 = blockIdx.z * p.kb_per_split;
  const int kb1 = min(p.n_kb, kb0 + p.kb_per_split);
  const int nkb = kb1 - kb0;
  int seg = 0;
  if (!swiglu)
    while (seg + 1 < p.n_seg && p.seg_begin[seg + 1] <= n0) ++seg;
  const int wrow0 = swiglu ? n0 : n0 - p.seg_begin[seg];
  const uint32_t tmem_cols = BN <= 32 ? 32u : (BN <= 64 ? 64u : (BN <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // let the next kernel launch now: its CTAs take free slots and wait for
  // this grid's completion before they read anything it writes
  pdl_trigger();

  if (warp == 0) {
   if (lane == 0) {
    // TMA producer
    tma_prefetch_desc(&wmaps.m[seg]);
    if (swiglu) tma_prefetch_desc(&wmaps.m[1]);
    tma_prefetch_desc(&xmap);
    // Weights are never written by an earlier kernel: fill the first stages'
    // weight tiles before waiting on the preceding kernel (programmatic
    // dependent launch), then add the activation tiles.  Weights are read
    // once per pass: their lines are first in line for eviction from L2.
    const uint64_t wpol = l2_policy_evict_first();
    const int pre = min(S, nkb);
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], a_bytes + b_bytes);
      if (swiglu) {
        tma_load_2d_hint(a_s + i * a_bytes, &wmaps.m[0], (kb0 + i) * 64, wrow0, &full[i], wpol);
        tma_load_2d_hint(a_s + i * a_bytes + a_bytes / 2, &wmaps.m[1], (kb0 + i) * 64, wrow0,
                         &full[i], wpol);
      } else {
        tma_load_2d_hint(a_s + i * a_bytes, &wmaps.m[seg], (kb0 + i) * 64, wrow0, &full[i], wpol);
      }
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i)
      tma_load_2d(b_s + i * b_bytes, &xmap, (kb0 + i) * 64, m0, &full[i]);
    int issued = pre;
    for (int i = pre; i < nkb; ++i) {
      const int s = i % S;
      const uint32_t ph = (uint32_t)(i / S) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u, p.status)) break;
      mbar_arrive_expect_tx(&full[s], a_bytes + b_bytes);
      const int kx = (kb0 + i) * 64;
      if (swiglu) {
        tma_load_2d_hint(a_s + s * a_bytes, &wmaps.m[0], kx, wrow0, &full[s], wpol);
        tma_load_2d_hint(a_s + s * a_bytes + a_bytes / 2, &wmaps.m[1], kx, wrow0, &full[s], wpol);
      } else {
        tma_load_2d_hint(a_s + s * a_bytes, &wmaps.m[seg], kx, wrow0, &full[s], wpol);
      }
      tma_load_2d(b_s + s * b_bytes, &xmap, kx, m0, &full[s]);
      ++issued;
    }
    // drain: every issued copy has landed before this thread leaves
    for (int i = max(0, issued - S); i < issued; ++i)
      mbar_wait(&full[i % S], (uint32_t)(i / S) & 1u, p.status);
   }
    __syncwarp();  // lanes 1..31 park here instead of spinning beside the producer
  } else if (warp == 1) {
   if (lane == 0) {
    // MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, BN);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % S;
      const uint32_t ph = (uint32_t)(i / S) & 1u;
      if (!mbar_wait(&full[s], ph, p.status)) break;
      tc_fence_after();
      const uint64_t ad = sw128_desc(smem_u32(a_s + s * a_bytes));
      const uint64_t bd = sw128_desc(smem_u32(b_s + s * b_bytes));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc_mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&empty[s]);
    }
    tc_commit(accum);
   }
    __syncwarp();
  }

  // epilogue: TMEM lane = weight row (output feature), column = token row.
  // Every thread orders itself after the preceding kernel before writing.
  pdl_wait();
  mbar_wait_sleep(accum, 0, p.status);
  __syncwarp();
  tc_fence_after();
  // a warp reads TMEM lane quarter warp % 4; with 8 warps the two groups of
  // 4 take alternate 16-row chunks
  const int quarter = warp & 3, c_first = (warp >> 2) * 16, c_step = ((int)blockDim.x >> 7) * 16;
  if (p.epi.kind == kEpiVocab) {  // lm_head: reduce the tile over its 128 features
    const EpiArgs& e = p.epi;
    const int pitch = BN + 1;
    float* tile = reinterpret_cast<float*>(smem);  // the pipeline buffers are idle now
    const int f = quarter * 32 + lane, feat = n0 + f;
    for (int c = c_first; c < BN; c += c_step) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) tile[f * pitch + c + i] = v[i];
      if (e.vr_logits && feat < p.N) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = m0 + c + i;
          const int vi = t < p.M ? __ldg(e.vr_vec + t) : -1;
          if (vi >= 0) e.vr_logits[(size_t)vi * p.N + feat] = v[i];
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, tmem_cols);
    vocab_tile_reduce(e, tile, pitch, min(128, p.N - n0), n0, m0, BN, p.M);
    return;
  }
  if (p.epi.kind == kEpiSlab) {  // plain fp32 result (lm_head logits), no K split
    const int feat = n0 + quarter * 32 + lane;
    for (int c = c_first; c < BN; c += c_step) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = m0 + c + i;
        if (t < p.M && feat < p.N) p.out[(size_t)t * p.N + feat] = v[i];
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, tmem_cols);
    return;
  }
  if (p.epi.splits == 1) {  // no K split: straight from TMEM
    run_epilogue_direct<bf16>(p.epi, tmem, n0, m0, BN, reinterpret_cast<float*>(smem),
                              (int)threadIdx.x, (int)blockDim.x);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, tmem_cols);
    return;
  }

  // fused epilogue over the cluster of K splits: partial tile -> own smem
  // (the pipeline buffers are idle now), then a cluster-wide reduction
  __shared__ int32_t s_meta[256 * 3];
  float* part = reinterpret_cast<float*>(smem);
  for (int c = c_first; c < BN; c += c_step) {
    float v[16];
    tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) part[(c + i) * 128 + quarter * 32 + lane] = v[i];
  }
  for (int u = threadIdx.x; u < BN; u += blockDim.x) {
    const int t = m0 + u;
    int pos = -1, seq = -1, slot = -1;
    if (t < p.M && (p.epi.kind == kEpiQKV || p.epi.kind == kEpiInject)) {
      pos = p.epi.row_pos[t];
      seq = p.epi.row_seq[t];
      slot = p.epi.kind == kEpiQKV ? p.epi.row_slot[t] : pos;
    }
    s_meta[u * 3] = pos;
    s_meta[u * 3 + 1] = seq;
    s_meta[u * 3 + 2] = slot;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, tmem_cols);
  cluster_sync();
  run_epilogue_cluster<bf16>(p.epi, n0, m0, BN, part, s_meta);
  cluster_sync();  // peers may still be reading this CTA's partial tile
}

// ---------------------------------------------------------------------------
// Persistent form for passes of more tiles than SMs (wide token tiles, no K
// split): one CTA per SM walks the tiles t = v, v + gridDim.x, ... (token
// tile fastest, as in the grid above; v = blockIdx.x, or the CTA's ticket
// when the tiles past the last full round are split along K as a stream-K
// remainder, below).  Warp 0 issues TMA through the
// stage ring continuously across tiles, warp 1 issues the MMAs into one of
// two accumulators in tensor memory (columns 0 and 256), and warps 2..13 (three
// groups of four) run the epilogue of tile i from one accumulator while the
// MMAs of tile i + 1 fill the other, so the epilogue no longer idles the
// tensor pipe.  The epilogue's scratch (one 16 x 128 fp32 exchange buffer per
// group, 256 row offsets) has its own shared memory after the ring.
// ---------------------------------------------------------------------------
constexpr int kPersistEpiWarps = 12;
constexpr int kPersistThreads = 64 + 32 * kPersistEpiWarps;
constexpr uint32_t kPersistScratch = (kPersistEpiWarps / 4) * 16 * 128 * 4 + 256 * 8 + 256 * 4;
constexpr size_t kPersistSmemMax = 227 * 1024;  // the opt-in limit per CTA

// kSK: the launch has a stream-K remainder (p.sk_tiles > 0); the instance
// without one compiles to the plain round-robin walk.
template <bool kSK>
__global__ void __launch_bounds__(kPersistThreads, 1)
    gemm_tc_persistent_kernel(const __grid_constant__ TmapSet wmaps,
                              const __grid_constant__ CUtensorMap xmap, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int BN = p.BN, S = p.stages;
  const uint32_t a_bytes = 128 * 64 * 2;
  const uint32_t b_bytes = (uint32_t)BN * 64 * 2;
  uint8_t* a_s = smem;
  uint8_t* b_s = smem + S * a_bytes;
  float* scratch = reinterpret_cast<float*>(b_s + S * b_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(scratch) + kPersistScratch);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;   // [2] accumulator ready for the epilogue
  uint64_t* acc_empty = acc_full + 2;  // [2] accumulator read out (every epilogue warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* vid_slot = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool swiglu = p.epi.kind == kEpiSwiGLU;
  const int n_tiles_total = p.m_tiles * p.n_tiles;
  const int nkb = p.n_kb;
  // tile -> (first output feature, first token row, weight segment and row)
  auto tile_geo = [&](int tile, int& n0, int& m0, int& seg, int& wrow0) {
    const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
    n0 = swiglu ? nt * 64 : nt * 128;
    m0 = mt * BN;
    seg = 0;
    if (!swiglu)
      while (seg + 1 < p.n_seg && p.seg_begin[seg + 1] <= n0) ++seg;
    wrow0 = swiglu ? n0 : n0 - p.seg_begin[seg];
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kPersistEpiWarps);
    }
    mbar_fence_init();
    // With a stream-K remainder a CTA waits only for CTAs of lower work index,
    // and work indices are handed out in the order CTAs start: those CTAs are
    // running, so the waits end whatever else shares the GPU.  Every launch
    // takes exactly gridDim.x tickets, all before it lets the next kernel
    // launch, so ticket % gridDim.x numbers the CTAs 0 .. gridDim.x - 1.
    int v = (int)blockIdx.x;
    if (kSK) {
      v = (int)(atomicAdd(p.sk_ticket, 1ull) % (unsigned long long)gridDim.x);
      __threadfence();
    }
    *vid_slot = v;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int vid = kSK ? *vid_slot : (int)blockIdx.x;
  pdl_trigger();

  // Work of CTA vid: the k-blocks [lo, hi) of the last R tiles, taken in
  // (tile, k-block) order and cut into G contiguous ranges, then the whole
  // tiles vid, vid + G, ... below D = tiles - R.  R < G, so a range spans at
  // most nkb k-blocks and touches at most two tiles.  A piece that ends its
  // tile is that tile's owner: it adds the partial sums of the lower CTAs'
  // pieces of the tile and runs the epilogue; the other piece (the head of
  // the next tile, where the range ends) stores its partial sum to the CTA's
  // slot and counts itself in.  The pieces run first, the non-owner one
  // first of all: the partials an owner waits for are then the lower CTAs'
  // first items, and the owner's epilogue overlaps the first whole tile (a
  // short piece late in the order would wait for an accumulator still held by
  // the previous tile's epilogue).
  const int G = (int)gridDim.x, R = kSK ? p.sk_tiles : 0, D = n_tiles_total - R;
  const long long U = (long long)R * nkb;
  auto sk_at = [&](int c) -> int { return (int)(U * c / G); };
  const int nd = vid < D ? (D - 1 - vid) / G + 1 : 0;
  const int lo = sk_at(vid), hi = sk_at(vid + 1);
  const int n_sk = (kSK && hi > lo) ? (hi - 1) / nkb - lo / nkb + 1 : 0;
  const int n_items = nd + n_sk;
  auto item = [&](int i, int& tile, int& kb0, int& kb1, bool& owner) {
    if (i >= n_sk) {
      tile = vid + (i - n_sk) * G;
      kb0 = 0;
      kb1 = nkb;
      owner = true;
      return;
    }
    const int a = lo / nkb + (n_sk == 2 ? 1 - i : 0);
    const int s0 = max(lo, a * nkb), e0 = min(hi, (a + 1) * nkb);
    tile = D + a;
    kb0 = s0 - a * nkb;
    kb1 = e0 - a * nkb;
    owner = e0 == (a + 1) * nkb;
  };

  if (warp == 0) {
    if (lane == 0) {
      // TMA producer: k-block g of this CTA's stream goes to stage g % S
      tma_prefetch_desc(&xmap);
      const uint64_t wpol = l2_policy_evict_first();
      uint32_t g = 0;
      bool ok = true, waited = false;
      for (int it = 0; ok && it < n_items; ++it) {
        int tile, kb0, kb1, n0, m0, seg, wrow0;
        bool owner;
        item(it, tile, kb0, kb1, owner);
        tile_geo(tile, n0, m0, seg, wrow0);
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          const int s = (int)(g % (uint32_t)S);
          const uint32_t ph = (g / (uint32_t)S) & 1u;
          if (g >= (uint32_t)S && !mbar_wait(&empty[s], ph ^ 1u, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], a_bytes + b_bytes);
          const int kx = kb * 64;
          if (swiglu) {
            tma_load_2d_hint(a_s + s * a_bytes, &wmaps.m[0], kx, wrow0, &full[s], wpol);
            tma_load_2d_hint(a_s + s * a_bytes + a_bytes / 2, &wmaps.m[1], kx, wrow0, &full[s], wpol);
          } else {
            tma_load_2d_hint(a_s + s * a_bytes, &wmaps.m[seg], kx, wrow0, &full[s], wpol);
          }
          // the activations are the preceding kernel's output: wait for it
          // once, after the first weight tiles are on their way
          if (!waited) {
            pdl_wait();
            waited = true;
          }
          tma_load_2d(b_s + s * b_bytes, &xmap, kx, m0, &full[s]);
        }
      }
      // drain: every issued copy has landed before this thread leaves
      for (uint32_t i = g > (uint32_t)S ? g - (uint32_t)S : 0u; i < g; ++i)
        mbar_wait(&full[i % (uint32_t)S], (i / (uint32_t)S) & 1u, p.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer: work item i accumulates into buffer i & 1
      const uint32_t idesc = idesc_bf16_f32(128, BN);
      uint32_t g = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_items; ++i) {
        int tile, kb0, kb1;
        bool owner;
        item(i, tile, kb0, kb1, owner);
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait(&acc_empty[buf], ((i >> 1) - 1) & 1, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * 256);
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          const int s = (int)(g % (uint32_t)S);
          if (!mbar_wait(&full[s], (g / (uint32_t)S) & 1u, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_desc(smem_u32(a_s + s * a_bytes));
          const uint64_t bd = sw128_desc(smem_u32(b_s + s * b_bytes));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&acc_full[buf]);
      }
    }
    __syncwarp();
  } else {
    // epilogue warps 2..13 (ordered after the preceding kernel before they
    // read the residual or write anything)
    pdl_wait();
    const int ep_tid = (int)threadIdx.x - 64, ep_threads = kPersistThreads - 64;
    const int quarter = warp & 3, grp = (ep_tid >> 5) >> 2, ngrp = ep_threads >> 7;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const size_t slot_elems = (size_t)BN * 128;
    for (int i = 0; i < n_items; ++i) {
      const int buf = i & 1;
      // a wait that gives up has set the status word; the warps go on
      // together regardless (one warp leaving alone would strand the others
      // at the epilogue's named barriers, which have no time limit)
      mbar_wait_sleep(&acc_full[buf], (i >> 1) & 1, p.status);
      __syncwarp();
      tc_fence_after();
      int tile, kb0, kb1, n0, m0, seg, wrow0;
      bool owner;
      item(i, tile, kb0, kb1, owner);
      const uint32_t acc = tmem + (uint32_t)(buf * 256);
      if (kSK && !owner) {
        // partial sum -> this CTA's slot, [column][lane] so a warp's stores
        // of one column are 128 contiguous bytes
        float* slot = p.sk_part + (size_t)vid * slot_elems + quarter * 32 + lane;
        for (int c = grp * 16; c < BN; c += ngrp * 16) {
          float v[16];
          tmem_ld16(acc + lane_off + (uint32_t)c, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) __stcg(slot + (size_t)(c + k) * 128, v[k]);
        }
        __threadfence();
        epi_sync_all(ep_threads);
        if (ep_tid == 0) atomicAdd(p.sk_cnt + (tile - D), 1);
      } else {
        if (kSK && i < n_sk && kb0 > 0) {
          // lower CTAs whose ranges end inside this tile, each with one
          // partial in its slot: wait for all, then add them in CTA order
          const int a = tile - D, t0 = a * nkb;
          int first = vid, expect = 0;
          for (int c = vid - 1; c >= 0 && sk_at(c + 1) > t0; --c) {
            first = c;
            if (sk_at(c + 1) > sk_at(c)) ++expect;
          }
          if (ep_tid == 0) {
            int32_t* cnt = p.sk_cnt + a;
            bool ok = ld_acquire_gpu(cnt) >= expect;
            const uint64_t t_start = global_ns();
            for (uint32_t it = 1; !ok && it < kSpinLimit; ++it) {
              __nanosleep(256);
              ok = ld_acquire_gpu(cnt) >= expect;
              if ((it & 255u) == 0 && global_ns() - t_start > 2000000000ull) break;
            }
            if (!ok) set_dev_status(p.status, kDevTimeout);
            *cnt = 0;  // every partial of this tile has arrived: ready for the next launch
            __threadfence();
          }
          epi_sync_all(ep_threads);
          for (int c = grp * 16; c < BN; c += ngrp * 16) {
            float v[16];
            tmem_ld16(acc + lane_off + (uint32_t)c, v);
            for (int q = first; q < vid; ++q) {
              if (sk_at(q + 1) == sk_at(q)) continue;
              const float* src = p.sk_part + (size_t)q * slot_elems + quarter * 32 + lane;
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] += __ldcg(src + (size_t)(c + k) * 128);
            }
            tmem_st16(acc + lane_off + (uint32_t)c, v);
          }
          tmem_wait_st();
          tc_fence_before();
          epi_sync_all(ep_threads);
          tc_fence_after();
        }
        tile_geo(tile, n0, m0, seg, wrow0);
        run_epilogue_direct<bf16>(p.epi, acc, n0, m0, BN, scratch, ep_tid, ep_threads);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// fp32 storage: the epilogue runs as its own kernel over the slab (splits = 1)
__global__ void __launch_bounds__(128) epilogue_f32_kernel(const EpiArgs e) {
  pdl_wait();
  pdl_trigger();
  run_epilogue<float>(e, blockIdx.x * 128, 0, e.M);
}

// ---------------------------------------------------------------------------
// fp32 SIMT GEMM (small fp32 models)
// ---------------------------------------------------------------------------
struct SegPtrs {
  const float* w[kMaxSeg];
  int begin[kMaxSeg + 1];
  int n;
};

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ x, int M, int K,
                                                       const SegPtrs segs, int N,
                                                       float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float xs[16][64 + 1];
  __shared__ float wsm[16][64 + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int r = i / 16, kk = i % 16;
      const int m = m0 + r, n = n0 + r, k = k0 + kk;
      xs[kk][r] = (m < M && k < K) ? x[(size_t)m * K + k] : 0.f;
      float wv = 0.f;
      if (n < N && k < K) {
        int s = 0;
        while (s + 1 < segs.n && segs.begin[s + 1] <= n) ++s;
        wv = segs.w[s][(size_t)(n - segs.begin[s]) * K + k];
      }
      wsm[kk][r] = wv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = wsm[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) out[(size_t)m * N + n] = acc[i][j];
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static dflash_status get_tmap(dflash_ctx* ctx, const void* ptr, int64_t rows, int64_t cols,
                              int box_rows, const CUtensorMap** out);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || rank < 1 || rank > 3) return false;
  memset(m, 0, sizeof(*m));
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t bx[3], estride[3] = {1u, 1u, 1u};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gstride[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), gdim,
            gstride, bx, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

dflash_status tmap_2d(dflash_ctx* ctx, const void* ptr, int64_t rows, int64_t cols, int box_rows,
                      const CUtensorMap** out) {
  return get_tmap(ctx, ptr, rows, cols, box_rows, out);
}

// 2-D bf16 tensor [rows][cols] (row-major), box [box_rows][64], 128-byte swizzle.
static dflash_status get_tmap(dflash_ctx* ctx, const void* ptr, int64_t rows, int64_t cols,
                              int box_rows, const CUtensorMap** out) {
  auto key = std::make_tuple(ptr, rows, cols, box_rows);
  auto it = ctx->tmaps.find(key);
  if (it != ctx->tmaps.end()) {
    *out = &it->second;
    return DFLASH_OK;
  }
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    set_error(ctx, "cuTensorMapEncodeTiled entry point unavailable");
    return DFLASH_E_CUDA;
  }
  CUtensorMap m;
  memset(&m, 0, sizeof(m));
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estride[2] = {1u, 1u};
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim, gstride,
                  box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error(ctx, "cuTensorMapEncodeTiled failed (%d) rows=%lld cols=%lld box=%d", (int)r,
              (long long)rows, (long long)cols, box_rows);
    return DFLASH_E_CUDA;
  }
  auto res = ctx->tmaps.emplace(key, m);
  *out = &res.first->second;
  return DFLASH_OK;
}

static size_t tc_smem_bytes(int BN, int stages);

// Token rows up to which tiles run 4 warps, 2 CTAs per SM, with a 108 KB
// ring each (about 2 x rows flops per weight byte: at or under the machine
// balance; measured at 64 and 128 rows against one CTA per SM with a 200 KB
// ring and 8 warps).  Wider tiles hold an SM alone with 12 warps.
constexpr int kSmallTileRows = 128;

// Planning kind of an lm_head whose epilogue keeps the top 2 per row and
// 128-id tile and nothing else (no log-sum-exp, no logits): its reduction
// runs from tensor memory in registers, so it may take the persistent form,
// where the reduction of one tile overlaps the next tile's main loop.
constexpr int kPlanVocabTop2 = 7;

static int tc_stages(int BN) {
  const int per = 128 * 64 * 2 + BN * 64 * 2;
  // tiles of up to kSmallTileRows token rows stream weights: 2 CTAs per SM
  // (a third, left for the next launch's weight prefetch, measured slower:
  // its 3 stages per CTA hold too little in flight)
  // (108 KB of ring: two CTAs, each with its alignment pad, barriers, 3 KB
  // of static shared memory and the 1 KB per-CTA reserve, fit in 228 KB)
  int budget = (BN <= kSmallTileRows) ? 108 * 1024 : 200 * 1024;
  int s = budget / per;
  if (s > 8) s = 8;
  if (s < 2) s = 2;
  return s;
}

static size_t tc_smem_bytes(int BN, int stages) {
  return 1024 + (size_t)stages * (128 * 64 * 2 + BN * 64 * 2) + (2 * stages + 1) * 8 + 16;
}

// tile shape, K split and launch shape of one bf16 GEMM launch
struct TcPlan {
  int BN, m_tiles, n_tiles, stages, n_kb, splits, kb_per, threads;
  size_t smem_bytes;
  int persistent;  // CTAs of the persistent form (0: one CTA per tile)
  int sk_tiles;    // tiles of the persistent form's stream-K remainder
};

static size_t persist_smem_bytes(int BN, int stages) {
  return 1024 + (size_t)stages * (128 * 64 * 2 + BN * 64 * 2) + kPersistScratch +
         (2 * stages + 4) * 8 + 16;
}

static cudaError_t ensure_tc_smem() {
  static std::atomic<bool> done[kMaxDevices];
  return ensure_smem_attr(done, gemm_tc_kernel, 210 * 1024);
}
static cudaError_t ensure_persist_smem() {
  static std::atomic<bool> done[kMaxDevices];
  static std::atomic<bool> done_sk[kMaxDevices];
  const cudaError_t e = ensure_smem_attr(done, gemm_tc_persistent_kernel<false>, (int)kPersistSmemMax);
  if (e != cudaSuccess) return e;
  return ensure_smem_attr(done_sk, gemm_tc_persistent_kernel<true>, (int)kPersistSmemMax);
}

// the plan for a given number of token tiles
static TcPlan plan_tiles(int sm_count, int M, int N, int K, int kind, int max_splits, int m_tiles) {
  TcPlan t;
  t.m_tiles = m_tiles;
  int BN = (M + t.m_tiles - 1) / t.m_tiles;
  BN = ((BN + 15) / 16) * 16;
  t.BN = BN < 16 ? 16 : BN;
  t.stages = tc_stages(t.BN);
  t.n_tiles = (N + 127) / 128;
  t.n_kb = K / 64;
  const int ctas = t.n_tiles * t.m_tiles;
  // K splits: as many as fit in ONE wave of resident CTAs (a partial second
  // wave would double the latency of these short, bandwidth-bound launches)
  const int per_sm = (t.BN <= kSmallTileRows) ? 2 : 1;
  const int slots = per_sm * sm_count;
  int splits = ctas >= slots ? 1 : slots / ctas;
  // the K splits of a tile form one thread-block cluster (portable size <= 8);
  // a SwiGLU tile holds gate and up rows in one CTA and is never split
  const int max_cluster_splits = kind == kEpiSwiGLU ? 1 : 8;  // SwiGLU: direct epilogue only
  if (splits > max_cluster_splits) splits = max_cluster_splits;
  if (splits > max_splits) splits = max_splits;
  if (splits > t.n_kb / 4) splits = t.n_kb / 4;
  if (splits < 1 || kind == kEpiSlab || kind == kEpiVocab || kind == kPlanVocabTop2) splits = 1;
  // ... and every cluster of the launch resident at once: clusters that wait
  // for a second wave double the launch time.  A cluster sits inside one GPC,
  // so fewer than slots / size clusters fit; on GB300 (152 SMs, 2 CTAs per
  // SM) between 0.875 and 0.97 of that number were resident for cluster
  // sizes 2..8, so the plan counts on 7/8 of it.
  while (splits > 1 && (int64_t)ctas * splits * 8 > (int64_t)slots * 7) --splits;
  // the cluster epilogue stages each split's fp32 partial tile (BN x 128) in
  // the CTA's ring memory: a tile whose partial does not fit is not split
  if (splits > 1 && (size_t)t.BN * 128 * 4 > (size_t)t.stages * (128 * 64 * 2 + t.BN * 64 * 2))
    splits = 1;
  t.kb_per = (t.n_kb + splits - 1) / splits;
  t.splits = (t.n_kb + t.kb_per - 1) / t.kb_per;
  // tiles of more than kSmallTileRows token rows hold an SM alone (shared
  // memory): three groups of 4 warps share the epilogue at no occupancy cost
  t.threads = t.BN > kSmallTileRows ? 384 : 128;
  t.smem_bytes = tc_smem_bytes(t.BN, t.stages);
  // More tiles than SMs, wide token tiles and no K split: the persistent
  // form (one CTA per SM, the epilogue of a tile overlapping the next tile's
  // main loop).  The lm_head's general vocabulary epilogue stages its tile
  // in the ring's memory, so it keeps one CTA per tile; the top-2 one does
  // not (kPlanVocabTop2).
  t.persistent = 0;
  t.sk_tiles = 0;
  if (t.splits == 1 && t.BN > 64 && kind != kEpiSlab && kind != kEpiVocab &&
      (int64_t)t.n_tiles * t.m_tiles > sm_count) {
    t.persistent = sm_count;
    t.threads = kPersistThreads;
    const int per = 128 * 64 * 2 + t.BN * 64 * 2;
    const size_t fixed = persist_smem_bytes(t.BN, 0);
    int st = (int)((kPersistSmemMax - fixed) / (per + 16));
    if (st > 8) st = 8;
    t.stages = st;
    t.smem_bytes = persist_smem_bytes(t.BN, st);
    // The tiles past the last full round (R = tiles mod CTAs) would run on R
    // CTAs while the rest idle; split along K over all CTAs instead, when the
    // idle share is worth the partial-sum exchange (R at most 3/4 of the CTAs)
    // and every CTA gets at least 8 k-blocks of it.  Not for the top-2
    // lm_head: its many rounds leave little idle, and its measured time grew.
    const int R = (int)(((int64_t)t.n_tiles * t.m_tiles) % sm_count);
    if (kind != kPlanVocabTop2 && R > 0 && R * 4 <= sm_count * 3 &&
        (int64_t)R * t.n_kb >= 8LL * sm_count)
      t.sk_tiles = R;
  }
  return t;
}

static TcPlan plan_tc(int sm_count, int M, int N, int K, int kind, int max_splits) {
  // Token tiles as wide as the MMA allows: a 64-column K block takes about
  // the same time at 80, 128, 144 or 256 token rows, so a pass that leaves
  // SMs idle is split along K rather than cut into narrower tiles.  A pass
  // that K splits cannot spread within one wave (a single split) takes more,
  // narrower token tiles while they still fit one wave: each CTA keeps its
  // main loop and gets a shorter epilogue (QKV at 512 rows: three tiles of
  // 176 rows on 144 SMs instead of two of 256 on 96).
  TcPlan t = plan_tiles(sm_count, M, N, K, kind, max_splits, (M + 255) / 256);
  if (t.splits == 1 && t.persistent == 0 && t.m_tiles > 1 && kind != kEpiSlab && kind != kEpiVocab &&
      kind != kPlanVocabTop2) {
    int m = t.m_tiles;
    while ((int64_t)t.n_tiles * (m + 1) <= sm_count && (M + m) / (m + 1) > 48) ++m;  // >= 64-row tiles
    if (m > t.m_tiles) t = plan_tiles(sm_count, M, N, K, kind, max_splits, m);
  }
  return t;
}

dflash_status plan_gemm(int sm_count, int M, int N, int K, int kind, int max_splits, int32_t* out) {
  if (!out || sm_count < 1 || M < 1 || N < 1 || K < 64 || K % 64 != 0 || max_splits < 1 ||
      kind < kEpiSlab || kind > kPlanVocabTop2 || (kind == kEpiSwiGLU && N % 128 != 0))
    return DFLASH_E_INVALID_ARG;
  const TcPlan t = plan_tc(sm_count, M, N, K, kind, max_splits);
  out[0] = t.BN;
  out[1] = t.m_tiles;
  out[2] = t.n_tiles;
  out[3] = t.stages;
  out[4] = t.splits;
  out[5] = t.threads;
  out[6] = (int32_t)t.smem_bytes;
  out[7] = t.persistent;
  return DFLASH_OK;
}

dflash_status gemm(dflash_ctx* ctx, const void* x, int M, int K, const GemmSegs& segs,
                   const EpiArgs& epi_in, int max_splits, int* splits_used, cudaStream_t st) {
  float* out = ctx->ws;
  if (M <= 0) {
    *splits_used = 1;
    return DFLASH_OK;
  }
  int N = 0;
  for (int i = 0; i < segs.n; ++i) N += segs.rows[i];
  if (segs.n < 1 || segs.n > kMaxSeg) return DFLASH_E_INVALID_ARG;
  // result bytes: the fp32 logits, or the vocabulary partials of every tile
  const double out_bytes = epi_in.kind == kEpiVocab
                               ? (double)M * ((N + 127) / 128) * (8.0 * epi_in.vr_k +
                                                                  (epi_in.vr_lse ? 8.0 : 0.0))
                               : 4.0 * M * N;
  ProfScope prof(ctx, kProfGemm, st, ((double)N * K + (double)M * K) * ctx->esize + out_bytes,
                 2.0 * M * N * K);

  if (ctx->cfg.dtype == DFLASH_F32) {
    if (epi_in.kind == kEpiVocab) {
      set_error(ctx, "the fused lm_head reduction needs bf16 storage");
      return DFLASH_E_UNSUPPORTED;
    }
    SegPtrs sp;
    memset(&sp, 0, sizeof(sp));
    sp.n = segs.n;
    sp.begin[0] = 0;
    for (int i = 0; i < segs.n; ++i) {
      sp.w[i] = static_cast<const float*>(segs.w[i]);
      sp.begin[i + 1] = sp.begin[i] + segs.rows[i];
    }
    if ((size_t)M * N > ctx->ws_elems) {
      set_error(ctx, "GEMM output %dx%d exceeds workspace", M, N);
      return DFLASH_E_CAPACITY;
    }
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, gemm_f32_kernel, dim3(grid), dim3(256), 0, st, static_cast<const float*>(x), M, K, sp, N, out));
    DF_LAUNCHED(ctx);
    *splits_used = 1;
    if (epi_in.kind != kEpiSlab) {
      EpiArgs e = epi_in;
      e.M = M;
      e.N = N;
      e.splits = 1;
      e.split_stride = (long long)M * N;
      e.slab = out;
      e.status = ctx->dev_status;
      const int groups = e.kind == kEpiSwiGLU ? (e.F + 127) / 128 : (N + 127) / 128;
      DF_CUDA_TRY(ctx, launch_k(ctx->pdl, epilogue_f32_kernel, dim3(groups), dim3(128), 0, st, e));
      DF_LAUNCHED(ctx);
    }
    return DFLASH_OK;
  }

  if (K % 64 != 0) {
    set_error(ctx, "GEMM K=%d is not a multiple of 64", K);
    return DFLASH_E_UNSUPPORTED;
  }
  for (int i = 0; i + 1 < segs.n; ++i)
    if (segs.rows[i] % 128 != 0) {
      set_error(ctx, "GEMM segment %d has %d rows (not a multiple of 128)", i, segs.rows[i]);
      return DFLASH_E_UNSUPPORTED;
    }
  const bool vocab_top2 = epi_in.kind == kEpiVocab && epi_in.vr_k == 2 && !epi_in.vr_lse &&
                          !epi_in.vr_logits;
  const TcPlan plan =
      plan_tc(ctx->sm_count, M, N, K, vocab_top2 ? kPlanVocabTop2 : epi_in.kind, max_splits);
  const int m_tiles = plan.m_tiles, BN = plan.BN, stages = plan.stages, n_tiles = plan.n_tiles;
  const int n_kb = plan.n_kb;
  const int kb_per = plan.kb_per;
  int splits = plan.splits;
  if (epi_in.kind == kEpiSlab && (size_t)M * N > ctx->ws_elems) {
    set_error(ctx, "GEMM output %dx%d exceeds workspace", M, N);
    return DFLASH_E_CAPACITY;
  }
  if (epi_in.kind == kEpiVocab &&
      (epi_in.vr_k < 2 || epi_in.vr_k > 16 || !epi_in.vr_id || !epi_in.vr_v ||
       (epi_in.vr_logits && !epi_in.vr_vec) ||
       (plan.persistent == 0 &&
        (size_t)128 * (BN + 1) * sizeof(float) > (size_t)stages * (128 * 64 * 2 + BN * 64 * 2)))) {
    set_error(ctx, "lm_head reduction: bad candidate count or buffers");
    return DFLASH_E_INVALID_ARG;
  }
  if (epi_in.kind == kEpiSwiGLU &&
      (segs.n != 2 || segs.rows[0] != epi_in.F || segs.rows[1] != epi_in.F || epi_in.F % 64 != 0)) {
    set_error(ctx, "SwiGLU GEMM needs gate and up segments of F %% 64 == 0 rows each");
    return DFLASH_E_UNSUPPORTED;
  }

  TmapSet maps;
  memset(&maps, 0, sizeof(maps));
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.seg_begin[0] = 0;
  for (int i = 0; i < segs.n; ++i) {
    const CUtensorMap* m = nullptr;
    // SwiGLU: 64-row boxes (gate rows over up rows in one 128-row tile)
    DF_TRY(get_tmap(ctx, segs.w[i], segs.rows[i], K, epi_in.kind == kEpiSwiGLU ? 64 : 128, &m));
    maps.m[i] = *m;
    p.seg_begin[i + 1] = p.seg_begin[i] + segs.rows[i];
  }
  const CUtensorMap* xm = nullptr;
  DF_TRY(get_tmap(ctx, x, M, K, BN, &xm));
  p.M = M;
  p.N = N;
  p.K = K;
  p.n_seg = segs.n;
  p.BN = BN;
  p.stages = stages;
  p.kb_per_split = kb_per;
  p.n_kb = n_kb;
  p.out = out;
  p.split_stride = (long long)M * N;
  p.status = ctx->dev_status;
  p.epi = epi_in;
  p.epi.M = M;
  p.epi.N = N;
  p.epi.splits = splits;
  p.epi.split_stride = (long long)M * N;
  p.epi.slab = out;
  p.epi.status = ctx->dev_status;

  p.m_tiles = m_tiles;
  p.n_tiles = n_tiles;
  p.sk_tiles = plan.sk_tiles;
  p.sk_part = ctx->sk_part;
  p.sk_ticket = static_cast<unsigned long long*>(ctx->sk_sync);
  p.sk_cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ctx->sk_sync) + 8);
  if (plan.persistent > 0) {
    DF_CUDA_TRY(ctx, ensure_persist_smem());
    const int ctas = (int)std::min<int64_t>((int64_t)m_tiles * n_tiles, plan.persistent);
    auto kern = plan.sk_tiles > 0 ? gemm_tc_persistent_kernel<true> : gemm_tc_persistent_kernel<false>;
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, kern, dim3(ctas), dim3(kPersistThreads), plan.smem_bytes, st,
                              maps, *xm, p));
    DF_LAUNCHED(ctx);
    *splits_used = 1;
    return DFLASH_OK;
  }
  DF_CUDA_TRY(ctx, ensure_tc_smem());
  dim3 grid(m_tiles, n_tiles, splits);
  const size_t smem_bytes = plan.smem_bytes;
  const dim3 block(plan.threads);
  // the K splits of a tile form a cluster; an unsplit launch needs none
  if (splits > 1) {
    DF_CUDA_TRY(ctx, launch_k_cluster(ctx->pdl, dim3(1, 1, splits), gemm_tc_kernel, grid, block,
                                      smem_bytes, st, maps, *xm, p));
  } else {
    DF_CUDA_TRY(ctx, launch_k(ctx->pdl, gemm_tc_kernel, grid, block, smem_bytes, st, maps, *xm, p));
  }
  DF_LAUNCHED(ctx);
  *splits_used = splits;
  return DFLASH_OK;
}

}  // namespace dflash

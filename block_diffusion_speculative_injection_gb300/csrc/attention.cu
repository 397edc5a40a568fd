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
// HBM feeds G heads at once.  Q and the K/V tiles (128 keys) arrive by TMA;
// S = Q K^T and O += P V run on tcgen05 with the accumulators in tensor
// memory; the online softmax (exp2 domain) runs in one warp group, two
// threads per query row, each taking 64 of the 128 keys of a tile
// (attn_tc_kernel).  Long contexts are split across CTAs; a combine kernel
// merges the partial (m, l, O).
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
  int q_stride, H, Hkv, G, hd;
  KvPages kp;  // cache slot -> row of the K/V tensors
  int mask;
  const uint64_t* anc;
  int anc_words;
  int n_splits, keys_per_split;
  float* part_o;
  float* part_ml;
  int rows_total;
  float scale_log2;
  int uni_ctx, uni_blk;  // used when pass_seq == nullptr: seq = b, same lengths
  int32_t* status;       // sticky device status (bounded waits that gave up)
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

// (x0, x1) -> packed bf16 high parts and packed bf16 residuals x - hi
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l =
      __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
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

constexpr int kHd = 128;
constexpr int kTK = 128;  // keys per tile

// 2^x on the special-function unit (approximate, flushing results below the
// normal range to zero); P never needs more than fp32's normal range
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// bf16 attention on the 5th-generation tensor cores.
//
// One CTA: 64 query rows (64 / G block positions x the G query heads of one
// KV head) against one split of the sequence's keys, in tiles of 128 keys.
// Shared memory (1024-aligned), 128-byte-swizzled K-major boxes of 64 columns:
//   Q     [64 rows][128 hd]             2 boxes of 8 KB       (TMA, 3-D box)
//   stage s = 0, 1: K [128 keys][128 hd] 2 boxes of 16 KB; V the same
//   P buffer u = 0, 1: P_hi [64 rows][128 keys] 2 boxes of 8 KB; P_lo the same
// Tensor memory (512 columns): S buffers at columns 0 and 128 (fp32 scores of
// a tile), O at column 256 (fp32 [64 rows][128 hd]).  An M = 64 accumulator
// keeps row m in lane (m / 16) * 32 + m % 16, so warp w of the softmax group
// owns rows 16w .. 16w + 15 in its lanes 0 .. 15.
//
// Warps 0-3 (softmax): per tile, read S, mask, running max, P = exp2(S - m)
// split into a bf16 high part and a bf16 residual (P keeps ~16 bits), write
// P to shared memory in the MMA's K-major layout.  The running max used for
// the exponentials is raised only when a tile's max exceeds it by more than
// 8 (a factor 256): then O is rescaled in tensor memory (after the previous
// P.V has completed) and the sum l with it.  Any consistent max gives the
// same O / l; the threshold keeps the rescales rare.
// Warp 4 (producer): TMA of Q, then K and V tiles into a two-stage ring.
// Warp 5 (MMA): S(t) = Q K(t)^T, then O += P_hi(t-1) V(t-1) + P_lo(t-1) V(t-1)
// with V as an MN-major operand, so S of the next tile forms while the
// softmax works on the current one.
// Only one CTA fits an SM (shared memory), so the 512-column allocation never
// waits on another CTA of this kernel, and no other kernel of the library
// that holds tensor memory fits beside it.
// ---------------------------------------------------------------------------
constexpr uint32_t kQBox = 64 * 128, kQBytes = 2 * kQBox;
constexpr uint32_t kKBox = kTK * 128, kKBytes = 2 * kKBox;
constexpr uint32_t kPBox = 64 * 128, kPBytes = 4 * kPBox;
constexpr uint32_t kOffKV = kQBytes;
constexpr uint32_t kOffP = kOffKV + 2 * 2 * kKBytes;
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
constexpr int kAttnSmem = (int)kOffBar + 256 + 1024;  // barriers + alignment slack
constexpr int kAttnThreads = 192;
constexpr uint32_t kTmemCols = 512, kTmemO = 256;
constexpr float kRescaleLog2 = 8.f;

struct AttnMaps {
  CUtensorMap q, k, v;
};

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnMaps maps, const AttnK p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G, POS = 64 / G;
  const int b = blockIdx.z / p.n_splits, split = blockIdx.z % p.n_splits;
  const int kvh = blockIdx.y;
  int seq, ctx_len, blk;
  seq_meta(p, b, seq, ctx_len, blk);
  const int j0 = blockIdx.x * POS;
  if (j0 >= blk) return;
  const int jmax = min(j0 + POS, blk);  // exclusive
  const int key_end = (p.mask == kMaskCausal) ? ctx_len + jmax : ctx_len + blk;
  // causal and draft passes: this sequence's keys in equal whole-tile shares
  // over the splits (the launch is sized for the longest context); tree
  // verify keeps the plan's fixed share unless its keys need more (the plan
  // is sized from a host bound on the length; the splits always cover every
  // key, whatever that bound was when a graph of this launch was captured)
  const int share = max(kTK, (key_end + p.n_splits * kTK - 1) / (p.n_splits * kTK) * kTK);
  const int kps = p.mask == kMaskTree ? max(p.keys_per_split, share) : share;
  const int k_begin = split * kps;
  const int k_stop = min(key_end, k_begin + kps);

  // the row this thread works on (softmax warps; lanes t and t + 16 share
  // row 16 w + t)
  const bool row_thr = warp < 4;
  const int r = warp * 16 + (lane & 15);
  const int jr = j0 + r / G, hr = kvh * G + r % G;
  const bool live = row_thr && jr < blk;
  const size_t grow = (size_t)b * p.q_stride + jr;

  if (k_begin >= k_stop) {  // empty split: neutral partial
    if (p.n_splits > 1 && live) {
      const size_t base = ((size_t)split * p.rows_total + grow) * p.H + hr;
      if (lane < 16) *reinterpret_cast<float2*>(p.part_ml + base * 2) = make_float2(-INFINITY, 0.f);
      float4* o = reinterpret_cast<float4*>(p.part_o + base * kHd) + (lane >> 4) * (kHd / 8);
      for (int i = 0; i < kHd / 8; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const int n_tiles = (k_stop - k_begin + kTK - 1) / kTK;

  uint8_t* const qs = sm;
  uint8_t* const kvs = sm + kOffKV;   // stage s: K at s * 2 * kKBytes, V after it
  uint8_t* const ps = sm + kOffP;     // buffer u: hi boxes, then lo boxes
  uint64_t* const bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* const q_full = bars;
  uint64_t* const k_full = bars + 1;
  uint64_t* const v_full = bars + 3;
  uint64_t* const k_empty = bars + 5;
  uint64_t* const v_empty = bars + 7;
  uint64_t* const s_full = bars + 9;
  uint64_t* const s_free = bars + 11;
  uint64_t* const p_full = bars + 13;
  uint64_t* const pv_done = bars + 15;
  uint32_t* const tslot = reinterpret_cast<uint32_t*>(bars + 17);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  int32_t* const status = p.status;

  if (warp == 4) {
    if (lane == 0) {
      // ---- producer: K(t) once S(t-2) has read its stage, V(t) once
      // P.V(t-2) has; K runs one tile ahead of V in issue order
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      mbar_arrive_expect_tx(q_full, kQBytes);
      const int qz = b * p.q_stride + j0;
      tma_load_3d(qs, &maps.q, 0, kvh * G, qz, q_full);
      tma_load_3d(qs + kQBox, &maps.q, 64, kvh * G, qz, q_full);
      // a tile is one page (k_begin and the tile stride are multiples of the
      // page size); pass setup has checked that every page is mapped
      static_assert(kTK == kPageSlots, "one key tile per KV page");
      int k_issued = 0, v_issued = 0;
      // page of tile t (a raw table read, consumed only when the tile is
      // loaded), and the tile's first row in the K/V tensors; an unmapped
      // page, which pass setup rules out, loads page 0 and flags the pass
      auto tile_page = [&](int t) -> int {
        return p.kp.tab ? p.kp.tab[seq * p.kp.pps + (k_begin + t * kTK) / kPageSlots] : 0;
      };
      auto load = [&](int t, bool is_v, int pg) -> bool {
        long long row;
        if (!p.kp.tab) {
          row = kv_row(p.kp, p.Hkv, seq, kvh, k_begin + t * kTK);
        } else if (pg < 0 || pg >= p.kp.n_pages) {
          set_dev_status(status, kDevCapacity);
          row = 0;
        } else {
          row = ((long long)pg * p.Hkv + kvh) * kPageSlots;
        }
        const int y = (int)row;
        const int st = t & 1;
        uint64_t* empty = is_v ? &v_empty[st] : &k_empty[st];
        uint64_t* full = is_v ? &v_full[st] : &k_full[st];
        if (t >= 2 && !mbar_wait(empty, ((t >> 1) - 1) & 1, status)) return false;
        uint8_t* dst = kvs + st * 2 * kKBytes + (is_v ? kKBytes : 0);
        const CUtensorMap* map = is_v ? &maps.v : &maps.k;
        mbar_arrive_expect_tx(full, kKBytes);
        tma_load_2d(dst, map, 0, y, full);
        tma_load_2d(dst + kKBox, map, 64, y, full);
        return true;
      };
      // pages are read one tile ahead, so that the table read's latency
      // hides behind the wait for a free ring stage
      int pg_k = tile_page(0), pg_v = 0;
      for (int t = 0; t <= n_tiles; ++t) {
        const int pg_next = t + 1 < n_tiles ? tile_page(t + 1) : 0;
        if (t < n_tiles) {
          if (!load(t, false, pg_k)) break;
          k_issued = t + 1;
        }
        if (t >= 1) {
          if (!load(t - 1, true, pg_v)) break;
          v_issued = t;
        }
        pg_v = pg_k;
        pg_k = pg_next;
      }
      // every issued copy has landed before this thread leaves
      mbar_wait(q_full, 0, status);
      for (int t = max(0, k_issued - 2); t < k_issued; ++t)
        mbar_wait(&k_full[t & 1], (t >> 1) & 1, status);
      for (int t = max(0, v_issued - 2); t < v_issued; ++t)
        mbar_wait(&v_full[t & 1], (t >> 1) & 1, status);
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      // ---- MMA issuer: S(t), then P.V(t-1)
      const uint32_t id_s = idesc_bf16_f32(64, kTK);
      const uint32_t id_o = idesc_bf16_f32(64, kHd) | kIdescBMajorMN;
      const uint32_t qa = smem_u32(qs);
      bool ok = mbar_wait(q_full, 0, status);
      for (int t = 0; ok && t <= n_tiles; ++t) {
        if (t < n_tiles) {
          const int st = t & 1;
          if (!mbar_wait(&k_full[st], (t >> 1) & 1, status)) break;
          if (t >= 2 && !mbar_wait(&s_free[st], ((t >> 1) - 1) & 1, status)) break;
          tc_fence_after();
          const uint32_t ka = smem_u32(kvs + st * 2 * kKBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_bf16(tmem + st * kTK, sw128_desc(qa + (kk >> 2) * kQBox + (kk & 3) * 32),
                        sw128_desc(ka + (kk >> 2) * kKBox + (kk & 3) * 32), id_s,
                        kk > 0 ? 1u : 0u);
          tc_commit(&s_full[st]);
          tc_commit(&k_empty[st]);
        }
        if (t >= 1) {
          const int u = t - 1, su = u & 1;
          if (!mbar_wait(&p_full[su], (u >> 1) & 1, status)) break;
          if (!mbar_wait(&v_full[su], (u >> 1) & 1, status)) break;
          tc_fence_after();
          const uint32_t va = smem_u32(kvs + su * 2 * kKBytes + kKBytes);
          const uint32_t pa = smem_u32(ps + su * kPBytes);
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc_mma_bf16(tmem + kTmemO,
                          sw128_desc(pa + half * 2 * kPBox + (kk >> 2) * kPBox + (kk & 3) * 32),
                          sw128_desc_mn(va + kk * 16 * 128, kKBox), id_o,
                          (u > 0 || half > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&pv_done[su]);
          tc_commit(&v_empty[su]);
        }
      }
    }
    __syncwarp();
  } else {
    // ---- softmax warps 0..3: lanes t and t + 16 share row 16 w + t; the
    // half h = lane / 16 holds columns 64 h .. 64 h + 63 of every S tile
    // (keys) and of O (head dims)
    const int h = lane >> 4;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint64_t* anc = nullptr;
    if (p.mask == kMaskTree)
      anc = p.anc + ((size_t)b * p.q_stride + (live ? jr : 0)) * p.anc_words;
    const int mask_from = (p.mask == kMaskNone)     ? ctx_len + blk
                          : (p.mask == kMaskCausal) ? ctx_len + j0 + 1
                                                    : ctx_len;
    // bits below n set (n clamped to 0..32)
    auto below = [](int n) -> uint32_t {
      return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
    };
    // visibility of keys kb .. kb+31 for this thread's row
    auto visible32 = [&](int kb) -> uint32_t {
      uint32_t m = below(k_stop - kb);
      if (p.mask == kMaskCausal) return m & below(ctx_len + jr + 1 - kb);
      if (p.mask == kMaskNone) return m & below(ctx_len + blk - kb);
      // tree: the context, then block key i where bit i of the ancestor set
      const int i0 = kb - ctx_len;
      uint32_t tb = 0;
      if (i0 >= 0) {
        const int w = i0 >> 6, sh = i0 & 63;
        uint64_t x = w < p.anc_words ? anc[w] >> sh : 0ull;
        if (sh > 32 && w + 1 < p.anc_words) x |= anc[w + 1] << (64 - sh);
        tb = (uint32_t)x;
      } else if (i0 > -32) {
        tb = (uint32_t)(anc[0] << (-i0));
      }
      return m & (below(-i0) | (tb & below(blk - i0)));
    };
    const float scale = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;  // l: this thread's half of the row sum
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const int st = t & 1;
      const int tile_start = k_begin + t * kTK;
      const int kb0 = tile_start + 64 * h;
      if (lane == 0) ok = mbar_wait(&s_full[st], (t >> 1) & 1, status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = tile_start + kTK > mask_from || tile_start + kTK > k_stop;
      // pass 1: tile max of the visible scores (scaled after the max: scale > 0)
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld_half32_nowait<64>(lane_base + st * kTK + c * 32, v);
        tmem_wait_ld();
        if (need_mask) {
          const uint32_t vis = visible32(kb0 + 32 * c);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            mx = fmaxf(mx, ((vis >> i) & 1u) ? __uint_as_float(v[i]) : -INFINITY);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(v[i]));
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * scale;
      // raise the running max only when it would otherwise grow by > 2^8
      const bool resc = mx > m_used + kRescaleLog2;
      const float alpha = resc ? ex2_approx(m_used - mx) : 1.f;
      if (__any_sync(0xffffffffu, resc) && t > 0) {
        // O holds tiles 0 .. t-1 once P.V(t-1) has completed
        if (lane == 0) ok = mbar_wait(&pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld_half32_nowait<64>(lane_base + kTmemO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_half32<64>(lane_base + kTmemO + c * 32, o);
        }
        tmem_wait_st();
      }
      if (resc) {
        l *= alpha;
        m_used = mx;
      }
      const float nbase = m_used == -INFINITY ? 0.f : -m_used;
      // the P buffer of this tile was last read by P.V(t-2)
      if (t >= 2) {
        if (lane == 0) ok = mbar_wait(&pv_done[st], ((t >> 1) - 1) & 1, status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      // pass 2: P = 2^(s * scale - max), split into a bf16 high part and a
      // bf16 residual, stored in the K-major layout of the P.V MMA's A
      // operand (this half's 64 keys are box h)
      uint8_t* const pb = ps + st * kPBytes + h * kPBox;
      float rs = 0.f;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld_half32_nowait<64>(lane_base + st * kTK + c * 32, v);
        tmem_wait_ld();
        const uint32_t vis = need_mask ? visible32(kb0 + 32 * c) : 0xffffffffu;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float e[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int k = q8 * 8 + i;
            e[i] = ex2_approx(fmaf(__uint_as_float(v[k]), scale, nbase));
            if (need_mask && !((vis >> k) & 1u)) e[i] = 0.f;
            rs += e[i];
          }
          uint4 hi, lo;
          split_bf16(e[0], e[1], hi.x, lo.x);
          split_bf16(e[2], e[3], hi.y, lo.y);
          split_bf16(e[4], e[5], hi.z, lo.z);
          split_bf16(e[6], e[7], hi.w, lo.w);
          const int c8 = c * 4 + q8;
          const uint32_t off = (uint32_t)r * 128 + ((uint32_t)(c8 ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(pb + off) = hi;
          *reinterpret_cast<uint4*>(pb + 2 * kPBox + off) = lo;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[st]);
      l += rs;
      // a partial last tile: the V rows past the split's keys may hold any
      // bits (another sequence's rows, or a caller's tensor); zero them so
      // that P = 0 never meets a non-finite value
      if (tile_start + kTK > k_stop) {
        if (lane == 0) ok = mbar_wait(&v_full[st], (t >> 1) & 1, status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int first = k_stop - tile_start;
        uint8_t* vs = kvs + st * 2 * kKBytes + kKBytes;
        for (int i = warp * 32 + lane; i < (kTK - first) * 16; i += 128) {
          const int row = first + (i >> 4), ch = i & 15;
          *reinterpret_cast<uint4*>(vs + (ch >> 3) * kKBox + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[st]);
    }
    // ---- epilogue: this half of the row's O (unnormalised) once the last
    // P.V is done
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    if (ok) {
      const int u = n_tiles - 1;
      if (lane == 0) ok = mbar_wait(&pv_done[u & 1], (u >> 1) & 1, status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t pbase = ((size_t)split * p.rows_total + grow) * p.H + hr;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld_half32_nowait<64>(lane_base + kTmemO + c * 32, o);
        tmem_wait_ld();
        const int d0 = 64 * h + 32 * c;
        if (live && p.n_splits == 1) {
          uint4* og = reinterpret_cast<uint4*>(static_cast<bf16*>(p.out) + (grow * p.H + hr) * kHd + d0);
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(o[q8 * 8 + 2 * i]) * inv,
                                                        __uint_as_float(o[q8 * 8 + 2 * i + 1]) * inv);
              w[i] = *reinterpret_cast<uint32_t*>(&hv);
            }
            og[q8] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else if (live) {
          float4* po = reinterpret_cast<float4*>(p.part_o + pbase * kHd + d0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
        }
      }
      if (live && h == 0 && p.n_splits > 1)
        *reinterpret_cast<float2*>(p.part_ml + pbase * 2) = make_float2(m_used, l);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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
  const float* const kc = static_cast<const float*>(p.kc);
  const float* const vc = static_cast<const float*>(p.vc);
  const uint64_t* anc = p.mask == kMaskTree ? p.anc + (size_t)row * p.anc_words : nullptr;
  const int key_end = (p.mask == kMaskCausal) ? ctx_len + j + 1 : ctx_len + blk;
  const float scale = p.scale_log2;  // log2 domain
  float m = -INFINITY, l = 0.f;
  for (int k = 0; k < key_end; ++k) {
    if (!key_visible(p.mask, k, ctx_len, blk, j, anc)) continue;
    const long long kr = kv_row(p.kp, p.Hkv, seq, kvh, k);
    if (kr < 0) {
      if (lane == 0) set_dev_status(p.status, kDevCapacity);
      continue;
    }
    const float* kg = kc + (size_t)kr * p.hd;
    const float* vg = vc + (size_t)kr * p.hd;
    float dot = 0.f;
    for (int i = 0; i < per; ++i) dot += qr[i] * kg[lane + 32 * i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float sc = dot * scale;
    const float mn = fmaxf(m, sc);
    const float corr = exp2f(m - mn), pk = exp2f(sc - mn);
    l = l * corr + pk;
    for (int i = 0; i < per; ++i) acc[i] = acc[i] * corr + pk * vg[lane + 32 * i];
    m = mn;
  }
  float* og = static_cast<float*>(p.out) + ((size_t)row * p.H + h) * p.hd;
  for (int i = 0; i < per; ++i) og[lane + 32 * i] = acc[i] / l;
}

// number of KV splits and keys per split for a launch of `ctas` CTAs.  The
// split count minimises the estimated makespan: waves of resident CTAs (one
// per SM) x (key tiles per split + a fixed cost of about two tiles for the Q
// load, the partial write and the combine), so that a launch never ends with
// a nearly empty extra wave of full-length splits.
static void plan_splits(int sm_count, int ctas, int64_t max_keys, size_t part_cap, int rows_heads,
                        int* n_splits, int* keys_per_split, int min_splits = 1) {
  const int64_t key_tiles = std::max<int64_t>(1, (max_keys + kTK - 1) / kTK);
  const int64_t slots = (int64_t)sm_count;
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
    *keys_per_split = (int)(tiles_per * kTK);
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
  return ensure_smem_attr(done, attn_tc_kernel, kAttnSmem);
}

// Q tensor map: [rows][H][128] bf16 read as a 3-D box of (64 of hd) x (the G
// heads of one KV head) x (64/G block positions)
static bool q_map(CUtensorMap* m, const void* q, int H, int64_t rows, int G) {
  const uint64_t dims[3] = {(uint64_t)kHd, (uint64_t)H, (uint64_t)rows};
  const uint64_t strides[2] = {(uint64_t)kHd * 2, (uint64_t)H * kHd * 2};
  const uint32_t box[3] = {64u, (uint32_t)G, (uint32_t)(64 / G)};
  return encode_tmap_bf16(m, q, 3, dims, strides, box);
}
// K or V rows [rows][128] bf16, box of 128 rows x 64
static bool kv_map(CUtensorMap* m, const void* base, int64_t rows) {
  const uint64_t dims[2] = {(uint64_t)kHd, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)kHd * 2};
  const uint32_t box[2] = {64u, (uint32_t)kTK};
  return encode_tmap_bf16(m, base, 2, dims, strides, box);
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
  p.kp = ctx_pages(ctx);
  p.status = ctx->dev_status;
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
  AttnMaps maps;
  const int64_t kv_rows = (int64_t)ctx->n_pages * c.n_kv_heads * kPageSlots;
  if (kv_rows >= (int64_t)1 << 31) {
    set_error(ctx, "bf16 attention needs pages * n_kv_heads * %d < 2^31", kPageSlots);
    return DFLASH_E_UNSUPPORTED;
  }
  {
    const CUtensorMap* mk = nullptr;
    const CUtensorMap* mv = nullptr;
    DF_TRY(tmap_2d(ctx, a.kc, kv_rows, kHd, kTK, &mk));
    DF_TRY(tmap_2d(ctx, a.vc, kv_rows, kHd, kTK, &mv));
    maps.k = *mk;
    maps.v = *mv;
    // Q maps are cached under a key no 2-D map uses (a negative box height)
    const auto key = std::make_tuple(a.q, (int64_t)p.rows_total, (int64_t)c.n_heads, -p.G);
    auto it = ctx->tmaps.find(key);
    if (it == ctx->tmaps.end()) {
      CUtensorMap m;
      if (!q_map(&m, a.q, c.n_heads, p.rows_total, p.G)) {
        set_error(ctx, "cuTensorMapEncodeTiled failed for the query map");
        return DFLASH_E_CUDA;
      }
      it = ctx->tmaps.emplace(key, m).first;
    }
    maps.q = it->second;
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
  DF_CUDA_TRY(ctx, launch_k(ctx->pdl, attn_tc_kernel, dim3(grid), dim3(kAttnThreads), kAttnSmem, st,
                            maps, p));
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
         ctx_len >= 0 && block >= 1 && block <= 64 && (int64_t)ctx_len + block < (1 << 30) &&
         (int64_t)batch * Hkv * (ctx_len + block) < ((int64_t)1 << 31) &&
         (int64_t)batch * block * H < ((int64_t)1 << 31);
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
  p.kp = KvPages{nullptr, 0, 0, ctx_len + block};
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
  plan_splits(device_sms(), ctas, (int64_t)ctx_len + block, cap_units, p.rows_total * H, &splits,
              &p.keys_per_split);
  if (splits > 1) {
    p.part_o = static_cast<float*>(workspace);
    p.part_ml = p.part_o + (size_t)splits * p.rows_total * H * kHd;
  }
  p.n_splits = splits;
  if (ensure_attn_smem() != cudaSuccess) return DFLASH_E_CUDA;
  AttnMaps maps;
  const int64_t kv_rows = (int64_t)batch * Hkv * (ctx_len + block);
  if (!q_map(&maps.q, q, H, p.rows_total, p.G) || !kv_map(&maps.k, k, kv_rows) ||
      !kv_map(&maps.v, v, kv_rows))
    return DFLASH_E_CUDA;
  dim3 grid(q_tiles, Hkv, batch * splits);
  if (launch_k(true, attn_tc_kernel, dim3(grid), dim3(kAttnThreads), kAttnSmem, st, maps, p) !=
      cudaSuccess)
    return DFLASH_E_CUDA;
  if (splits > 1) {
    dim3 g2(p.rows_total, (H + 3) / 4);
    if (launch_k(true, combine_for(splits), dim3(g2), dim3(128), 0, st, p) != cudaSuccess)
      return DFLASH_E_CUDA;
  }
  return DFLASH_OK;
}

}  // namespace dflash

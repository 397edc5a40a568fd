// Fused GEMM epilogues.  A tile's accumulator comes straight from tensor
// memory when the tile took the whole K range (run_epilogue_direct); else
// its K splits are summed in split order (so the result does not depend on
// timing) -- from the partial tiles in the shared memory of a thread-block
// cluster (bf16 tensor-core GEMM, run_epilogue_cluster) or from fp32 slabs
// in global memory (fp32 SIMT GEMM, run_epilogue).  Then the operation that
// follows the projection in the pass is applied:
//   QKV    RoPE on Q and K at the row's position; Q -> q_out, K/V -> cache
//   SWIGLU act = SiLU(gate) * up            (tile pair: gate tile, up tile)
//   RESID  residual += projection (+ bf16 capture of an injected layer)
//   STORE  out = projection in the storage type
//   INJECT per draft layer: K = RoPE(.), V -> draft cache at the row position
//   SLAB   nothing (the fp32 slab is the result, e.g. lm_head logits)
#pragma once

#include "internal.cuh"

namespace dflash {

enum EpiKind { kEpiSlab = 0, kEpiQKV = 1, kEpiSwiGLU = 2, kEpiResid = 3, kEpiStore = 4,
               kEpiInject = 5, kEpiVocab = 6 };

struct EpiArgs {
  int kind;
  int M, N, splits;
  long long split_stride;  // elements between slabs (= M * N)
  const float* slab;
  // QKV / INJECT
  const int32_t* row_pos;
  const int32_t* row_slot;
  const int32_t* row_seq;
  const float* rcos;
  const float* rsin;
  void* q_out;
  void* kc;  // QKV: this layer's cache base; INJECT: draft cache base (all layers)
  void* vc;
  int H, Hkv, hd, max_ctx, max_batch;
  KvPages kp;  // cache slot -> page row
  size_t layer_elems;
  int layer0;
  // SWIGLU
  void* act;
  int F;
  // RESID
  float* resid;
  void* capture;
  int cap_slot, n_inject;
  float* trace;  // optional fp32 copy of the updated residual rows
  // STORE
  void* out;
  // VOCAB (lm_head): per token row and 128-feature tile, the best vr_k
  // logits (value descending, id ascending) and, with vr_lse, the tile's
  // (max, sum exp(x - max)); the logits themselves only for rows with
  // vr_vec[row] >= 0 when vr_logits is set
  int32_t* vr_id;          // [row][tile][vr_k]
  float* vr_v;             // [row][tile][vr_k]
  float* vr_lse;           // [row][tile][2] or NULL
  const int32_t* vr_vec;   // [row] row of vr_logits, < 0: none
  float* vr_logits;        // [vec row][N] or NULL
  int vr_k;                // 2..16
  int32_t* status;
};

template <typename T>
__device__ __forceinline__ float slab_sum(const EpiArgs& e, int t, int n) {
  const float* p = e.slab + (size_t)t * e.N + n;
  float v = 0.f;
  int s = 0;
  for (; s + 4 <= e.splits; s += 4) {
    const float a = p[(size_t)s * e.split_stride], b = p[(size_t)(s + 1) * e.split_stride];
    const float c = p[(size_t)(s + 2) * e.split_stride], d = p[(size_t)(s + 3) * e.split_stride];
    v += a;
    v += b;
    v += c;
    v += d;
  }
  for (; s < e.splits; ++s) v += p[(size_t)s * e.split_stride];
  return v;
}

// RoPE-rotated head (64 pairs of one 128-wide tile) for rows m0..m1.
template <typename T, bool kInject>
__device__ void epi_rotate_head(const EpiArgs& e, int n0, int m0, int m1, T* dst_base, int head,
                                bool is_q) {
  const int half = e.hd / 2;
  for (int idx = threadIdx.x; idx < (m1 - m0) * half; idx += blockDim.x) {
    const int t = m0 + idx / half, i = idx % half;
    int pos, seq, slot;
    if (kInject) {
      seq = e.row_seq[t];
      pos = e.row_pos[t];
      slot = pos;
      if (seq < 0) continue;
      if (seq >= e.max_batch || pos < 0 || pos >= e.max_ctx) {
        set_dev_status(e.status, kDevCheck);
        continue;
      }
    } else {
      pos = e.row_pos[t];
      if (pos < 0) continue;
      seq = e.row_seq[t];
      slot = e.row_slot[t];
    }
    long long row = (long long)t * e.H + head;
    if (!is_q) {
      row = kv_row(e.kp, e.Hkv, seq, head, slot);
      if (row < 0) {
        set_dev_status(e.status, kDevCapacity);
        continue;
      }
    }
    const float lo = slab_sum<T>(e, t, n0 + i), hi = slab_sum<T>(e, t, n0 + i + half);
    const float c = e.rcos[(size_t)pos * half + i], s = e.rsin[(size_t)pos * half + i];
    T* dst = dst_base + (size_t)row * e.hd;
    st_f(dst + i, lo * c - hi * s);
    st_f(dst + i + half, hi * c + lo * s);
  }
}

template <typename T, bool kInject>
__device__ void epi_copy_head(const EpiArgs& e, int n0, int m0, int m1, T* dst_base, int head) {
  for (int idx = threadIdx.x; idx < (m1 - m0) * e.hd; idx += blockDim.x) {
    const int t = m0 + idx / e.hd, c = idx % e.hd;
    int seq, slot;
    if (kInject) {
      seq = e.row_seq[t];
      slot = e.row_pos[t];
      if (seq < 0 || seq >= e.max_batch || slot < 0 || slot >= e.max_ctx) continue;
    } else {
      if (e.row_pos[t] < 0) continue;
      seq = e.row_seq[t];
      slot = e.row_slot[t];
    }
    const long long row = kv_row(e.kp, e.Hkv, seq, head, slot);
    if (row < 0) {
      set_dev_status(e.status, kDevCapacity);
      continue;
    }
    st_f(dst_base + (size_t)row * e.hd + c, slab_sum<T>(e, t, n0 + c));
  }
}

// Runs the epilogue of the 128-feature tile starting at n0, rows m0..m0+BN-1.
// All threads of the CTA take part (any block size).
template <typename T>
__device__ void run_epilogue(const EpiArgs& e, int n0, int m0, int BN) {
  const int m1 = min(e.M, m0 + BN);
  switch (e.kind) {
    case kEpiQKV: {  // a 128-wide tile holds 128 / head_dim whole heads
      for (int h0 = n0; h0 < min(e.N, n0 + 128); h0 += e.hd) {
        const int head = h0 / e.hd;
        if (head < e.H)
          epi_rotate_head<T, false>(e, h0, m0, m1, static_cast<T*>(e.q_out), head, true);
        else if (head < e.H + e.Hkv)
          epi_rotate_head<T, false>(e, h0, m0, m1, static_cast<T*>(e.kc), head - e.H, false);
        else
          epi_copy_head<T, false>(e, h0, m0, m1, static_cast<T*>(e.vc), head - e.H - e.Hkv);
      }
      break;
    }
    case kEpiInject: {
      const int kvd = e.Hkv * e.hd;
      for (int h0 = n0; h0 < min(e.N, n0 + 128); h0 += e.hd) {
        const int l = h0 / (2 * kvd), o = h0 % (2 * kvd);
        T* kbase = static_cast<T*>(e.kc) + (size_t)(e.layer0 + l) * e.layer_elems;
        T* vbase = static_cast<T*>(e.vc) + (size_t)(e.layer0 + l) * e.layer_elems;
        if (o < kvd)
          epi_rotate_head<T, true>(e, h0, m0, m1, kbase, o / e.hd, false);
        else
          epi_copy_head<T, true>(e, h0, m0, m1, vbase, (o - kvd) / e.hd);
      }
      break;
    }
    case kEpiSwiGLU: {
      for (int f = n0 + (int)threadIdx.x; f < min(e.F, n0 + 128); f += blockDim.x)
        for (int t = m0; t < m1; ++t) {
          const float g = slab_sum<T>(e, t, f), u = slab_sum<T>(e, t, e.F + f);
          st_f(static_cast<T*>(e.act) + (size_t)t * e.F + f, g / (1.f + __expf(-g)) * u);
        }
      break;
    }
    case kEpiResid: {
      T* cap = static_cast<T*>(e.capture);
      for (int n = n0 + (int)threadIdx.x; n < min(e.N, n0 + 128); n += blockDim.x)
        for (int t = m0; t < m1; ++t) {
          const float r = e.resid[(size_t)t * e.N + n] + slab_sum<T>(e, t, n);
          e.resid[(size_t)t * e.N + n] = r;
          if (cap) st_f(cap + ((size_t)t * e.n_inject + e.cap_slot) * e.N + n, r);
          if (e.trace) e.trace[(size_t)t * e.N + n] = r;
        }
      break;
    }
    case kEpiStore: {
      for (int n = n0 + (int)threadIdx.x; n < min(e.N, n0 + 128); n += blockDim.x)
        for (int t = m0; t < m1; ++t)
          st_f(static_cast<T*>(e.out) + (size_t)t * e.N + n, slab_sum<T>(e, t, n));
      break;
    }
    default:
      break;
  }
}

// ---------------------------------------------------------------------------
// Epilogue straight from tensor memory, for a tile without K splits.  The
// thread of TMEM lane f holds feature n0 + f for 16 token rows per
// tcgen05.ld.  A warp may only read the TMEM lane quarter warp % 4, so a
// CTA of 8 or 12 warps runs two or three groups of 4 warps over interleaved
// 16-row chunks (one group: all chunks); each group has its own named
// barrier and its own exchange buffer.  QKV / INJECT rotate the pairs (f, f + 64) of a head and
// SwiGLU multiplies gate row f by up row f + 64: those partners sit in warps
// w and w ^ 2, split each chunk's rows between them and trade through the
// two [8][128] fp32 halves of the group's buffer.  Row
// metadata (destination offset, RoPE table offset) is worked out once per
// row before the chunks.  All of it lives in the idle stage memory: one
// 8 KB buffer per group, then 256 x 8 + 256 x 4 bytes.
// ---------------------------------------------------------------------------
// (barrier 3 is the persistent kernel's all-epilogue barrier, so a third
// group takes 4)
__device__ __forceinline__ void group_bar_sync(int grp) {
  if (grp == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
  else if (grp == 1) asm volatile("bar.sync 2, 128;" ::: "memory");
  else asm volatile("bar.sync 4, 128;" ::: "memory");
}

// All threads that run the epilogue: the whole CTA (ep_threads == blockDim.x)
// or, in the persistent kernel, its ep_threads epilogue warps (named barrier 3).
__device__ __forceinline__ void epi_sync_all(int ep_threads) {
  if (ep_threads == (int)blockDim.x) __syncthreads();
  else asm volatile("bar.sync 3, %0;" ::"r"(ep_threads) : "memory");
}

// ep_tid / ep_threads: this thread's index among the threads that run the
// epilogue, and their count (a multiple of 128); a warp reads the TMEM lane
// quarter of its hardware warp index.
// Top-2 lists (value descending, id ascending; empty slots are (-inf,
// INT_MAX)): merge list B into list A.  The order is total, so the merged
// list is the top 2 of the union whatever the merge order.
__device__ __forceinline__ bool top_better(float x, int xi, float y, int yi) {
  return x > y || (x == y && xi < yi);
}
__device__ __forceinline__ void top2_merge(float& a1, int& j1, float& a2, int& j2, float b1, int k1,
                                           float b2, int k2) {
  if (top_better(b1, k1, a1, j1)) {
    if (top_better(a1, j1, b2, k2)) {
      a2 = a1;
      j2 = j1;
    } else {
      a2 = b2;
      j2 = k2;
    }
    a1 = b1;
    j1 = k1;
  } else if (top_better(b1, k1, a2, j2)) {
    a2 = b1;
    j2 = k1;
  }
}

// One halving round of a warp's top-2 reduce-scatter over R rows: lanes l
// and l ^ off trade lists; the lane with bit `off` set keeps rows R/2 .. R-1
// (the other rows 0 .. R/2-1) and merges the partner's lists for them.
template <int R>
__device__ __forceinline__ void top2_halve(const float (&a1)[R], const int (&j1)[R],
                                           const float (&a2)[R], const int (&j2)[R],
                                           float (&b1)[R / 2], int (&k1)[R / 2],
                                           float (&b2)[R / 2], int (&k2)[R / 2], int lane, int off) {
  const bool hi = (lane & off) != 0;
#pragma unroll
  for (int i = 0; i < R / 2; ++i) {
    const float s1 = hi ? a1[i] : a1[R / 2 + i], s2 = hi ? a2[i] : a2[R / 2 + i];
    const int t1 = hi ? j1[i] : j1[R / 2 + i], t2 = hi ? j2[i] : j2[R / 2 + i];
    const float r1 = __shfl_xor_sync(0xffffffffu, s1, off);
    const int q1 = __shfl_xor_sync(0xffffffffu, t1, off);
    const float r2 = __shfl_xor_sync(0xffffffffu, s2, off);
    const int q2 = __shfl_xor_sync(0xffffffffu, t2, off);
    b1[i] = hi ? a1[R / 2 + i] : a1[i];
    k1[i] = hi ? j1[R / 2 + i] : j1[i];
    b2[i] = hi ? a2[R / 2 + i] : a2[i];
    k2[i] = hi ? j2[R / 2 + i] : j2[i];
    top2_merge(b1[i], k1[i], b2[i], k2[i], r1, q1, r2, q2);
  }
}

template <typename T>
__device__ void run_epilogue_direct(const EpiArgs& e, uint32_t tmem, int n0, int m0, int BN,
                                    float* xbuf, int ep_tid, int ep_threads) {
  const int warp = ep_tid >> 5, lane = ep_tid & 31;
  const int quarter = ((int)threadIdx.x >> 5) & 3, grp = warp >> 2, ngrp = ep_threads >> 7;
  const int f = quarter * 32 + lane;
  const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
  const int c0 = grp * 16, cstep = ngrp * 16;
  float* const xb = xbuf + grp * 16 * 128;
  const int M = e.M;
  switch (e.kind) {
    case kEpiResid: {
      float* const resid = e.resid;
      float* const trace = e.trace;
      T* const cap = static_cast<T*>(e.capture);
      const int N = e.N, n_inj = e.n_inject, cap_slot = e.cap_slot, n = n0 + f;
      // the residual rows of the next chunk load while this one is stored
      auto load_r = [&](int c, float* r) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          r[i] = (m0 + c + i < M) ? resid[(size_t)(m0 + c + i) * N + n] : 0.f;
      };
      float r[16], rn[16];
      if (c0 < BN) load_r(c0, r);
      for (int c = c0; c < BN; c += cstep) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
        if (c + cstep < BN) load_r(c + cstep, rn);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = m0 + c + i;
          if (t >= M) continue;
          const float x = r[i] + v[i];
          resid[(size_t)t * N + n] = x;
          if (cap) st_f(cap + ((size_t)t * n_inj + cap_slot) * N + n, x);
          if (trace) trace[(size_t)t * N + n] = x;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = rn[i];
      }
      break;
    }
    case kEpiSwiGLU: {
      // lanes 0..63: gate of features n0 + f; lanes 64..127: up of n0 + f - 64.
      // Of each 16-row chunk the gate thread finishes rows 0..7 and the up
      // thread rows 8..15: each hands its partner (lane f ^ 64) the 8 values
      // the partner needs, through one of two alternating 8 x 128 halves of
      // the group's buffer (a half is rewritten two chunks later, after the
      // partner's read has passed the next chunk's barrier).
      T* const act = static_cast<T*>(e.act);
      const int F = e.F;
      const bool is_gate = f < 64;
      const int keep = is_gate ? 0 : 8;
      int parity = 0;
      for (int c = c0; c < BN; c += cstep, parity ^= 1) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
        float* const xh = xb + parity * 8 * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) xh[i * 128 + f] = is_gate ? v[8 + i] : v[i];
        group_bar_sync(grp);
        float other[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) other[i] = xh[i * 128 + (f ^ 64)];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = m0 + c + keep + i;
          if (t >= M) continue;
          const float g = is_gate ? v[i] : other[i];
          const float u = is_gate ? other[i] : v[8 + i];
          st_f(act + (size_t)t * F + n0 + (f & 63), g / (1.f + __expf(-g)) * u);
        }
      }
      break;
    }
    case kEpiStore: {
      T* const out = static_cast<T*>(e.out);
      const int N = e.N, n = n0 + f;
      for (int c = c0; c < BN; c += cstep) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (m0 + c + i < M) st_f(out + (size_t)(m0 + c + i) * N + n, v[i]);
      }
      break;
    }
    case kEpiQKV:
    case kEpiInject: {
      const bool inject = e.kind == kEpiInject;
      const int H = e.H, Hkv = e.Hkv, max_ctx = e.max_ctx, max_batch = e.max_batch;
      const int kvd = Hkv * 128;
      int head, layer = 0;
      bool is_q = false, is_v = false;
      if (!inject) {
        head = n0 / 128;
        if (head < H) is_q = true;
        else if (head < H + Hkv) head -= H;
        else { head -= H + Hkv; is_v = true; }
      } else {
        layer = n0 / (2 * kvd);
        const int o = n0 % (2 * kvd);
        is_v = o >= kvd;
        head = (is_v ? o - kvd : o) / 128;
      }
      T* base;
      if (is_q) base = static_cast<T*>(e.q_out);
      else base = static_cast<T*>(is_v ? e.vc : e.kc) +
                  (inject ? (size_t)(e.layer0 + layer) * e.layer_elems : 0);
      // per tile row: element offset of its 128-wide destination row (-1:
      // nothing to write) and of its cos/sin table row (-1: no rotation)
      long long* const s_dst = reinterpret_cast<long long*>(xbuf + ngrp * 16 * 128);
      int* const s_rope = reinterpret_cast<int*>(s_dst + 256);
      epi_sync_all(ep_threads);  // the previous tile's readers are done with s_dst / s_rope
      for (int u = ep_tid; u < BN; u += ep_threads) {
        const int t = m0 + u;
        long long dst = -1;
        int rope = -1;
        if (t < M) {
          const int pos = e.row_pos[t], seq = e.row_seq[t];
          if (pos >= 0 && seq >= 0) {
            if (inject && (seq >= max_batch || pos >= max_ctx)) {
              set_dev_status(e.status, kDevCheck);
            } else {
              const int slot = inject ? pos : e.row_slot[t];
              const long long row = is_q ? (long long)t * H + head : kv_row(e.kp, Hkv, seq, head, slot);
              if (row < 0) {
                set_dev_status(e.status, kDevCapacity);
              } else {
                dst = row * 128;
                if (pos < max_ctx) rope = pos * 64;  // the tables hold max_ctx positions
              }
            }
          }
        }
        s_dst[u] = dst;
        s_rope[u] = rope;
      }
      epi_sync_all(ep_threads);
      const float* const rcos = e.rcos;
      const float* const rsin = e.rsin;
      const int j = f & 63;
      const bool low = f < 64;
      if (is_v) {
        for (int c = c0; c < BN; c += cstep) {
          float v[16];
          tmem_ld16(taddr + (uint32_t)c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const long long off = s_dst[c + i];
            if (off >= 0) st_f(base + off + f, v[i]);
          }
        }
        break;
      }
      // Q and K: of each 16-row chunk the thread of feature j (low) rotates
      // rows 0..7 and the thread of feature j + 64 rows 8..15, writing both
      // features of the pair; each hands its partner (lane f ^ 64) the 8
      // values the partner needs through one of two alternating 8 x 128
      // halves of the group's buffer (a half is rewritten two chunks later,
      // after the partner's read has passed the next chunk's barrier).  The
      // cos/sin of a thread's 8 rows load one chunk ahead.
      const int keep = low ? 0 : 8;
      float cs[8], sn[8], cs_n[8], sn_n[8];
      auto load_rope = [&](int c, float* cn, float* snn) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ro = s_rope[c + keep + i];
          cn[i] = ro >= 0 ? rcos[ro + j] : 1.f;
          snn[i] = ro >= 0 ? rsin[ro + j] : 0.f;
        }
      };
      if (c0 < BN) load_rope(c0, cs_n, sn_n);
      int parity = 0;
      for (int c = c0; c < BN; c += cstep, parity ^= 1) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          cs[i] = cs_n[i];
          sn[i] = sn_n[i];
        }
        if (c + cstep < BN) load_rope(c + cstep, cs_n, sn_n);
        float* const xh = xb + parity * 8 * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) xh[i * 128 + f] = low ? v[8 + i] : v[i];
        group_bar_sync(grp);
        float other[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) other[i] = xh[i * 128 + (f ^ 64)];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const long long off = s_dst[c + keep + i];
          if (off < 0) continue;
          const float lo = low ? v[i] : other[i], hi = low ? other[i] : v[8 + i];
          st_f(base + off + j, lo * cs[i] - hi * sn[i]);
          st_f(base + off + j + 64, hi * cs[i] + lo * sn[i]);
        }
      }
      break;
    }
    case kEpiVocab: {
      // lm_head with K = 2 (argmax and margin; no log-sum-exp, no logits):
      // per token row, the top 2 of the tile's 128 ids (value descending, id
      // ascending; NaN and -inf never enter), which is what a scan of the ids
      // in order with strict comparisons keeps.  Per 16-row chunk a warp
      // reduce-scatters its 32 lanes' lists (five shuffle rounds, each
      // halving the rows a lane keeps, the last a full exchange): lane l ends
      // with row l / 2; then a warp of lane quarter 0 merges the four
      // quarters' lists through the group's buffer.
      const int nf = min(128, e.N - n0), nvt = (e.N + 127) / 128, vt = n0 / 128;
      const bool fvalid = f < nf;
      const int fid = n0 + f;
      float4* const sc = reinterpret_cast<float4*>(xb);  // [16 rows][4 quarters]
      for (int c = c0; c < BN; c += cstep) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
        float a1[16], a2[16];
        int j1[16], j2[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool ok = fvalid && v[i] > -INFINITY;
          a1[i] = ok ? v[i] : -INFINITY;
          j1[i] = ok ? fid : INT_MAX;
          a2[i] = -INFINITY;
          j2[i] = INT_MAX;
        }
        float b1[8], b2[8], d1[4], d2[4], g1[2], g2[2], h1[1], h2[1];
        int k1[8], k2[8], e1[4], e2[4], m1[2], m2[2], n1[1], n2[1];
        top2_halve<16>(a1, j1, a2, j2, b1, k1, b2, k2, lane, 16);
        top2_halve<8>(b1, k1, b2, k2, d1, e1, d2, e2, lane, 8);
        top2_halve<4>(d1, e1, d2, e2, g1, m1, g2, m2, lane, 4);
        top2_halve<2>(g1, m1, g2, m2, h1, n1, h2, n2, lane, 2);
        {
          const float r1 = __shfl_xor_sync(0xffffffffu, h1[0], 1);
          const int q1 = __shfl_xor_sync(0xffffffffu, n1[0], 1);
          const float r2 = __shfl_xor_sync(0xffffffffu, h2[0], 1);
          const int q2 = __shfl_xor_sync(0xffffffffu, n2[0], 1);
          top2_merge(h1[0], n1[0], h2[0], n2[0], r1, q1, r2, q2);
        }
        if ((lane & 1) == 0)
          sc[(lane >> 1) * 4 + quarter] =
              make_float4(h1[0], __int_as_float(n1[0]), h2[0], __int_as_float(n2[0]));
        group_bar_sync(grp);
        if (quarter == 0 && lane < 16) {
          const int t = m0 + c + lane;
          float4 q = sc[lane * 4];
          float x1 = q.x, x2 = q.z;
          int y1 = __float_as_int(q.y), y2 = __float_as_int(q.w);
#pragma unroll
          for (int w = 1; w < 4; ++w) {
            q = sc[lane * 4 + w];
            top2_merge(x1, y1, x2, y2, q.x, __float_as_int(q.y), q.z, __float_as_int(q.w));
          }
          if (t < M) {
            const size_t pb = (size_t)t * nvt + vt;
            e.vr_id[pb * 2] = y1;
            e.vr_id[pb * 2 + 1] = y2;
            e.vr_v[pb * 2] = x1;
            e.vr_v[pb * 2 + 1] = x2;
          }
        }
        group_bar_sync(grp);  // sc is rewritten by the next chunk
      }
      break;
    }
    default:
      break;
  }
}

// Partial sums of NI work items over the S splits of a cluster: item k is
// features c[k] .. c[k] + 3 of tile row u[k].  Every load (S per item) is
// issued before the first add; each item's sum starts from 0 and runs in
// split order.
template <int S, int NI>
__device__ __forceinline__ void cluster_sums(uint32_t local, const int (&u)[NI], const int (&c)[NI],
                                             const bool (&ok)[NI], float4 (&v)[NI]) {
  float4 x[NI][S];
#pragma unroll
  for (int k = 0; k < NI; ++k)
#pragma unroll
    for (int s = 0; s < S; ++s)
      if (ok[k]) x[k][s] = ld_peer_f32x4(map_peer(local + (uint32_t)((u[k] * 128 + c[k]) * 4), (uint32_t)s));
#pragma unroll
  for (int k = 0; k < NI; ++k) {
    v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < S; ++s)
      if (ok[k]) {
        v[k].x += x[k][s].x;
        v[k].y += x[k][s].y;
        v[k].z += x[k][s].z;
        v[k].w += x[k][s].w;
      }
  }
}

// Epilogue of a tile whose K splits form a thread-block cluster (residual,
// store, QKV and injection projections): each CTA has its fp32 partial tile in
// its own shared memory as part[token][feature]; after a cluster barrier, CTA
// `rank` takes every S-th work item of the tile (four consecutive features of
// one tile row), sums the partials of all splits in split order through
// distributed shared memory, and applies the epilogue operation.  A thread
// keeps U = 8 / S work items in flight (4 / S for the rotary projections,
// whose items carry a partner feature group and table rows): it issues their
// global loads (residual, rotary table) and every split's partial loads
// before the first add, so that the whole batch waits for one round trip of
// each kind.
// meta[u] = (position, sequence, slot) of tile row u.
template <typename T, int S>
__device__ void epilogue_cluster_s(const EpiArgs& e, int n0, int m0, int BN, uint32_t local,
                                   const int32_t* meta, int rank) {
  constexpr int U = S >= 8 ? 1 : 8 / S;
  constexpr int UQ = S >= 4 ? 1 : 4 / S;
  const int cn = min(BN, e.M - m0);
  const int first = rank * (int)blockDim.x + (int)threadIdx.x;
  const int step = S * (int)blockDim.x;
  switch (e.kind) {
    case kEpiResid:
    case kEpiStore: {
      const bool resid = e.kind == kEpiResid;
      T* cap = static_cast<T*>(e.capture);
      const int total = cn * 32;
      for (int i0 = first; i0 < total; i0 += U * step) {
        int u[U], c[U];
        bool ok[U];
        float4 r0[U], v[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int i = i0 + k * step;
          ok[k] = i < total;
          u[k] = ok[k] ? i >> 5 : 0;
          c[k] = ok[k] ? (i & 31) * 4 : 0;
          if (resid && ok[k])
            r0[k] = *reinterpret_cast<const float4*>(e.resid + (size_t)(m0 + u[k]) * e.N + n0 + c[k]);
        }
        cluster_sums<S, U>(local, u, c, ok, v);
#pragma unroll
        for (int k = 0; k < U; ++k) {
          if (!ok[k]) continue;
          const size_t t = (size_t)(m0 + u[k]);
          const int n = n0 + c[k];
          if (!resid) {
            st_f4(static_cast<T*>(e.out) + t * e.N + n, v[k]);
            continue;
          }
          const float4 r = make_float4(r0[k].x + v[k].x, r0[k].y + v[k].y, r0[k].z + v[k].z,
                                       r0[k].w + v[k].w);
          *reinterpret_cast<float4*>(e.resid + t * e.N + n) = r;
          if (cap) st_f4(cap + (t * e.n_inject + e.cap_slot) * e.N + n, r);
          if (e.trace) *reinterpret_cast<float4*>(e.trace + t * e.N + n) = r;
        }
      }
      break;
    }
    case kEpiQKV:
    case kEpiInject: {
      const bool inject = e.kind == kEpiInject;
      const int kvd = e.Hkv * 128;
      int head, layer = 0;
      bool is_q = false, is_v = false;
      if (!inject) {
        head = n0 / 128;
        if (head < e.H) is_q = true;
        else if (head < e.H + e.Hkv) head -= e.H;
        else { head -= e.H + e.Hkv; is_v = true; }
      } else {
        layer = n0 / (2 * kvd);
        const int o = n0 % (2 * kvd);
        is_v = o >= kvd;
        head = (is_v ? o - kvd : o) / 128;
      }
      T* base;
      if (is_q) base = static_cast<T*>(e.q_out);
      else base = static_cast<T*>(is_v ? e.vc : e.kc) +
                  (inject ? (size_t)(e.layer0 + layer) * e.layer_elems : 0);
      // V: 32 items of 4 features per row; Q, K: 16 items, each with the
      // rotary partner features 64 further on (items UQ .. 2 UQ - 1 below)
      const int per = is_v ? 32 : 16;
      const int total = cn * per;
      for (int i0 = first; i0 < total; i0 += UQ * step) {
        int u[2 * UQ], c[2 * UQ], pos[UQ];
        bool ok[2 * UQ];
        T* dst[UQ];
        float4 cs[UQ], sn[UQ], v[2 * UQ];
#pragma unroll
        for (int k = 0; k < UQ; ++k) {
          const int i = i0 + k * step;
          bool g = i < total;
          u[k] = g ? i / per : 0;
          c[k] = g ? (i % per) * 4 : 0;
          pos[k] = 0;
          dst[k] = nullptr;
          if (g) {
            const int t = m0 + u[k];
            const int ps = meta[u[k] * 3], seq = meta[u[k] * 3 + 1], slot = meta[u[k] * 3 + 2];
            pos[k] = ps;
            if (ps < 0 || seq < 0) {
              g = false;
            } else if (inject && (seq >= e.max_batch || ps >= e.max_ctx)) {
              set_dev_status(e.status, kDevCheck);
              g = false;
            } else {
              const long long row =
                  is_q ? (long long)t * e.H + head : kv_row(e.kp, e.Hkv, seq, head, slot);
              if (row < 0) {
                set_dev_status(e.status, kDevCapacity);
                g = false;
              } else {
                dst[k] = base + (size_t)row * 128;
              }
            }
          }
          ok[k] = g;
          // rotary partner: only for Q and K
          u[UQ + k] = u[k];
          c[UQ + k] = c[k] + 64;
          ok[UQ + k] = g && !is_v;
          if (g && !is_v) {
            cs[k] = *reinterpret_cast<const float4*>(e.rcos + (size_t)pos[k] * 64 + c[k]);
            sn[k] = *reinterpret_cast<const float4*>(e.rsin + (size_t)pos[k] * 64 + c[k]);
          }
        }
        cluster_sums<S, 2 * UQ>(local, u, c, ok, v);
#pragma unroll
        for (int k = 0; k < UQ; ++k) {
          if (!ok[k]) continue;
          if (is_v) {
            st_f4(dst[k] + c[k], v[k]);
          } else {
            const float4 lo = v[k], hi = v[UQ + k];
            st_f4(dst[k] + c[k],
                  make_float4(lo.x * cs[k].x - hi.x * sn[k].x, lo.y * cs[k].y - hi.y * sn[k].y,
                              lo.z * cs[k].z - hi.z * sn[k].z, lo.w * cs[k].w - hi.w * sn[k].w));
            st_f4(dst[k] + c[k] + 64,
                  make_float4(hi.x * cs[k].x + lo.x * sn[k].x, hi.y * cs[k].y + lo.y * sn[k].y,
                              hi.z * cs[k].z + lo.z * sn[k].z, hi.w * cs[k].w + lo.w * sn[k].w));
          }
        }
      }
      break;
    }
    default:
      break;
  }
}

template <typename T>
__device__ void run_epilogue_cluster(const EpiArgs& e, int n0, int m0, int BN, const float* part,
                                     const int32_t* meta) {
  const int rank = (int)cluster_ctarank();
  const uint32_t local = smem_u32(part);
  switch (e.splits) {
    case 1: epilogue_cluster_s<T, 1>(e, n0, m0, BN, local, meta, rank); break;
    case 2: epilogue_cluster_s<T, 2>(e, n0, m0, BN, local, meta, rank); break;
    case 3: epilogue_cluster_s<T, 3>(e, n0, m0, BN, local, meta, rank); break;
    case 4: epilogue_cluster_s<T, 4>(e, n0, m0, BN, local, meta, rank); break;
    case 5: epilogue_cluster_s<T, 5>(e, n0, m0, BN, local, meta, rank); break;
    case 6: epilogue_cluster_s<T, 6>(e, n0, m0, BN, local, meta, rank); break;
    case 7: epilogue_cluster_s<T, 7>(e, n0, m0, BN, local, meta, rank); break;
    default: epilogue_cluster_s<T, 8>(e, n0, m0, BN, local, meta, rank); break;
  }
}

}  // namespace dflash

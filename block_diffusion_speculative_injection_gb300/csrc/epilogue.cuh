// Fused GEMM epilogues.  The K splits of a tile are summed in split order
// (so the result does not depend on timing) -- from the partial tiles in
// the shared memory of a thread-block cluster (bf16 tensor-core GEMM,
// run_epilogue_cluster) or from fp32 slabs in global memory (fp32 SIMT
// GEMM, run_epilogue) -- and the operation that follows the projection in
// the pass is applied:
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
               kEpiInject = 5 };

struct EpiArgs {
  int kind;
  int M, N, splits;
  long long split_stride;  // elements between slabs (= M * N)
  const float* slab;
  int32_t* counters;
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
    const float lo = slab_sum<T>(e, t, n0 + i), hi = slab_sum<T>(e, t, n0 + i + half);
    const float c = e.rcos[(size_t)pos * half + i], s = e.rsin[(size_t)pos * half + i];
    T* dst = is_q ? dst_base + ((size_t)t * e.H + head) * e.hd
                  : dst_base + (((size_t)seq * e.Hkv + head) * e.max_ctx + slot) * e.hd;
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
    st_f(dst_base + (((size_t)seq * e.Hkv + head) * e.max_ctx + slot) * e.hd + c,
         slab_sum<T>(e, t, n0 + c));
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
// Cluster variant for the tensor-core GEMM (bf16, head_dim 128, N % 128 == 0).
// The thread-block cluster holds the K splits of one 128-feature output tile
// (SwiGLU: of a gate tile and the matching up tile, interleaved by rank:
// rank = h + 2*split with h = 0 gate, 1 up).  Each CTA has its fp32 partial
// tile in its own shared memory as part[token][feature]; after a cluster
// barrier, CTA `rank` takes every csize-th work item of the tile, sums the
// partials of all splits through distributed shared memory in split order,
// and applies the epilogue operation.  meta[u] = (position, sequence, slot)
// of tile row u (QKV / INJECT).
// ---------------------------------------------------------------------------
#ifndef DFLASH_EPI_UNROLL
#define DFLASH_EPI_UNROLL 1
#endif

template <typename T>
__device__ void run_epilogue_cluster(const EpiArgs& e, int n0, int m0, int BN, const float* part,
                                     const int32_t* meta) {
  // Every thread takes kU work items per round and issues all of their
  // loads (global operands, then partials) before using any.
  constexpr int kU = DFLASH_EPI_UNROLL;
  const int S = e.splits;
  const bool two = e.kind == kEpiSwiGLU;
  const int csize = two ? 2 * S : S;
  const int rank = (int)cluster_ctarank();
  const int cn = min(BN, e.M - m0);
  const uint32_t local = smem_u32(part);
  // sum over the splits of the partial (gate h = 0 / up h = 1 for SwiGLU) at
  // tile row u, column c, in split order through distributed shared memory;
  // a cluster of one CTA reads its own tile with ordinary shared loads
  const bool alone = S == 1 && !two;
  auto val = [&](int u, int c, int h) {
    if (alone) return part[u * 128 + c];
    const uint32_t addr = local + (uint32_t)((u * 128 + c) * 4);
    float v = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < S) v += ld_peer_f32(map_peer(addr, (uint32_t)(two ? h + 2 * s : s)));
    return v;
  };
  const int first = rank * (int)blockDim.x + (int)threadIdx.x;
  const int step = csize * (int)blockDim.x;
  switch (e.kind) {
    case kEpiResid: {
      T* cap = static_cast<T*>(e.capture);
      const int total = cn * 128;
      for (int i0 = first; i0 < total; i0 += kU * step) {
        float r[kU], v[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          r[k] = i < total ? e.resid[(size_t)(m0 + (i >> 7)) * e.N + n0 + (i & 127)] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          v[k] = i < total ? val(i >> 7, i & 127, 0) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          if (i >= total) continue;
          const int t = m0 + (i >> 7), n = n0 + (i & 127);
          const float x = r[k] + v[k];
          e.resid[(size_t)t * e.N + n] = x;
          if (cap) st_f(cap + ((size_t)t * e.n_inject + e.cap_slot) * e.N + n, x);
          if (e.trace) e.trace[(size_t)t * e.N + n] = x;
        }
      }
      break;
    }
    case kEpiStore: {
      const int total = cn * 128;
      for (int i0 = first; i0 < total; i0 += kU * step) {
        float v[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          v[k] = i < total ? val(i >> 7, i & 127, 0) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          if (i < total)
            st_f(static_cast<T*>(e.out) + (size_t)(m0 + (i >> 7)) * e.N + n0 + (i & 127), v[k]);
        }
      }
      break;
    }
    case kEpiSwiGLU: {
      const int total = cn * 128;
      for (int i0 = first; i0 < total; i0 += kU * step) {
        float g[kU], up[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          g[k] = i < total ? val(i >> 7, i & 127, 0) : 0.f;
          up[k] = i < total ? val(i >> 7, i & 127, 1) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          if (i < total)
            st_f(static_cast<T*>(e.act) + (size_t)(m0 + (i >> 7)) * e.F + n0 + (i & 127),
                 g[k] / (1.f + __expf(-g[k])) * up[k]);
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
      const int per = is_v ? 128 : 64;
      const int total = cn * per;
      for (int i0 = first; i0 < total; i0 += kU * step) {
        float lo[kU], hi[kU], cs[kU], sn[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          cs[k] = 1.f;
          sn[k] = 0.f;
          if (i < total && !is_v) {
            const int pos = meta[(i / per) * 3];
            if (pos >= 0 && pos < e.max_ctx) {  // the tables hold max_ctx positions
              cs[k] = e.rcos[(size_t)pos * 64 + i % per];
              sn[k] = e.rsin[(size_t)pos * 64 + i % per];
            }
          }
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          lo[k] = i < total ? val(i / per, i % per, 0) : 0.f;
          hi[k] = (i < total && !is_v) ? val(i / per, i % per + 64, 0) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int i = i0 + k * step;
          if (i >= total) continue;
          const int u = i / per, c = i % per, t = m0 + u;
          const int pos = meta[u * 3], seq = meta[u * 3 + 1], slot = meta[u * 3 + 2];
          if (pos < 0 || seq < 0) continue;
          if (inject && (seq >= e.max_batch || pos >= e.max_ctx)) {
            set_dev_status(e.status, kDevCheck);
            continue;
          }
          T* dst = is_q ? base + ((size_t)t * e.H + head) * 128
                        : base + (((size_t)seq * e.Hkv + head) * e.max_ctx + slot) * 128;
          if (is_v) {
            st_f(dst + c, lo[k]);
          } else {
            st_f(dst + c, lo[k] * cs[k] - hi[k] * sn[k]);
            st_f(dst + c + 64, hi[k] * cs[k] + lo[k] * sn[k]);
          }
        }
      }
      break;
    }
    default:
      break;
  }
}

}  // namespace dflash

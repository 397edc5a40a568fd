// C ABI of the DFlash step: context creation, weight registration and the
// orchestration of the target pass, the block-draft pass, acceptance, KV
// injection and the DDTree calls.  Every call validates its arguments on the
// host, then only enqueues kernels on the caller's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "epilogue.cuh"
#include "internal.cuh"

namespace dflash {

void set_error(dflash_ctx* ctx, const char* fmt, ...) {
  if (!ctx) return;
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  ctx->last_error = buf;
}

static dflash_status fail(dflash_ctx* ctx, dflash_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (ctx) ctx->last_error = buf;
  return s;
}

// refuses a call made while another device than the context's is current
#define DF_ON_DEVICE(ctx)                                                              \
  do {                                                                                 \
    if (!ctx_on_current_device(ctx))                                                   \
      return fail(ctx, DFLASH_E_STATE, "called with another device current than the " \
                                       "context's (device %d)", (ctx)->device);         \
  } while (0)

// draft pass keeps its own per-sequence metadata so that a draft issued
// between a verify and its accept never disturbs the verify's record
struct DraftMeta {
  int32_t *seq, *ctx, *blk;
};
static std::map<const dflash_ctx*, DraftMeta> g_draft_meta;

static int64_t target_layer_qkv_rows(const dflash_config& c) {
  return (int64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
}

static dflash_status validate_config(const dflash_config* c, std::string* why) {
  char b[256];
  auto bad = [&](const char* m) {
    *why = m;
    return DFLASH_E_INVALID_ARG;
  };
  if (c->d_model <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->ffn_dim <= 0 || c->vocab < 2)
    return bad("non-positive model dimension");
  if (c->n_heads % c->n_kv_heads) return bad("n_heads must be a multiple of n_kv_heads");
  if (c->head_dim % 2 || c->head_dim > 128) return bad("head_dim must be even and <= 128");
  if (c->n_target_layers <= 0 || c->n_draft_layers <= 0) return bad("layer counts must be > 0");
  if (c->n_inject < 1 || c->n_inject > 16) return bad("n_inject must be in 1..16");
  for (int i = 0; i < c->n_inject; ++i) {
    if (c->inject_layers[i] < 0 || c->inject_layers[i] >= c->n_target_layers)
      return bad("inject layer out of range");
    if (i && c->inject_layers[i] <= c->inject_layers[i - 1])
      return bad("inject layers must be ascending");
  }
  if (c->block_size < 1 || c->block_size > 16) return bad("block_size must be in 1..16");
  if (c->max_batch < 1 || c->max_batch > 1024) return bad("max_batch must be in 1..1024");
  if (c->max_ctx < c->block_size + 1) return bad("max_ctx too small");
  if (c->max_tree_nodes != 0 && (c->max_tree_nodes < 2 || c->max_tree_nodes > 128))
    return bad("max_tree_nodes must be 0 or 2..128");
  if (c->max_rows < c->max_batch * c->block_size ||
      c->max_rows < c->max_batch * c->max_tree_nodes)
    return bad("max_rows must cover max_batch * max(block_size, max_tree_nodes)");
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return bad("rms_eps and rope_theta must be > 0");
  if (c->kv_pages < 0) return bad("kv_pages must be >= 0");
  if (c->d_model > 8192) return bad("d_model must be <= 8192");
  if (c->dtype == DFLASH_F32) {
    if (c->head_dim % 32) return bad("fp32 path needs head_dim a multiple of 32");
  } else if (c->dtype == DFLASH_BF16) {
    if (c->head_dim != 128) return bad("bf16 path needs head_dim 128");
    if (64 % (c->n_heads / c->n_kv_heads)) return bad("bf16 path needs (n_heads/n_kv_heads) | 64");
    if (c->d_model % 128 || c->ffn_dim % 128) return bad("bf16 path needs d_model, ffn_dim % 128 == 0");
    if ((c->n_kv_heads * c->head_dim) % 128) return bad("bf16 path needs kv width % 128 == 0");
  } else {
    snprintf(b, sizeof(b), "unknown dtype %d", c->dtype);
    *why = b;
    return DFLASH_E_INVALID_ARG;
  }
  return DFLASH_OK;
}

static const char* kLayerNames[9] = {"attn_norm", "wq",   "wk",   "wv",    "wo",
                                     "ffn_norm",  "w_gate", "w_up", "w_down"};

static void layer_shape(const dflash_config& c, int which, int64_t* s, int* nd) {
  const int64_t d = c.d_model, q = (int64_t)c.n_heads * c.head_dim,
                kv = (int64_t)c.n_kv_heads * c.head_dim, F = c.ffn_dim;
  switch (which) {
    case 0: case 5: s[0] = d; *nd = 1; break;
    case 1: s[0] = q; s[1] = d; *nd = 2; break;
    case 2: case 3: s[0] = kv; s[1] = d; *nd = 2; break;
    case 4: s[0] = d; s[1] = q; *nd = 2; break;
    case 6: case 7: s[0] = F; s[1] = d; *nd = 2; break;
    default: s[0] = d; s[1] = F; *nd = 2; break;
  }
}

// expected shape of a named weight; false if the name is unknown
static bool expected_shape(const dflash_config& c, const std::string& name, int64_t* s, int* nd) {
  const int64_t d = c.d_model, V = c.vocab;
  if (name == "tok_emb" || name == "lm_head") { s[0] = V; s[1] = d; *nd = 2; return true; }
  if (name == "final_norm" || name == "draft.mask_emb" || name == "draft.final_norm") {
    s[0] = d; *nd = 1; return true;
  }
  if (name == "draft.fuse") { s[0] = d; s[1] = d * c.n_inject; *nd = 2; return true; }
  auto parse = [&](const char* prefix, int n_layers) -> bool {
    const size_t pl = strlen(prefix);
    if (name.compare(0, pl, prefix) != 0) return false;
    const char* rest = name.c_str() + pl;
    char* end = nullptr;
    const long l = strtol(rest, &end, 10);
    if (end == rest || *end != '.' || l < 0 || l >= n_layers) return false;
    for (int w = 0; w < 9; ++w)
      if (strcmp(end + 1, kLayerNames[w]) == 0) {
        layer_shape(c, w, s, nd);
        return true;
      }
    return false;
  };
  if (parse("draft.layers.", c.n_draft_layers)) return true;
  if (parse("layers.", c.n_target_layers)) return true;
  return false;
}

static dflash_status resolve_weights(dflash_ctx* ctx) {
  if (ctx->resolved) return DFLASH_OK;
  const dflash_config& c = ctx->cfg;
  auto get = [&](const std::string& n, const void** out) -> bool {
    auto it = ctx->weights.find(n);
    if (it == ctx->weights.end() || !it->second.ptr) {
      set_error(ctx, "weight '%s' not set", n.c_str());
      return false;
    }
    *out = it->second.ptr;
    return true;
  };
  if (!get("tok_emb", &ctx->tok_emb) || !get("lm_head", &ctx->lm_head) ||
      !get("final_norm", &ctx->final_norm) || !get("draft.fuse", &ctx->fuse) ||
      !get("draft.mask_emb", &ctx->mask_emb) || !get("draft.final_norm", &ctx->draft_final_norm))
    return DFLASH_E_STATE;
  auto layers = [&](const char* prefix, int n, std::vector<LayerW>& v) -> bool {
    v.assign(n, LayerW{});
    for (int l = 0; l < n; ++l) {
      const void** f[9] = {&v[l].attn_norm, &v[l].wq, &v[l].wk, &v[l].wv, &v[l].wo,
                           &v[l].ffn_norm, &v[l].w_gate, &v[l].w_up, &v[l].w_down};
      for (int w = 0; w < 9; ++w)
        if (!get(std::string(prefix) + std::to_string(l) + "." + kLayerNames[w], f[w])) return false;
    }
    return true;
  };
  if (!layers("layers.", c.n_target_layers, ctx->tl)) return DFLASH_E_STATE;
  if (!layers("draft.layers.", c.n_draft_layers, ctx->dl)) return DFLASH_E_STATE;
  ctx->resolved = true;
  return DFLASH_OK;
}


// ---------------------------------------------------------------------------
// one transformer layer (target or draft) over the rows of the current pass
// ---------------------------------------------------------------------------
static EpiArgs epi_base(dflash_ctx* ctx, int kind) {
  const dflash_config& c = ctx->cfg;
  EpiArgs e;
  memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.row_pos = ctx->row_pos;
  e.row_slot = ctx->row_slot;
  e.row_seq = ctx->row_seq;
  e.rcos = ctx->rope_cos;
  e.rsin = ctx->rope_sin;
  e.H = c.n_heads;
  e.Hkv = c.n_kv_heads;
  e.hd = c.head_dim;
  e.max_ctx = c.max_ctx;
  e.max_batch = c.max_batch;
  e.layer_elems = ctx->layer_cache_elems;
  e.kp = ctx_pages(ctx);
  e.F = c.ffn_dim;
  e.n_inject = c.n_inject;
  e.resid = ctx->resid;
  return e;
}

static dflash_status run_layer(dflash_ctx* ctx, const LayerW& w, int rows, void* kc, void* vc,
                               const AttnArgs& attn_base, const void* next_gain, void* capture,
                               int cap_slot, float* trace, cudaStream_t st, void* copy_q = nullptr,
                               void* copy_ao = nullptr) {
  const dflash_config& c = ctx->cfg;
  const int d = c.d_model, qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
  int sp = 1;
  EpiArgs eq = epi_base(ctx, kEpiQKV);
  eq.q_out = ctx->qb;
  eq.kc = kc;
  eq.vc = vc;
  GemmSegs qkv{{w.wq, w.wk, w.wv}, {qd, kvd, kvd}, 3};
  DF_TRY(gemm(ctx, ctx->xn, rows, d, qkv, eq, 16, &sp, st));
  AttnArgs a = attn_base;
  a.kc = kc;
  a.vc = vc;
  DF_TRY(attention(ctx, a, st));
  // debug copies of the attention inputs / outputs (dflash_debug_trace_draft_attn)
  const size_t qbytes = (size_t)rows * qd * ctx->esize;
  if (copy_q) DF_CUDA_TRY(ctx, cudaMemcpyAsync(copy_q, ctx->qb, qbytes, cudaMemcpyDeviceToDevice, st));
  if (copy_ao) DF_CUDA_TRY(ctx, cudaMemcpyAsync(copy_ao, ctx->ao, qbytes, cudaMemcpyDeviceToDevice, st));
  EpiArgs er = epi_base(ctx, kEpiResid);
  GemmSegs o{{w.wo}, {d}, 1};
  DF_TRY(gemm(ctx, ctx->ao, rows, qd, o, er, 16, &sp, st));
  DF_TRY(launch_norm(ctx, rows, nullptr, w.ffn_norm, ctx->xn, st));
  EpiArgs es = epi_base(ctx, kEpiSwiGLU);
  es.act = ctx->act;
  GemmSegs gu{{w.w_gate, w.w_up}, {c.ffn_dim, c.ffn_dim}, 2};
  DF_TRY(gemm(ctx, ctx->xn, rows, d, gu, es, 16, &sp, st));
  EpiArgs ed = epi_base(ctx, kEpiResid);
  ed.capture = capture;
  ed.cap_slot = cap_slot;
  ed.trace = trace;
  GemmSegs dn{{w.w_down}, {d}, 1};
  DF_TRY(gemm(ctx, ctx->act, rows, c.ffn_dim, dn, ed, 16, &sp, st));
  if (next_gain) DF_TRY(launch_norm(ctx, rows, nullptr, next_gain, ctx->xn, st));
  return DFLASH_OK;
}

// lm_head over the gathered rows lm_in[0..n) with reductions
static dflash_status run_lm_head(dflash_ctx* ctx, int n, int topk, int32_t* argmax, float* margin,
                                 int32_t* topk_ids, float* topk_logp, float* logits,
                                 cudaStream_t st) {
  const dflash_config& c = ctx->cfg;
  const int32_t* lm_arg = ctx->lm_rows + c.max_rows;
  GemmSegs lm_w{{ctx->lm_head}, {c.vocab}, 1};
  if (c.dtype != DFLASH_F32) {
    // the lm_head epilogue reduces every 128-feature tile of the vocabulary
    // to candidates, and the logits reach memory only for the rows the
    // caller asked for; a small second kernel merges the tiles
    const int K = topk > 2 ? topk : 2;
    const int n_tiles = (c.vocab + 127) / 128;
    // rows per launch: what the candidate buffers hold (every decode pass
    // fits in one; a long prefill that keeps every row's result takes several)
    const int chunk = (int)std::min<size_t>(ctx->vpart_cap / ((size_t)n_tiles * K), (size_t)n);
    if (n > 0 && chunk < 1) return fail(ctx, DFLASH_E_CAPACITY, "vocab partial buffer too small");
    for (int i0 = 0; i0 < n; i0 += chunk) {
      const int m = std::min(chunk, n - i0);
      EpiArgs e = epi_base(ctx, kEpiVocab);
      e.vr_id = ctx->vk_part;
      e.vr_v = ctx->vv_part;
      e.vr_lse = topk > 0 ? ctx->vv_part + ctx->vpart_cap : nullptr;
      e.vr_vec = lm_arg + i0 + c.max_rows;
      e.vr_logits = logits;
      e.vr_k = K;
      int sp = 1;
      const void* x = static_cast<const uint8_t*>(ctx->lm_in) + (size_t)i0 * c.d_model * ctx->esize;
      DF_TRY(gemm(ctx, x, m, c.d_model, lm_w, e, 1, &sp, st));
      DF_TRY(launch_vocab_merge(ctx, m, n_tiles, K, lm_arg + i0, topk, argmax, margin, topk_ids,
                                topk_logp, st));
    }
    return DFLASH_OK;
  }
  const size_t chunk_rows = ctx->ws_elems / (size_t)c.vocab;
  if (chunk_rows < 1) return fail(ctx, DFLASH_E_CAPACITY, "workspace smaller than one vocab row");
  for (int i0 = 0; i0 < n; i0 += (int)chunk_rows) {
    const int m = (int)std::min<size_t>(chunk_rows, (size_t)(n - i0));
    int sp = 1;
    const void* x = static_cast<const uint8_t*>(ctx->lm_in) + (size_t)i0 * c.d_model * ctx->esize;
    DF_TRY(gemm(ctx, x, m, c.d_model, lm_w, epi_base(ctx, kEpiSlab), 1, &sp, st));
    DF_TRY(launch_vocab_reduce(ctx, m, c.vocab, lm_arg + i0, topk, argmax, margin, topk_ids,
                               topk_logp, logits, st));
  }
  return DFLASH_OK;
}

// target pass shared by dflash_verify and dtree_verify
static dflash_status target_pass(dflash_ctx* ctx, int batch, int q, int mask,
                                 const uint64_t* anc, int anc_words, const int32_t* tokens,
                                 int last_only, int32_t* argmax, float* margin, float* logits,
                                 cudaStream_t st) {
  const dflash_config& c = ctx->cfg;
  const int rows = batch * q;
  DF_TRY(launch_embed(ctx, tokens, rows, 0, q, st));
  AttnArgs ab;
  memset(&ab, 0, sizeof(ab));
  ab.q = ctx->qb;
  ab.out = ctx->ao;
  ab.batch = batch;
  ab.q_stride = q;
  ab.mask = mask;
  ab.anc = anc;
  ab.anc_words = anc_words;
  ab.max_keys_ub = pages_key_bound(ctx);
  DF_TRY(launch_norm(ctx, rows, nullptr, ctx->tl[0].attn_norm, ctx->xn, st));
  int inj = 0;
  for (int l = 0; l < c.n_target_layers; ++l) {
    const size_t off = (size_t)l * ctx->layer_cache_elems * ctx->esize;
    void* kc = static_cast<uint8_t*>(ctx->kc) + off;
    void* vc = static_cast<uint8_t*>(ctx->vc) + off;
    const void* next_gain = l + 1 < c.n_target_layers ? ctx->tl[l + 1].attn_norm : nullptr;
    void* cap = nullptr;
    int slot = 0;
    if (inj < c.n_inject && c.inject_layers[inj] == l) {
      cap = ctx->capture;
      slot = inj++;
    }
    float* tr = ctx->trace ? ctx->trace + (size_t)l * c.max_rows * c.d_model : nullptr;
    DF_TRY(run_layer(ctx, ctx->tl[l], rows, kc, vc, ab, next_gain, cap, slot, tr, st));
  }
  const int n_lm = last_only ? batch : rows;
  DF_TRY(launch_norm(ctx, n_lm, ctx->lm_rows, ctx->final_norm, ctx->lm_in, st));
  DF_CUDA_TRY(ctx, cudaMemsetAsync(argmax, 0xFF, sizeof(int32_t) * rows, st));
  DF_TRY(run_lm_head(ctx, n_lm, 0, argmax, margin, nullptr, nullptr, logits, st));
  ctx->pending_rows = 0;
  return DFLASH_OK;
}

static bool aligned_ptr(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace dflash

using namespace dflash;

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

dflash_status dflash_create(const dflash_config* cfg, dflash_ctx** out) {
  if (!cfg || !out) return DFLASH_E_INVALID_ARG;
  *out = nullptr;
  std::string why;
  if (validate_config(cfg, &why) != DFLASH_OK) {
    fprintf(stderr, "dflash_create: %s\n", why.c_str());
    return DFLASH_E_INVALID_ARG;
  }
  dflash_ctx* ctx = new dflash_ctx();
  ctx->cfg = *cfg;
  ctx->active_block = cfg->block_size;
  const dflash_config& c = ctx->cfg;
  ctx->esize = c.dtype == DFLASH_BF16 ? 2 : 4;
  // programmatic dependent launch between kernels (DFLASH_NO_PDL=1 turns it off)
  ctx->pdl = getenv("DFLASH_NO_PDL") == nullptr;
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device) !=
          cudaSuccess) {
    delete ctx;
    return DFLASH_E_CUDA;
  }
  if (c.dtype == DFLASH_BF16) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, ctx->device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, ctx->device);
    if (major != 10 || minor != 3) {
      fprintf(stderr, "dflash_create: bf16 kernels are built for sm_103a, device is sm_%d%d\n",
              major, minor);
      delete ctx;
      return DFLASH_E_UNSUPPORTED;
    }
  }
  const size_t es = ctx->esize;
  const size_t R = c.max_rows, d = c.d_model, F = c.ffn_dim;
  const size_t qd = (size_t)c.n_heads * c.head_dim;
  if (pages_init(ctx) != DFLASH_OK) {
    delete ctx;
    return DFLASH_E_INVALID_ARG;
  }
  ctx->layer_cache_elems = (size_t)ctx->n_pages * c.n_kv_heads * kPageSlots * c.head_dim;
  // GEMM workspace: the widest non-lm_head GEMM over max_rows rows, or the
  // lm_head over the rows of one decode pass, whichever is larger
  size_t wsn = R * std::max<size_t>({(size_t)target_layer_qkv_rows(c), 2 * F, d,
                                      (size_t)std::min(c.n_draft_layers, 6) * 2 * c.n_kv_heads *
                                          c.head_dim});
  const size_t lm_rows = (size_t)c.max_batch * std::max(c.block_size, std::max(c.max_tree_nodes, 1));
  // fp32 storage writes the lm_head logits to the workspace (bf16 reduces
  // them in the GEMM epilogue)
  if (c.dtype == DFLASH_F32) wsn = std::max(wsn, lm_rows * (size_t)c.vocab);
  ctx->ws_elems = wsn;
  ctx->part_rows_cap = std::max<size_t>(R * c.n_heads, 1 << 18);
  // vocabulary candidates: up to 16 per row and chunk (4096 ids for fp32,
  // one 128-feature lm_head tile for bf16)
  const size_t n_chunks = c.dtype == DFLASH_F32 ? (c.vocab + 4095) / 4096 : (c.vocab + 127) / 128;
  ctx->vpart_cap = std::max<size_t>(lm_rows, 1) * n_chunks * 16;
  ctx->rope_len = c.max_ctx;

  bool ok = true;
  auto alloc = [&](void** p, size_t bytes) {
    if (!ok) return;
    if (cudaMalloc(p, bytes ? bytes : 16) != cudaSuccess) ok = false;
  };
  const size_t cache_layer_bytes = ctx->layer_cache_elems * ctx->esize;
  alloc((void**)&ctx->seq_len, sizeof(int32_t) * c.max_batch);
  alloc((void**)&ctx->gen_count, sizeof(int32_t) * c.max_batch);
  alloc((void**)&ctx->dev_status, sizeof(int32_t) * 4);
  alloc(&ctx->kc, cache_layer_bytes * c.n_target_layers);
  alloc(&ctx->vc, cache_layer_bytes * c.n_target_layers);
  alloc(&ctx->dkc, cache_layer_bytes * c.n_draft_layers);
  alloc(&ctx->dvc, cache_layer_bytes * c.n_draft_layers);
  alloc(&ctx->capture, R * c.n_inject * d * es);
  alloc((void**)&ctx->resid, R * d * sizeof(float));
  alloc(&ctx->xn, R * d * es);
  alloc(&ctx->qb, R * qd * es);
  alloc(&ctx->ao, R * qd * es);
  alloc(&ctx->act, R * F * es);
  alloc(&ctx->fb, R * d * es);
  alloc(&ctx->lm_in, R * d * es);
  alloc((void**)&ctx->ws, wsn * sizeof(float));
  alloc((void**)&ctx->sk_part, (size_t)ctx->sm_count * 128 * 256 * sizeof(float));
  alloc(&ctx->sk_sync, sk_sync_bytes(ctx->sm_count));
  alloc((void**)&ctx->part_o, ctx->part_rows_cap * c.head_dim * sizeof(float));
  alloc((void**)&ctx->part_ml, ctx->part_rows_cap * 2 * sizeof(float));
  alloc((void**)&ctx->vk_part, ctx->vpart_cap * sizeof(int32_t));
  alloc((void**)&ctx->vv_part, ctx->vpart_cap * 2 * sizeof(float));
  alloc((void**)&ctx->pass_seq, sizeof(int32_t) * c.max_batch * 3);
  alloc((void**)&ctx->row_pos, sizeof(int32_t) * R);
  alloc((void**)&ctx->row_slot, sizeof(int32_t) * R);
  alloc((void**)&ctx->row_seq, sizeof(int32_t) * R);
  alloc((void**)&ctx->lm_rows, sizeof(int32_t) * R * 3);
  alloc((void**)&ctx->inj_seq, sizeof(int32_t) * R);
  alloc((void**)&ctx->inj_pos, sizeof(int32_t) * R);
  alloc((void**)&ctx->path, sizeof(int32_t) * c.max_batch * 34);
  alloc((void**)&ctx->page_tab, sizeof(int32_t) * c.max_batch * ctx->pps);
  alloc((void**)&ctx->rope_cos, sizeof(float) * ctx->rope_len * (c.head_dim / 2));
  alloc((void**)&ctx->rope_sin, sizeof(float) * ctx->rope_len * (c.head_dim / 2));
  DraftMeta dm{nullptr, nullptr, nullptr};
  alloc((void**)&dm.seq, sizeof(int32_t) * c.max_batch * 3);
  if (!ok) {
    dflash_destroy(ctx);
    return DFLASH_E_OOM;
  }
  dm.ctx = dm.seq + c.max_batch;
  dm.blk = dm.seq + 2 * c.max_batch;
  g_draft_meta[ctx] = dm;
  ctx->pass_ctx = ctx->pass_seq + c.max_batch;
  ctx->pass_blk = ctx->pass_seq + 2 * c.max_batch;
  // caches start at zero so that stale slots always hold finite values
  bool mok = pages_fill_table(ctx) == DFLASH_OK &&
             cudaMemset(ctx->kc, 0, cache_layer_bytes * c.n_target_layers) == cudaSuccess &&
             cudaMemset(ctx->vc, 0, cache_layer_bytes * c.n_target_layers) == cudaSuccess &&
             cudaMemset(ctx->dkc, 0, cache_layer_bytes * c.n_draft_layers) == cudaSuccess &&
             cudaMemset(ctx->dvc, 0, cache_layer_bytes * c.n_draft_layers) == cudaSuccess &&
             cudaMemset(ctx->seq_len, 0, sizeof(int32_t) * c.max_batch) == cudaSuccess &&
             cudaMemset(ctx->gen_count, 0, sizeof(int32_t) * c.max_batch) == cudaSuccess &&
             cudaMemset(ctx->dev_status, 0, sizeof(int32_t) * 4) == cudaSuccess &&
             cudaMemset(ctx->sk_sync, 0, sk_sync_bytes(ctx->sm_count)) == cudaSuccess &&
             cudaMemset(ctx->inj_seq, 0xFF, sizeof(int32_t) * R) == cudaSuccess &&
             cudaMemset(ctx->capture, 0, R * c.n_inject * d * es) == cudaSuccess &&
             cudaMemset(ctx->resid, 0, R * d * sizeof(float)) == cudaSuccess;
  // RoPE tables in double precision on the host: angle = pos * theta^(-2i/hd)
  const int half = c.head_dim / 2;
  std::vector<float> cs((size_t)ctx->rope_len * half), sn((size_t)ctx->rope_len * half);
  for (int p = 0; p < ctx->rope_len; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)p * pow((double)c.rope_theta, -2.0 * i / c.head_dim);
      cs[(size_t)p * half + i] = (float)cos(ang);
      sn[(size_t)p * half + i] = (float)sin(ang);
    }
  mok = mok &&
        cudaMemcpy(ctx->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
        cudaMemcpy(ctx->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
        cudaDeviceSynchronize() == cudaSuccess;
  if (!mok) {
    dflash_destroy(ctx);
    return DFLASH_E_CUDA;
  }
  *out = ctx;
  return DFLASH_OK;
}

void dflash_destroy(dflash_ctx* ctx) {
  if (!ctx) return;
  void* ptrs[] = {ctx->seq_len, ctx->gen_count, ctx->dev_status, ctx->kc,      ctx->vc,      ctx->dkc,
                  ctx->dvc,     ctx->capture,    ctx->resid,   ctx->xn,      ctx->qb,
                  ctx->ao,      ctx->act,        ctx->fb,      ctx->lm_in,   ctx->ws,
                  ctx->part_o,  ctx->part_ml,    ctx->vk_part, ctx->vv_part, ctx->pass_seq,
                  ctx->row_pos, ctx->row_slot,   ctx->row_seq, ctx->lm_rows, ctx->inj_seq,
                  ctx->inj_pos, ctx->path,       ctx->rope_cos, ctx->rope_sin, ctx->page_tab,
                  ctx->sk_part, ctx->sk_sync};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  pages_destroy(ctx);
  for (cudaEvent_t e : ctx->prof_ev) cudaEventDestroy(e);
  auto it = g_draft_meta.find(ctx);
  if (it != g_draft_meta.end()) {
    if (it->second.seq) cudaFree(it->second.seq);
    g_draft_meta.erase(it);
  }
  delete ctx;
}

dflash_status dflash_set_weight(dflash_ctx* ctx, const char* name, const void* dev_ptr,
                                int32_t dtype, const int64_t* shape, int32_t ndim) {
  if (!ctx || !name || !dev_ptr || !shape) return fail(ctx, DFLASH_E_INVALID_ARG, "null argument");
  if (dtype != ctx->cfg.dtype)
    return fail(ctx, DFLASH_E_INVALID_ARG, "weight '%s': dtype %d != context dtype %d", name, dtype,
                ctx->cfg.dtype);
  int64_t s[2] = {0, 0};
  int nd = 0;
  if (!expected_shape(ctx->cfg, name, s, &nd))
    return fail(ctx, DFLASH_E_INVALID_ARG, "unknown weight name '%s'", name);
  if (nd != ndim || shape[0] != s[0] || (nd == 2 && shape[1] != s[1]))
    return fail(ctx, DFLASH_E_INVALID_ARG, "weight '%s': shape mismatch", name);
  if (!aligned_ptr(dev_ptr, 16))
    return fail(ctx, DFLASH_E_INVALID_ARG, "weight '%s': pointer not 16-byte aligned", name);
  WeightRef w;
  w.ptr = dev_ptr;
  w.ndim = nd;
  w.shape[0] = s[0];
  w.shape[1] = s[1];
  ctx->weights[name] = w;
  ctx->resolved = false;
  return DFLASH_OK;
}

dflash_status dflash_reset_seq(dflash_ctx* ctx, int32_t seq_id, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  if (seq_id < 0 || seq_id >= ctx->cfg.max_batch)
    return fail(ctx, DFLASH_E_INVALID_ARG, "seq_id %d out of range", seq_id);
  DF_CUDA_TRY(ctx, cudaMemsetAsync(ctx->seq_len + seq_id, 0, sizeof(int32_t),
                                   (cudaStream_t)stream));
  DF_CUDA_TRY(ctx, cudaMemsetAsync(ctx->gen_count + seq_id, 0, sizeof(int32_t),
                                   (cudaStream_t)stream));
  return DFLASH_OK;
}

dflash_status dflash_verify(dflash_ctx* ctx, int32_t batch, const int32_t* seq_ids_dev,
                            const int32_t* tokens_dev, int32_t q, const int32_t* q_lens_dev,
                            int32_t flags, int32_t* argmax_dev, float* margin_dev,
                            float* logits_dev, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  if (!seq_ids_dev || !tokens_dev || !argmax_dev)
    return fail(ctx, DFLASH_E_INVALID_ARG, "null pointer argument");
  if (batch < 1 || batch > ctx->cfg.max_batch || q < 1)
    return fail(ctx, DFLASH_E_INVALID_ARG, "batch %d / q %d out of range", batch, q);
  if ((int64_t)batch * q > ctx->cfg.max_rows)
    return fail(ctx, DFLASH_E_CAPACITY, "batch*q = %lld exceeds max_rows %d",
                (long long)batch * q, ctx->cfg.max_rows);
  if (q > ctx->cfg.max_ctx) return fail(ctx, DFLASH_E_CAPACITY, "q exceeds max_ctx");
  if ((flags & ~DFLASH_VERIFY_LAST_ONLY) != 0) return fail(ctx, DFLASH_E_INVALID_ARG, "bad flags");
  if (logits_dev && (flags & DFLASH_VERIFY_LAST_ONLY))
    return fail(ctx, DFLASH_E_INVALID_ARG, "logits copy needs all rows");
  DF_TRY(resolve_weights(ctx));
  cudaStream_t st = (cudaStream_t)stream;
  const int last_only = (flags & DFLASH_VERIFY_LAST_ONLY) ? 1 : 0;
  DF_TRY(launch_pass_setup_full(ctx, batch, seq_ids_dev, q, q_lens_dev, nullptr, nullptr,
                                kPassLinear, last_only, nullptr, nullptr, ctx->pass_seq,
                                ctx->pass_ctx, ctx->pass_blk, st));
  DF_TRY(target_pass(ctx, batch, q, kMaskCausal, nullptr, 0, tokens_dev, last_only, argmax_dev,
                     margin_dev, logits_dev, st));
  ctx->last_kind = kPassLinear;
  ctx->last_batch = batch;
  ctx->last_q = q;
  return DFLASH_OK;
}

dflash_status dflash_set_block_size(dflash_ctx* ctx, int32_t block) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  if (block < 1 || block > ctx->cfg.block_size)
    return fail(ctx, DFLASH_E_INVALID_ARG, "block %d outside 1..%d (the configured block size)",
                block, ctx->cfg.block_size);
  ctx->active_block = block;
  return DFLASH_OK;
}

dflash_status dflash_draft_block(dflash_ctx* ctx, int32_t batch, const int32_t* seq_ids_dev,
                                 const int32_t* anchor_dev, int32_t* block_dev, int32_t topk,
                                 int32_t* topk_ids_dev, float* topk_logp_dev, float* logits_dev,
                                 dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  const dflash_config& c = ctx->cfg;
  if (!seq_ids_dev || !anchor_dev || !block_dev)
    return fail(ctx, DFLASH_E_INVALID_ARG, "null pointer argument");
  if (batch < 1 || batch > c.max_batch) return fail(ctx, DFLASH_E_INVALID_ARG, "batch out of range");
  if (topk < 0 || topk > 16) return fail(ctx, DFLASH_E_INVALID_ARG, "topk must be in 0..16");
  if (topk > 0 && (!topk_ids_dev || !topk_logp_dev))
    return fail(ctx, DFLASH_E_INVALID_ARG, "topk outputs missing");
  if (topk > c.vocab) return fail(ctx, DFLASH_E_INVALID_ARG, "topk exceeds vocab");
  DF_TRY(resolve_weights(ctx));
  cudaStream_t st = (cudaStream_t)stream;
  const int B = ctx->active_block;
  const DraftMeta& dm = g_draft_meta[ctx];
  DF_TRY(launch_pass_setup_full(ctx, batch, seq_ids_dev, B, nullptr, nullptr, nullptr, kPassDraft,
                                0, anchor_dev, block_dev, dm.seq, dm.ctx, dm.blk, st));
  if (B == 1) return DFLASH_OK;  // nothing to draft: the block is the anchor alone
  const int rows = batch * B;
  DF_TRY(launch_embed(ctx, anchor_dev, rows, 1, B, st));
  AttnArgs ab;
  memset(&ab, 0, sizeof(ab));
  ab.q = ctx->qb;
  ab.out = ctx->ao;
  ab.batch = batch;
  ab.q_stride = B;
  ab.mask = kMaskNone;
  ab.max_keys_ub = pages_key_bound(ctx);
  // the attention kernels read per-sequence metadata from the pass arrays;
  // point them at the draft's copy for the duration of this pass
  int32_t* save[3] = {ctx->pass_seq, ctx->pass_ctx, ctx->pass_blk};
  ctx->pass_seq = dm.seq;
  ctx->pass_ctx = dm.ctx;
  ctx->pass_blk = dm.blk;
  dflash_status s = launch_norm(ctx, rows, nullptr, ctx->dl[0].attn_norm, ctx->xn, st);
  for (int l = 0; s == DFLASH_OK && l < c.n_draft_layers; ++l) {
    const size_t off = (size_t)l * ctx->layer_cache_elems * ctx->esize;
    void* kc = static_cast<uint8_t*>(ctx->dkc) + off;
    void* vc = static_cast<uint8_t*>(ctx->dvc) + off;
    const void* next_gain = l + 1 < c.n_draft_layers ? ctx->dl[l + 1].attn_norm : nullptr;
    float* tr = ctx->dtrace ? ctx->dtrace + (size_t)l * c.max_rows * c.d_model : nullptr;
    const size_t qoff = (size_t)l * c.max_rows * c.n_heads * c.head_dim * ctx->esize;
    void* cq = ctx->dtrace_q ? static_cast<uint8_t*>(ctx->dtrace_q) + qoff : nullptr;
    void* cao = ctx->dtrace_ao ? static_cast<uint8_t*>(ctx->dtrace_ao) + qoff : nullptr;
    s = run_layer(ctx, ctx->dl[l], rows, kc, vc, ab, next_gain, nullptr, 0, tr, st, cq, cao);
  }
  ctx->pass_seq = save[0];
  ctx->pass_ctx = save[1];
  ctx->pass_blk = save[2];
  if (s != DFLASH_OK) return s;
  const int n_lm = batch * (B - 1);
  DF_TRY(launch_norm(ctx, n_lm, ctx->lm_rows, ctx->draft_final_norm, ctx->lm_in, st));
  DF_TRY(run_lm_head(ctx, n_lm, topk, block_dev, nullptr, topk_ids_dev, topk_logp_dev, logits_dev,
                     st));
  return DFLASH_OK;
}

dflash_status dflash_accept_commit(dflash_ctx* ctx, int32_t batch, const int32_t* seq_ids_dev,
                                   const int32_t* block_dev, const int32_t* argmax_dev,
                                   const dtree_buffers* tree, int32_t mode,
                                   int32_t* accept_len_dev, int32_t* next_anchor_dev,
                                   int32_t* emitted_dev, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  if (!argmax_dev || !accept_len_dev || !next_anchor_dev || !emitted_dev)
    return fail(ctx, DFLASH_E_INVALID_ARG, "null pointer argument");
  if (mode != DFLASH_ACCEPT_GREEDY && mode != DFLASH_ACCEPT_ALL && mode != DFLASH_ACCEPT_GIVEN)
    return fail(ctx, DFLASH_E_INVALID_ARG, "unknown accept mode %d", mode);
  if (ctx->last_kind == kPassNone)
    return fail(ctx, DFLASH_E_STATE, "accept_commit without a preceding verify");
  if (batch != ctx->last_batch)
    return fail(ctx, DFLASH_E_INVALID_ARG, "batch differs from the last verify");
  cudaStream_t st = (cudaStream_t)stream;
  if (ctx->last_kind == kPassTree) {
    if (!tree) return fail(ctx, DFLASH_E_INVALID_ARG, "tree pass needs the tree buffers");
    if (mode != DFLASH_ACCEPT_GREEDY) return fail(ctx, DFLASH_E_INVALID_ARG, "tree pass is greedy only");
    if (tree->max_nodes != ctx->last_q) return fail(ctx, DFLASH_E_INVALID_ARG, "tree stride mismatch");
    DF_TRY(launch_tree_accept(ctx, batch, seq_ids_dev, tree, argmax_dev, accept_len_dev,
                              next_anchor_dev, emitted_dev, st));
  } else {
    if (tree) return fail(ctx, DFLASH_E_INVALID_ARG, "last pass was linear, tree given");
    if (mode != DFLASH_ACCEPT_ALL && !block_dev)
      return fail(ctx, DFLASH_E_INVALID_ARG, "block accept needs the block tokens");
    DF_TRY(launch_accept_linear(ctx, batch, seq_ids_dev, block_dev, argmax_dev, ctx->last_q, mode,
                                accept_len_dev, next_anchor_dev, emitted_dev, st));
  }
  ctx->pending_rows = batch * ctx->last_q;
  ctx->last_kind = kPassNone;
  return DFLASH_OK;
}

dflash_status dflash_advance_lengths(dflash_ctx* ctx, int32_t batch, const int32_t* seq_ids_dev,
                                    const int32_t* counts_dev, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  if (!seq_ids_dev || !counts_dev) return fail(ctx, DFLASH_E_INVALID_ARG, "null pointer argument");
  if (batch < 0 || batch > ctx->cfg.max_batch)
    return fail(ctx, DFLASH_E_INVALID_ARG, "batch %d outside 0..max_batch", batch);
  if (batch == 0) return DFLASH_OK;
  return launch_advance_lengths(ctx, batch, seq_ids_dev, counts_dev, (cudaStream_t)stream);
}

dflash_status dflash_injection_rows(const dflash_ctx* ctx, const void** hidden_dev,
                                    const int32_t** row_seq_dev, const int32_t** row_pos_dev,
                                    int32_t* n_rows) {
  if (!ctx || !hidden_dev || !row_seq_dev || !row_pos_dev || !n_rows) return DFLASH_E_INVALID_ARG;
  *hidden_dev = ctx->capture;
  *row_seq_dev = ctx->inj_seq;
  *row_pos_dev = ctx->inj_pos;
  *n_rows = ctx->pending_rows;
  return DFLASH_OK;
}

dflash_status dflash_inject_kv(dflash_ctx* ctx, int32_t n_rows, const int32_t* row_seq_dev,
                               const int32_t* row_pos_dev, const void* hidden_dev,
                               dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  const dflash_config& c = ctx->cfg;
  DF_TRY(resolve_weights(ctx));
  cudaStream_t st = (cudaStream_t)stream;
  const void* hidden = hidden_dev;
  const int32_t* rseq = row_seq_dev;
  const int32_t* rpos = row_pos_dev;
  int rows = n_rows;
  if (!hidden_dev) {
    rows = ctx->pending_rows;
    hidden = ctx->capture;
    rseq = ctx->inj_seq;
    rpos = ctx->inj_pos;
    if (rows == 0) return DFLASH_OK;
  } else {
    if (!row_seq_dev || !row_pos_dev) return fail(ctx, DFLASH_E_INVALID_ARG, "null row arrays");
    if (n_rows < 0 || n_rows > c.max_rows)
      return fail(ctx, DFLASH_E_CAPACITY, "n_rows %d exceeds max_rows", n_rows);
    if (!aligned_ptr(hidden_dev, 16)) return fail(ctx, DFLASH_E_INVALID_ARG, "hidden not aligned");
    if (n_rows == 0) return DFLASH_OK;
  }
  const int d = c.d_model, kvd = c.n_kv_heads * c.head_dim;
  int sp = 1;
  GemmSegs fz{{ctx->fuse}, {d}, 1};
  EpiArgs ef = epi_base(ctx, kEpiStore);
  ef.out = ctx->fb;
  DF_TRY(gemm(ctx, hidden, rows, c.n_inject * d, fz, ef, 16, &sp, st));
  for (int l0 = 0; l0 < c.n_draft_layers; l0 += 6) {
    const int nl = std::min(6, c.n_draft_layers - l0);
    GemmSegs kv;
    kv.n = 2 * nl;
    for (int i = 0; i < nl; ++i) {
      kv.w[2 * i] = ctx->dl[l0 + i].wk;
      kv.w[2 * i + 1] = ctx->dl[l0 + i].wv;
      kv.rows[2 * i] = kvd;
      kv.rows[2 * i + 1] = kvd;
    }
    EpiArgs ei = epi_base(ctx, kEpiInject);
    ei.row_seq = rseq;
    ei.row_pos = rpos;
    ei.kc = ctx->dkc;
    ei.vc = ctx->dvc;
    ei.layer0 = l0;
    DF_TRY(gemm(ctx, ctx->fb, rows, d, kv, ei, 16, &sp, st));
  }
  if (!hidden_dev) ctx->pending_rows = 0;
  return DFLASH_OK;
}

dflash_status dtree_build(dflash_ctx* ctx, int32_t batch, const int32_t* anchor_dev,
                          const int32_t* topk_ids_dev, const float* topk_logp_dev, int32_t topk,
                          int32_t budget, const dtree_buffers* tree, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  const dflash_config& c = ctx->cfg;
  if (!anchor_dev || !topk_ids_dev || !topk_logp_dev || !tree || !tree->tok || !tree->parent ||
      !tree->depth || !tree->anc || !tree->n_nodes)
    return fail(ctx, DFLASH_E_INVALID_ARG, "null pointer argument");
  if (batch < 1 || batch > c.max_batch) return fail(ctx, DFLASH_E_INVALID_ARG, "batch out of range");
  if (topk < 1 || topk > 16) return fail(ctx, DFLASH_E_INVALID_ARG, "topk must be in 1..16");
  if (budget < 0 || budget + 1 > tree->max_nodes)
    return fail(ctx, DFLASH_E_CAPACITY, "budget + 1 exceeds tree max_nodes");
  if (tree->max_nodes > c.max_tree_nodes || tree->max_nodes > 128)
    return fail(ctx, DFLASH_E_CAPACITY, "tree max_nodes exceeds max_tree_nodes");
  if (tree->anc_words != (tree->max_nodes + 63) / 64)
    return fail(ctx, DFLASH_E_INVALID_ARG, "anc_words must be ceil(max_nodes/64)");
  if (ctx->active_block < 2) return fail(ctx, DFLASH_E_INVALID_ARG, "tree needs block size >= 2");
  return launch_tree_build(ctx, batch, anchor_dev, topk_ids_dev, topk_logp_dev, topk,
                           ctx->active_block - 1, budget, tree, (cudaStream_t)stream);
}

dflash_status dtree_verify(dflash_ctx* ctx, int32_t batch, const int32_t* seq_ids_dev,
                           const dtree_buffers* tree, int32_t* node_argmax_dev, float* margin_dev,
                           float* logits_dev, dflash_stream_t stream) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  const dflash_config& c = ctx->cfg;
  if (!seq_ids_dev || !tree || !node_argmax_dev || !tree->tok || !tree->depth || !tree->anc ||
      !tree->n_nodes)
    return fail(ctx, DFLASH_E_INVALID_ARG, "null pointer argument");
  if (batch < 1 || batch > c.max_batch) return fail(ctx, DFLASH_E_INVALID_ARG, "batch out of range");
  if (tree->max_nodes < 1 || tree->max_nodes > c.max_tree_nodes)
    return fail(ctx, DFLASH_E_CAPACITY, "tree max_nodes exceeds max_tree_nodes");
  if (tree->anc_words != (tree->max_nodes + 63) / 64)
    return fail(ctx, DFLASH_E_INVALID_ARG, "anc_words must be ceil(max_nodes/64)");
  if ((int64_t)batch * tree->max_nodes > c.max_rows)
    return fail(ctx, DFLASH_E_CAPACITY, "batch*max_nodes exceeds max_rows");
  DF_TRY(resolve_weights(ctx));
  cudaStream_t st = (cudaStream_t)stream;
  const int q = tree->max_nodes;
  DF_TRY(launch_pass_setup_full(ctx, batch, seq_ids_dev, q, nullptr, tree->depth, tree->n_nodes,
                                kPassTree, 0, nullptr, nullptr, ctx->pass_seq, ctx->pass_ctx,
                                ctx->pass_blk, st));
  DF_TRY(target_pass(ctx, batch, q, kMaskTree, tree->anc, tree->anc_words, tree->tok, 0,
                     node_argmax_dev, margin_dev, logits_dev, st));
  ctx->last_kind = kPassTree;
  ctx->last_batch = batch;
  ctx->last_q = q;
  return DFLASH_OK;
}

dflash_status dflash_check(dflash_ctx* ctx) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  DF_ON_DEVICE(ctx);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(ctx, DFLASH_E_CUDA, "device: %s", cudaGetErrorString(e));
  int32_t s = 0;
  if (cudaMemcpy(&s, ctx->dev_status, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DFLASH_E_CUDA;
  cudaMemset(ctx->dev_status, 0, sizeof(int32_t));
  // a wait that gave up may have left stream-K arrival counts behind (the
  // launch ticket stays aligned: every CTA takes its ticket first)
  if (s == kDevTimeout)
    cudaMemset(static_cast<uint8_t*>(ctx->sk_sync) + 8, 0, sk_sync_bytes(ctx->sm_count) - 8);
  switch (s) {
    case kDevOk: return DFLASH_OK;
    case kDevCapacity:
      return fail(ctx, DFLASH_E_CAPACITY, "device: sequence exceeded max_ctx or its mapped KV pages");
    case kDevTimeout: return fail(ctx, DFLASH_E_TIMEOUT, "device: bounded wait expired");
    default: return fail(ctx, DFLASH_E_DEVICE_CHECK, "device: argument check failed");
  }
}

dflash_status dflash_block_attention(int32_t batch, int32_t n_heads, int32_t n_kv_heads,
                                     int32_t ctx_len, int32_t block, int32_t causal,
                                     const void* q_dev, const void* k_dev, const void* v_dev,
                                     void* out_dev, void* workspace_dev, int64_t workspace_bytes,
                                     dflash_stream_t stream) {
  if (workspace_bytes < 0) return DFLASH_E_INVALID_ARG;
  return block_attention(batch, n_heads, n_kv_heads, 128, ctx_len, block, causal ? 1 : 0, q_dev,
                         k_dev, v_dev, out_dev, workspace_dev, workspace_bytes,
                         (cudaStream_t)stream);
}

dflash_status dflash_plan_gemm(int32_t sm_count, int32_t M, int32_t N, int32_t K, int32_t kind,
                              int32_t max_splits, int32_t* plan_out) {
  return plan_gemm(sm_count, M, N, K, kind, max_splits, plan_out);
}

dflash_status dflash_plan_attention(int32_t sm_count, int32_t batch, int32_t n_heads,
                                   int32_t n_kv_heads, int32_t q_per_seq, int64_t max_keys,
                                   int32_t min_splits, int32_t* plan_out) {
  return plan_attention(sm_count, batch, n_heads, n_kv_heads, q_per_seq, max_keys, min_splits,
                        plan_out);
}

int64_t dflash_block_attention_workspace(int32_t batch, int32_t n_heads, int32_t n_kv_heads,
                                         int32_t ctx_len, int32_t block) {
  return block_attention_workspace(batch, n_heads, n_kv_heads, 128, ctx_len, block);
}

dflash_status dflash_debug_trace(dflash_ctx* ctx, float* dst_dev, int64_t bytes) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  const dflash_config& c = ctx->cfg;
  if (dst_dev && bytes < (int64_t)c.n_target_layers * c.max_rows * c.d_model * (int64_t)sizeof(float))
    return fail(ctx, DFLASH_E_CAPACITY, "trace buffer needs n_target_layers*max_rows*d_model floats");
  if (reinterpret_cast<uintptr_t>(dst_dev) % 16 != 0)
    return fail(ctx, DFLASH_E_INVALID_ARG, "trace buffer must be 16-byte aligned");
  ctx->trace = dst_dev;
  return DFLASH_OK;
}

dflash_status dflash_debug_trace_draft(dflash_ctx* ctx, float* dst_dev, int64_t bytes) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  const dflash_config& c = ctx->cfg;
  if (dst_dev && bytes < (int64_t)c.n_draft_layers * c.max_rows * c.d_model * (int64_t)sizeof(float))
    return fail(ctx, DFLASH_E_CAPACITY, "trace buffer needs n_draft_layers*max_rows*d_model floats");
  if (reinterpret_cast<uintptr_t>(dst_dev) % 16 != 0)
    return fail(ctx, DFLASH_E_INVALID_ARG, "trace buffer must be 16-byte aligned");
  ctx->dtrace = dst_dev;
  return DFLASH_OK;
}

dflash_status dflash_debug_trace_draft_attn(dflash_ctx* ctx, void* q_dev, void* attn_dev,
                                            int64_t bytes_each) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  const dflash_config& c = ctx->cfg;
  const int64_t need =
      (int64_t)c.n_draft_layers * c.max_rows * c.n_heads * c.head_dim * (int64_t)ctx->esize;
  if ((q_dev || attn_dev) && bytes_each < need)
    return fail(ctx, DFLASH_E_CAPACITY,
                "each trace buffer needs n_draft_layers*max_rows*n_heads*head_dim elements");
  ctx->dtrace_q = q_dev;
  ctx->dtrace_ao = attn_dev;
  return DFLASH_OK;
}

dflash_status dflash_profile(dflash_ctx* ctx, int32_t enable) {
  if (!ctx) return DFLASH_E_INVALID_ARG;
  if (enable) {
    if (ctx->prof_ev.empty()) {
      ctx->prof_ev.resize(1 << 16);
      for (auto& e : ctx->prof_ev) DF_CUDA_TRY(ctx, cudaEventCreate(&e));
    }
    ctx->prof_recs.clear();
    ctx->prof_next = 0;
  }
  ctx->prof_on = enable != 0;
  return DFLASH_OK;
}

dflash_status dflash_profile_read(dflash_ctx* ctx, int32_t kind, int64_t* launches, double* ms,
                                  double* bytes, double* flops) {
  if (!ctx || !launches || !ms || !bytes || !flops) return DFLASH_E_INVALID_ARG;
  *launches = 0;
  *ms = *bytes = *flops = 0.0;
  if (!ctx->prof_recs.empty())
    DF_CUDA_TRY(ctx, cudaEventSynchronize(ctx->prof_ev[ctx->prof_recs.back().ev + 1]));
  for (const ProfRec& r : ctx->prof_recs) {
    if (kind >= 0 && r.kind != kind) continue;
    float t = 0.f;
    DF_CUDA_TRY(ctx, cudaEventElapsedTime(&t, ctx->prof_ev[r.ev], ctx->prof_ev[r.ev + 1]));
    *launches += 1;
    *ms += t;
    *bytes += r.bytes;
    *flops += r.flops;
  }
  return DFLASH_OK;
}

int64_t dflash_profile_list(dflash_ctx* ctx, int32_t kind, double* ms, double* flops,
                            int64_t max_out) {
  if (!ctx || max_out < 0) return -1;
  if (!ctx->prof_recs.empty() &&
      cudaEventSynchronize(ctx->prof_ev[ctx->prof_recs.back().ev + 1]) != cudaSuccess)
    return -1;
  int64_t n = 0;
  for (const ProfRec& r : ctx->prof_recs) {
    if (kind >= 0 && r.kind != kind) continue;
    if (n < max_out) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, ctx->prof_ev[r.ev], ctx->prof_ev[r.ev + 1]) != cudaSuccess)
        return -1;
      if (ms) ms[n] = t;
      if (flops) flops[n] = r.flops;
    }
    ++n;
  }
  return n;
}

const char* dflash_last_error(const dflash_ctx* ctx) {
  return ctx ? ctx->last_error.c_str() : "null context";
}

const int32_t* dflash_seq_lengths(const dflash_ctx* ctx) { return ctx ? ctx->seq_len : nullptr; }

int64_t dflash_launch_count(const dflash_ctx* ctx) { return ctx ? ctx->launches : -1; }

dflash_status dflash_debug_view(const dflash_ctx* ctx, const char* name, int32_t layer,
                                const void** dev_ptr, int64_t* bytes) {
  if (!ctx || !name || !dev_ptr || !bytes) return DFLASH_E_INVALID_ARG;
  const dflash_config& c = ctx->cfg;
  const size_t lb = ctx->layer_cache_elems * ctx->esize;
  const std::string n(name);
  if (n == "k_cache" || n == "v_cache") {
    if (layer < 0 || layer >= c.n_target_layers) return DFLASH_E_INVALID_ARG;
    *dev_ptr = static_cast<const uint8_t*>(n[0] == 'k' ? ctx->kc : ctx->vc) + layer * lb;
    *bytes = (int64_t)lb;
    return DFLASH_OK;
  }
  if (n == "dk_cache" || n == "dv_cache") {
    if (layer < 0 || layer >= c.n_draft_layers) return DFLASH_E_INVALID_ARG;
    *dev_ptr = static_cast<const uint8_t*>(n[1] == 'k' ? ctx->dkc : ctx->dvc) + layer * lb;
    *bytes = (int64_t)lb;
    return DFLASH_OK;
  }
  if (n == "page_table") {
    *dev_ptr = ctx->page_tab;
    *bytes = (int64_t)c.max_batch * ctx->pps * sizeof(int32_t);
    return DFLASH_OK;
  }
  if (n == "gen_count") {
    *dev_ptr = ctx->gen_count;
    *bytes = (int64_t)c.max_batch * sizeof(int32_t);
    return DFLASH_OK;
  }
  if (n == "fused") {
    *dev_ptr = ctx->fb;
    *bytes = (int64_t)c.max_rows * c.d_model * ctx->esize;
    return DFLASH_OK;
  }
  if (n == "capture") {
    *dev_ptr = ctx->capture;
    *bytes = (int64_t)c.max_rows * c.n_inject * c.d_model * ctx->esize;
    return DFLASH_OK;
  }
  return DFLASH_E_INVALID_ARG;
}

}  // extern "C"

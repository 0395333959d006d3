// C ABI of the drafter library: handle creation (weight packing, pool, RoPE table, FP8
// lm_head), the context-K/V writer and the gamma-block propose.  Host-side checks run
// before any launch; every launch is stream-ordered on the caller's stream.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <vector>

#include "dflash_internal.cuh"
#include "attn_tc.cuh"
#include "gemm_tc.cuh"
#include "markov.cuh"
#include "persist_tc.cuh"

using namespace dflash;

namespace {

thread_local std::string g_create_error;

int fail(dflash_handle* h, int code, const std::string& msg) {
  if (h) h->err = msg; else g_create_error = msg;
  return code;
}

int cuda_fail(dflash_handle* h, cudaError_t e, const char* where) {
  return fail(h, DFLASH_ECUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

#define CK(call, where)                                  \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, where); \
  } while (0)

cudaEvent_t ev_get(dflash_handle* h) {
  if (!h->prof.spare.empty()) {
    cudaEvent_t e = h->prof.spare.back();
    h->prof.spare.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Timing events: from the spare pool when launching eagerly; owned by the graph entry
// (recorded as external event nodes) while capturing.
cudaEvent_t ev_mark(dflash_handle* h, cudaStream_t st) {
  cudaEvent_t e = nullptr;
  if (h->cap_entry) {
    cudaEventCreate(&e);
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  } else {
    e = ev_get(h);
    cudaEventRecord(e, st);
  }
  return e;
}

// Launch `call` as kernel kind `kind`: counted always, bracketed by events when profiling.
#define KL(kind, call, where)                                                   \
  do {                                                                          \
    cudaEvent_t e0_ = h->prof.on ? ev_mark(h, st) : nullptr;                    \
    CK((call), where);                                                          \
    if (h->cap_entry)                                                           \
      h->cap_entry->kind_counts[kind]++;                                        \
    else                                                                        \
      h->prof.launches[kind]++;                                                 \
    if (h->prof.on) {                                                           \
      cudaEvent_t e1_ = ev_mark(h, st);                                         \
      auto& list_ = h->cap_entry ? h->cap_entry->evs : h->prof.pending;         \
      list_.push_back({(int)(kind), {e0_, e1_}});                               \
    }                                                                           \
  } while (0)

void graph_collect(dflash_handle* h) {
  for (dflash::GraphEntry* g : h->graphs) {
    if (!g->pending) continue;
    for (auto& p : g->evs) {
      float ms = 0.f;
      if (cudaEventSynchronize(p.second.second) == cudaSuccess &&
          cudaEventElapsedTime(&ms, p.second.first, p.second.second) == cudaSuccess)
        h->prof.ms[p.first] += ms;
    }
    g->pending = false;
  }
}

void graph_free(dflash::GraphEntry* g) {
  if (g->exec) cudaGraphExecDestroy(g->exec);
  for (auto& p : g->evs) {
    cudaEventDestroy(p.second.first);
    cudaEventDestroy(p.second.second);
  }
  delete g;
}

void prof_drain(dflash_handle* h) {
  graph_collect(h);
  for (auto& p : h->prof.pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.second.second) == cudaSuccess &&
        cudaEventElapsedTime(&ms, p.second.first, p.second.second) == cudaSuccess)
      h->prof.ms[p.first] += ms;
    h->prof.spare.push_back(p.second.first);
    h->prof.spare.push_back(p.second.second);
  }
  h->prof.pending.clear();
}

void* dev_alloc(dflash_handle* h, size_t bytes) {
  void* p = nullptr;
  if (bytes == 0) bytes = 16;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  h->allocs.push_back(p);
  return p;
}

void free_all(dflash_handle* h) {
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
  prof_drain(h);
  for (dflash::GraphEntry* g : h->graphs) graph_free(g);
  h->graphs.clear();
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  h->cap_stream = nullptr;
  for (cudaEvent_t e : h->prof.spare) cudaEventDestroy(e);
  h->prof.spare.clear();
}

// Host float64 RoPE table: inv_freq_j (plain theta^(-2j/d), or the YaRN remap of
// from_weights.rs / dflash.rs load) divided by pi, and the post-rotation scale.
void rope_table(const dflash_cfg& c, std::vector<double>& inv_pi, float& mscale) {
  const int half = c.head_dim / 2;
  const double d = c.head_dim, theta = c.rope_theta;
  inv_pi.resize(half);
  mscale = 1.f;
  double low = 0, high = 0, denom = 1, factor = 1;
  if (c.rope_yarn) {
    factor = c.yarn_factor;
    auto corr = [&](double r) { return d * log(c.yarn_orig_max_pos / (r * 2.0 * M_PI)) / (2.0 * log(theta)); };
    low = fmax(floor(corr(c.yarn_beta_fast)), 0.0);
    high = fmin(ceil(corr(c.yarn_beta_slow)), d - 1.0);
    denom = fabs(high - low) < 1e-6 ? high - low + 0.001 : high - low;
    mscale = (float)(0.1 * log(factor) + 1.0);
  }
  for (int j = 0; j < half; ++j) {
    const double base = pow(theta, -2.0 * j / d);
    double inv = base;
    if (c.rope_yarn) {
      double ramp = (j - low) / denom;
      ramp = ramp < 0 ? 0 : (ramp > 1 ? 1 : ramp);
      const double ex = 1.0 - ramp;
      inv = (base / factor) * (1.0 - ex) + base * ex;
    }
    inv_pi[j] = inv / M_PI;
  }
}

constexpr int64_t kCounters = 16384;  // split-K tile counters; the last 64 count argmax tiles

int check_cfg(const dflash_cfg& c) {
  auto bad = [](const char* m) { return fail(nullptr, DFLASH_EINVAL, m); };
  if (c.hidden <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 || c.n_ff <= 0 ||
      c.vocab <= 0 || c.n_taps <= 0 || c.target_hidden <= 0)
    return bad("non-positive dimension in cfg");
  if (c.n_layers < 1 || c.n_layers > 64) return bad("n_layers must be in [1, 64]");
  if (c.n_q_heads % c.n_kv_heads) return bad("n_q_heads must be a multiple of n_kv_heads");
  if (c.gamma != kGamma) return fail(nullptr, DFLASH_EUNSUPPORTED, "gamma must be 16");
  if (c.page_size != kPage) return fail(nullptr, DFLASH_EUNSUPPORTED, "page_size must be 16");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(nullptr, DFLASH_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (c.dtype != DFLASH_F32 && c.dtype != DFLASH_BF16) return bad("dtype must be DFLASH_F32 or DFLASH_BF16");
  if (c.lm_head_dtype != c.dtype && c.lm_head_dtype != DFLASH_FP8E4M3_ROWSCALE)
    return bad("lm_head_dtype must equal dtype or be DFLASH_FP8E4M3_ROWSCALE");
  if (c.mask_token_id < 0 || c.mask_token_id >= c.vocab) return bad("mask_token_id outside the vocabulary");
  if (c.num_pages < 1 || c.max_batch < 1 || c.max_pages_per_seq < 1) return bad("pool/batch sizes must be >= 1");
  if (c.max_write_rows < 16) return bad("max_write_rows must be >= 16");
  if (!(c.rms_eps > 0.f) || !(c.rope_theta > 1.f)) return bad("rms_eps must be > 0 and rope_theta > 1");
  if (c.rope_yarn && (!(c.yarn_factor >= 1.f) || !(c.yarn_orig_max_pos > 0.f) || !(c.yarn_beta_fast > 0.f) ||
                      !(c.yarn_beta_slow > 0.f)))
    return bad("bad YaRN parameters");
  for (int l = 0; l < c.n_layers; ++l)
    if (c.layer_sliding[l] && c.sliding_window <= 0) return bad("sliding layer with sliding_window <= 0");
  if ((int64_t)c.max_pages_per_seq * kPage > (1ll << 30)) return bad("max_pages_per_seq too large");
  if (c.layer_weight_dtype != c.dtype && c.layer_weight_dtype != 0 && c.layer_weight_dtype != DFLASH_FP8E4M3_ROWSCALE)
    return bad("layer_weight_dtype must be 0 (same as dtype), dtype or DFLASH_FP8E4M3_ROWSCALE");
  if (c.layer_weight_dtype == DFLASH_FP8E4M3_ROWSCALE && c.dtype != DFLASH_BF16)
    return fail(nullptr, DFLASH_EUNSUPPORTED, "FP8 layer weights need the bf16 drafter");
  if (c.markov_rank < 0) return bad("markov_rank must be >= 0");
  if (c.markov_rank > 0 &&
      (c.markov_rank % 32 || c.markov_rank > kMarkovMaxRank || c.max_batch > kMarkovMaxBatch ||
       markov_smem_bytes(c.max_batch, c.markov_rank) > (size_t)kMarkovMaxSmem))
    return fail(nullptr, DFLASH_EUNSUPPORTED,
                "Markov head needs markov_rank % 32 == 0, rank <= 1024, max_batch <= 64 and "
                "max_batch * rank <= 40960");
  return DFLASH_OK;
}

// The bf16 gamma-block forward of one sequence as ONE persistent kernel (persist_tc.cu):
// memra-engine dflash.rs forward_round (every layer: QKV with q/k RMSNorm and RoPE, the
// block's K/V into its pool slots, non-causal GQA attention over context + block, o_proj,
// SiLU-gated MLP) + final norm + lm_head + the draft step's argmax over rows 1..15; the same
// arithmetic as propose_tc's per-projection kernels, without launch or grid-drain gaps
// between the projections.
int propose_persist(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens,
                    const int32_t* page_tables, int nb, int max_ctx_len, int32_t* draft_tokens, void* logits,
                    void* final_hidden, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  PersistParams p{};
  p.L = c.n_layers;
  p.M = nb * kGamma;
  p.H = c.hidden;
  p.F = c.n_ff;
  p.nh = c.n_q_heads;
  p.nkv = c.n_kv_heads;
  p.V = c.vocab;
  p.mpps = c.max_pages_per_seq;
  p.mask = c.mask_token_id;
  p.max_ctx = max_ctx_len;
  p.G = h->num_sms;
  p.eps = c.rms_eps;
  p.mscale = h->rope_mscale;
  const int units = nb * c.n_kv_heads;
  persist_attn_split(units, max_ctx_len, 0, p.G, &p.attn_cps[0], &p.attn_splits[0]);
  persist_attn_split(units, max_ctx_len, c.sliding_window, p.G, &p.attn_cps[1], &p.attn_splits[1]);
  p.bonus = bonus_tokens;
  p.ctx_lens = ctx_lens;
  p.page_tables = page_tables;
  p.rope_pos0 = h->cur_rope_pos;
  p.widths = h->cur_widths;
  p.embed = static_cast<const __nv_bfloat16*>(h->embed);
  p.norm = static_cast<const __nv_bfloat16*>(h->norm);
  p.inv_pi = h->rope_inv_pi;
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& d = h->layer[l];
    p.layers[l].q_norm = static_cast<const __nv_bfloat16*>(d.q_norm);
    p.layers[l].k_norm = static_cast<const __nv_bfloat16*>(d.k_norm);
    p.layers[l].ln_in = static_cast<const __nv_bfloat16*>(d.ln_in);
    p.layers[l].ln_post = static_cast<const __nv_bfloat16*>(d.ln_post);
    p.layers[l].window = c.layer_sliding[l] ? c.sliding_window : 0;
  }
  p.maps = static_cast<const CUtensorMap*>(h->p_maps);
  p.x = h->x;
  p.xb = static_cast<__nv_bfloat16*>(h->xb);
  p.xb2 = static_cast<__nv_bfloat16*>(h->xb2);
  p.ss_a = h->ss_a;
  p.ss_b = h->ss_b;
  p.q = static_cast<__nv_bfloat16*>(h->q);
  p.attn = static_cast<__nv_bfloat16*>(h->attn);
  p.act = static_cast<__nv_bfloat16*>(h->act);
  p.pool = static_cast<__nv_bfloat16*>(h->pool);
  p.g = h->geom;
  p.ws = h->ws;
  p.ws_half = h->p_ws_half;
  p.o_part = h->attn_opart;
  p.ml_part = h->attn_ml;
  p.drafts = draft_tokens;
  p.logits = static_cast<__nv_bfloat16*>(logits);
  p.final_hidden = static_cast<__nv_bfloat16*>(final_hidden);
  p.status = h->d_status;
  p.trace = h->p_trace;
  persist_bind_ctl(p, h->p_ctl);
  CK(cudaMemsetAsync(h->p_ctl, 0, h->p_ctl_words * sizeof(unsigned), st), "persistent control reset");
  KL(K_PERSIST, launch_persist(p, st), "persistent forward");
  return DFLASH_OK;
}

// The bf16 gamma-block forward on the tensor-core kernels (dflash.rs forward_round +
// final norm + lm_head + argmax).  Every projection is one tcgen05 GEMM launch with its
// epilogue fused; launches after the first may start early (programmatic dependent launch)
// and prefetch their weights while the previous kernel drains.
int propose_tc(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens, const int32_t* page_tables,
               int nb, int max_ctx_len, int32_t* draft_tokens, void* logits, void* final_hidden, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  const int M = nb * kGamma;
  if (h->persist_on && M <= kPersistMaxM)
    return propose_persist(h, bonus_tokens, ctx_lens, page_tables, nb, max_ctx_len, draft_tokens, logits,
                           final_hidden, st);
  const int H = c.hidden, F = c.n_ff, qd = c.n_q_heads * c.head_dim;
  const int qkvd = qd + 2 * c.n_kv_heads * c.head_dim;
  const int Mp = h->rows_max;
  const int tn = pick_tn(M);
  const bool fp8w = c.layer_weight_dtype == DFLASH_FP8E4M3_ROWSCALE;
  auto splits = [&](int N, int K) {
    const int tiles = ((N + 127) / 128) * ((M + tn - 1) / tn);
    return pick_splits(tiles, K / 64, h->num_sms, tn);
  };
  GemmParams base;
  base.ws = h->ws;
  base.counters = h->counters;
  base.status = h->d_status;
  base.Mp = Mp;
  base.eps = c.rms_eps;
  base.ss_n = H;

  KL(K_EMBED, launch_embed_tc(h, bonus_tokens, nb, st), "embed");
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& w = h->layer[l];
    {
      GemmParams p = base;
      p.ss_in = h->ss_b;
      p.ss_parts = H / 128;
      p.q = static_cast<__nv_bfloat16*>(h->q);
      p.q_norm = static_cast<const __nv_bfloat16*>(w.q_norm);
      p.k_norm = static_cast<const __nv_bfloat16*>(w.k_norm);
      p.inv_pi = h->rope_inv_pi;
      p.mscale = h->rope_mscale;
      p.nh = c.n_q_heads;
      p.nkv = c.n_kv_heads;
      p.ctx_lens = ctx_lens;
      p.page_tables = page_tables;
      p.rope_pos0 = h->cur_rope_pos;
      p.mpps = c.max_pages_per_seq;
      p.g = h->geom;
      p.layer = l;
      p.pool = static_cast<__nv_bfloat16*>(h->pool);
      p.row_scale = fp8w ? w.qkv_s : nullptr;
      KL(K_QKV, launch_gemm_tc(EPI_QKV, fp8w ? (const void*)w.qkv8 : w.w_qkv, qkvd, H, h->xb, H, M, p,
                               splits(qkvd, H), st, l > 0, fp8w),
         "qkv");
    }
    if (h->tc_attn) {
      AttnParams a;
      a.q = static_cast<const __nv_bfloat16*>(h->q);
      a.pool = static_cast<const __nv_bfloat16*>(h->pool);
      a.g = h->geom;
      a.layer = l;
      a.ctx_lens = ctx_lens;
      a.widths = h->cur_widths;
      a.page_tables = page_tables;
      a.mpps = c.max_pages_per_seq;
      a.nh = c.n_q_heads;
      a.nkv = c.n_kv_heads;
      a.window = c.layer_sliding[l] ? c.sliding_window : 0;
      a.o_part = h->attn_opart;
      a.ml_part = h->attn_ml;
      a.out = static_cast<__nv_bfloat16*>(h->attn);
      a.status = h->d_status;
      KL(K_ATTN, launch_attn_tc(a, nb, max_ctx_len, h->num_sms, st), "attention");
    } else {
      KL(K_ATTN, launch_attention(h, l, h->q, ctx_lens, page_tables, nb, max_ctx_len, h->attn, st), "attention");
    }
    {
      GemmParams p = base;
      p.x = h->x;
      p.xb = static_cast<__nv_bfloat16*>(h->xb);
      p.ss_out = h->ss_a;
      p.ln_next = static_cast<const __nv_bfloat16*>(w.ln_post);
      p.H = H;
      p.row_scale = fp8w ? w.o_s : nullptr;
      KL(K_OPROJ, launch_gemm_tc(EPI_RESID, fp8w ? (const void*)w.o8 : w.w_o, H, qd, h->attn, qd, M, p,
                                 splits(H, qd), st, true, fp8w),
         "o_proj");
    }
    {
      GemmParams p = base;
      p.ss_in = h->ss_a;
      p.ss_parts = H / 128;
      p.act = static_cast<__nv_bfloat16*>(h->act);
      p.F = F;
      p.row_scale = fp8w ? w.gu_s : nullptr;
      KL(K_GATEUP, launch_gemm_tc(EPI_GATEUP, fp8w ? (const void*)w.gu8 : w.w_gu, 2 * F, H, h->xb, H, M, p,
                                  splits(2 * F, H), st, true, fp8w),
         "gate/up");
    }
    {
      GemmParams p = base;
      p.x = h->x;
      p.xb = static_cast<__nv_bfloat16*>(h->xb);
      p.ss_out = h->ss_b;
      p.ln_next = l + 1 < c.n_layers ? static_cast<const __nv_bfloat16*>(h->layer[l + 1].ln_in) : nullptr;
      p.H = H;
      p.row_scale = fp8w ? w.down_s : nullptr;
      KL(K_DOWN, launch_gemm_tc(EPI_RESID, fp8w ? (const void*)w.down8 : w.w_down, H, F, h->act, F, M, p,
                                splits(H, F), st, true, fp8w),
         "down");
    }
  }
  KL(K_NORM, launch_rmsnorm_f32in(h, h->x, h->norm, h->xn, M, H, st), "final norm");
  if (final_hidden) KL(K_COPY, launch_copy_hidden(h, h->xn, M, final_hidden, st), "final hidden");
  {
    const bool fp8 = c.lm_head_dtype == DFLASH_FP8E4M3_ROWSCALE;
    GemmParams p = base;
    p.logits = static_cast<__nv_bfloat16*>(logits);
    p.amax_best = h->amax_best;
    p.amax_counter = h->counters + kCounters - 64;
    p.drafts = draft_tokens;
    p.row_scale = fp8 ? h->lm_scale : nullptr;
    p.logits32 = c.markov_rank > 0 ? h->logits32 : nullptr;  // the Markov head reads fp32 logits
    p.widths = h->cur_widths;
    KL(K_LMHEAD, launch_gemm_tc(EPI_LMHEAD, fp8 ? (const void*)h->lm_fp8 : h->lm_head, c.vocab, H, h->xn, H, M, p, 1,
                                st, false, fp8),
       "lm_head");
  }
  return DFLASH_OK;
}

// Context-K/V writer (dflash.rs ctx_features + ingest_ctx; from_weights.rs fused K/V weight +
// reshape_and_cache) over n rows in chunks of max_write_rows: f = hidden_norm(fc . taps), then
// every layer's K (k_norm, RoPE at positions[i], mscale) and V into the pool.  Row i goes to row
// first + i of the one sequence whose table is page_tables (row_seq == nullptr), or to row
// row_index[i] of sequence row_seq[i] (the batched writer: page_tables is [nseq, mpps]).
int write_ctx_rows(dflash_handle* h, const void* taps, const int32_t* positions, const int32_t* page_tables,
                   int nseq, const int32_t* row_seq, const int32_t* row_index, int first, int n, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  const int64_t H = c.hidden, tapd = (int64_t)c.n_taps * c.target_hidden;
  const int kvall = c.n_layers * 2 * c.n_kv_heads * c.head_dim;
  for (int32_t done = 0; done < n; done += c.max_write_rows) {
    const int m = std::min<int32_t>(c.max_write_rows, n - done);
    const void* tp = static_cast<const char*>(taps) + (int64_t)done * tapd * h->esz;
    const int32_t* rs = row_seq ? row_seq + done : nullptr;
    const int32_t* ri = row_index ? row_index + done : nullptr;
    if (h->tc) {
      // tensor-core writer: fc GEMM -> hidden_norm (fp32) -> [hi | lo] bf16 -> one GEMM for every
      // layer's K and V (each weight tile times both halves) with the k_norm / RoPE / scatter
      // epilogue
      auto splits = [&](int64_t N, int64_t K) {
        const int tn = pick_tn(m);
        return pick_splits((int)(((N + 127) / 128) * ((m + tn - 1) / tn)), (int)(K / 64), h->num_sms, tn);
      };
      GemmParams pf;
      pf.ws = h->ws;
      pf.counters = h->counters;
      pf.status = h->d_status;
      pf.out = h->wy;
      pf.ldo = (int)H;
      KL(K_W_FC, launch_gemm_tc(EPI_STORE, h->fc, (int)H, (int)tapd, tp, (int)tapd, m, pf, splits(H, tapd), st, false),
         "writer fc");
      KL(K_W_NORM, launch_rmsnorm_f32out(h, h->wy, h->hidden_norm, h->wf, m, (int)H, st), "writer hidden_norm");
      KL(K_W_NORM, launch_split_hi_lo(h->wf, m, (int)H, h->wf2, st), "writer split");
      GemmParams pk;
      pk.ws = h->ws;
      pk.counters = h->counters;
      pk.status = h->d_status;
      pk.eps = c.rms_eps;
      pk.k_norm = static_cast<const __nv_bfloat16*>(h->kn_all);
      pk.inv_pi = h->rope_inv_pi;
      pk.mscale = h->rope_mscale;
      pk.nkv = c.n_kv_heads;
      pk.positions = positions + done;
      pk.page_tables = page_tables;
      pk.first = first + done;
      pk.row_seq = rs;
      pk.row_index = ri;
      pk.nseq = nseq;
      pk.mpps = c.max_pages_per_seq;
      pk.g = h->geom;
      pk.pool = static_cast<__nv_bfloat16*>(h->pool);
      KL(K_W_KV, launch_gemm_tc(EPI_CTXKV, h->w_ctxkv, kvall, (int)H, h->wf2, (int)(2 * H), m, pk,
                                splits(kvall, H), st, false),
         "writer kv");
      continue;
    }
    // f = hidden_norm(fc . taps)  (dflash.rs ctx_features)
    KL(K_W_FC, launch_gemm(h, tp, (int)tapd, h->fc, m, (int)H, (int)tapd, h->wy, (int)H, false, st), "writer fc");
    KL(K_W_NORM, launch_rmsnorm_f32out(h, h->wy, h->hidden_norm, h->wf, m, (int)H, st), "writer hidden_norm");
    // every layer's K and V in one GEMM over the fused weight (fp32 features), then
    // k_norm / RoPE / scatter
    KL(K_W_KV, launch_gemm_xf32(h, h->wf, (int)H, h->w_ctxkv, m, kvall, (int)H, h->wy, kvall, st), "writer kv");
    KL(K_W_POST, launch_ctxkv_post(h, h->wy, m, positions + done, page_tables, first + done, st, rs, ri, nseq),
       "writer post");
  }
  return DFLASH_OK;
}

int propose_graph(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens, const int32_t* page_tables,
                  int nb, int max_ctx_len, int32_t* draft_tokens, void* logits, void* final_hidden, cudaStream_t st);

}  // namespace

// The single launch cuts each projection's (128-row tile, 64-wide k-block) units into G equal
// ranges, one per CTA.  With fewer units than CTAs some ranges are empty, and a tile's finisher
// would wait for partials from the empty ranges between its first and last owner.
static bool persist_every_cta_has_work(int64_t H, int64_t F, int64_t nh, int64_t nkv, int64_t V, int G) {
  const int64_t shapes[5][2] = {{(nh + 2 * nkv) * 128, H}, {H, nh * 128}, {2 * F, H}, {H, F}, {V, H}};
  for (const auto& sh : shapes)
    if (((sh[0] + 127) / 128) * (sh[1] / 64) < (int64_t)G) return false;
  return true;
}

extern "C" {

const char* dflash_last_error(const dflash_handle* h) { return h ? h->err.c_str() : g_create_error.c_str(); }

int dflash_create(const dflash_cfg* cfg, const dflash_weights* w, dflash_stream stream, dflash_handle** out) {
  g_create_error.clear();
  if (!cfg || !w || !out) return fail(nullptr, DFLASH_EINVAL, "null argument");
  *out = nullptr;
  int rc = check_cfg(*cfg);
  if (rc) return rc;
  const dflash_cfg& c = *cfg;
  if (!w->fc || !w->hidden_norm || !w->norm || !w->embed || !w->lm_head || !w->layers)
    return fail(nullptr, DFLASH_EINVAL, "null weight pointer");
  if (c.markov_rank > 0 && (!w->markov_w1 || !w->markov_w2))
    return fail(nullptr, DFLASH_EINVAL, "null Markov head weight pointer");
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    if (!lw.ln_in || !lw.wq || !lw.wk || !lw.wv || !lw.q_norm || !lw.k_norm || !lw.wo || !lw.ln_post ||
        !lw.w_gate || !lw.w_up || !lw.w_down)
      return fail(nullptr, DFLASH_EINVAL, "null layer weight pointer");
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  dflash_handle* h = new dflash_handle();
  h->cfg = c;
  h->esz = c.dtype == DFLASH_F32 ? 4 : 2;
  auto bail = [&](int code) {
    g_create_error = h->err;
    cudaStreamSynchronize(st);
    free_all(h);
    delete h;
    return code;
  };
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    fail(h, DFLASH_ECUDA, "no CUDA device");
    return bail(DFLASH_ECUDA);
  }
  h->tc = c.dtype == DFLASH_BF16;
  if (h->tc && (c.head_dim != 128 || c.hidden % 128 || c.n_ff % 64 || c.target_hidden % 8)) {
    fail(h, DFLASH_EUNSUPPORTED, "bf16 path needs head_dim 128, hidden % 128 == 0, n_ff % 64 == 0 and target_hidden % 8 == 0");
    return bail(DFLASH_EUNSUPPORTED);
  }
  const size_t es = h->esz;
  const int64_t H = c.hidden, hd = c.head_dim, nh = c.n_q_heads, nkv = c.n_kv_heads, F = c.n_ff, V = c.vocab;
  const int64_t qd = nh * hd, kvd = nkv * hd, qkvd = qd + 2 * kvd, L = c.n_layers;
  const int64_t tapd = (int64_t)c.n_taps * c.target_hidden;

#define ALLOC(dst, bytes)                                                   \
  do {                                                                      \
    (dst) = (decltype(dst))dev_alloc(h, (bytes));                           \
    if (!(dst)) {                                                           \
      fail(h, DFLASH_ENOMEM, "cudaMalloc failed: " #dst);                   \
      return bail(DFLASH_ENOMEM);                                           \
    }                                                                       \
  } while (0)
#define D2D(dst, src, bytes)                                                                 \
  do {                                                                                       \
    cudaError_t e_ = cudaMemcpyAsync((dst), (src), (bytes), cudaMemcpyDeviceToDevice, st);   \
    if (e_ != cudaSuccess) {                                                                 \
      cuda_fail(h, e_, "weight copy");                                                       \
      return bail(DFLASH_ECUDA);                                                             \
    }                                                                                        \
  } while (0)

  // ---- weights: copy + repack (layer tensors), borrow embed / lm_head
  ALLOC(h->fc, H * tapd * es);
  D2D(h->fc, w->fc, H * tapd * es);
  ALLOC(h->hidden_norm, H * es);
  D2D(h->hidden_norm, w->hidden_norm, H * es);
  ALLOC(h->norm, H * es);
  D2D(h->norm, w->norm, H * es);
  h->embed = w->embed;
  h->lm_head = w->lm_head;
  ALLOC(h->w_ctxkv, L * 2 * kvd * H * es);
  ALLOC(h->kn_all, L * hd * es);
  for (int l = 0; l < L; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    LayerW& d = h->layer[l];
    ALLOC(d.ln_in, H * es);
    D2D(d.ln_in, lw.ln_in, H * es);
    ALLOC(d.ln_post, H * es);
    D2D(d.ln_post, lw.ln_post, H * es);
    ALLOC(d.q_norm, hd * es);
    D2D(d.q_norm, lw.q_norm, hd * es);
    ALLOC(d.k_norm, hd * es);
    D2D(d.k_norm, lw.k_norm, hd * es);
    ALLOC(d.w_qkv, qkvd * H * es);
    D2D(d.w_qkv, lw.wq, qd * H * es);
    D2D((char*)d.w_qkv + qd * H * es, lw.wk, kvd * H * es);
    D2D((char*)d.w_qkv + (qd + kvd) * H * es, lw.wv, kvd * H * es);
    ALLOC(d.w_o, H * qd * es);
    D2D(d.w_o, lw.wo, H * qd * es);
    ALLOC(d.w_gu, 2 * F * H * es);
    if (h->tc) {
      // tensor-core path: gate/up interleaved in 64-row blocks so one 128-row GEMM tile
      // holds matching gate and up rows
      cudaError_t e2 = launch_fold_norm(lw.w_gate, lw.w_up, 1, (int)(2 * F), (int)H, nullptr, d.w_gu, st);
      if (e2 != cudaSuccess) {
        cuda_fail(h, e2, "pack gate/up");
        return bail(DFLASH_ECUDA);
      }
    } else {
      D2D(d.w_gu, lw.w_gate, F * H * es);
      D2D((char*)d.w_gu + F * H * es, lw.w_up, F * H * es);
    }
    ALLOC(d.w_down, H * F * es);
    D2D(d.w_down, lw.w_down, H * F * es);
    // fused context K/V weight [K_0; V_0; K_1; V_1; ...] (from_weights.rs fused K/V block)
    D2D((char*)h->w_ctxkv + (2 * l) * kvd * H * es, lw.wk, kvd * H * es);
    D2D((char*)h->w_ctxkv + (2 * l + 1) * kvd * H * es, lw.wv, kvd * H * es);
    D2D((char*)h->kn_all + l * hd * es, lw.k_norm, hd * es);
  }

  // ---- FP8 drafter lane (from_weights.rs Phase G): every layer's packed q|k|v, o, gate/up and
  // down weights quantised to e4m3 with a per-row fp32 scale (rows are output features, so the
  // packing does not change any row's scale)
  if (c.layer_weight_dtype == DFLASH_FP8E4M3_ROWSCALE) {
    for (int l = 0; l < L; ++l) {
      LayerW& d = h->layer[l];
      const int64_t rows[4] = {qkvd, H, 2 * F, H}, cols[4] = {H, qd, H, F};
      void* src[4] = {d.w_qkv, d.w_o, d.w_gu, d.w_down};
      uint8_t** codes[4] = {&d.qkv8, &d.o8, &d.gu8, &d.down8};
      float** scales[4] = {&d.qkv_s, &d.o_s, &d.gu_s, &d.down_s};
      for (int k = 0; k < 4; ++k) {
        uint8_t* cd = nullptr;
        float* sc = nullptr;
        ALLOC(cd, rows[k] * cols[k]);
        ALLOC(sc, rows[k] * sizeof(float));
        *codes[k] = cd;
        *scales[k] = sc;
        cudaError_t e = launch_quantize_fp8(src[k], (int)rows[k], (int)cols[k], c.dtype, cd, sc, st);
        if (e != cudaSuccess) {
          cuda_fail(h, e, "FP8 layer quantisation");
          return bail(DFLASH_ECUDA);
        }
      }
    }
  }

  // ---- DSpark Markov head: both tables copied; per-step control words
  if (c.markov_rank > 0) {
    const size_t mb = (size_t)V * c.markov_rank * es;
    ALLOC(h->mk_w1, mb);
    D2D(h->mk_w1, w->markov_w1, mb);
    ALLOC(h->mk_w2, mb);
    D2D(h->mk_w2, w->markov_w2, mb);
    h->mk_ctl_bytes = markov_ctl_bytes(c.max_batch);
    ALLOC(h->mk_ctl, h->mk_ctl_bytes);
    int per_sm = 0;
    if (markov_occupancy(c.dtype, c.max_batch, c.markov_rank, &per_sm) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      fail(h, DFLASH_EUNSUPPORTED, "the Markov-chain kernel cannot keep one CTA per SM for this batch and rank");
      return bail(DFLASH_EUNSUPPORTED);
    }
  }

  // ---- RoPE table
  std::vector<double> inv_pi;
  rope_table(c, inv_pi, h->rope_mscale);
  std::vector<float2> inv_pi2(inv_pi.size());
  for (size_t j = 0; j < inv_pi.size(); ++j) {
    inv_pi2[j].x = (float)inv_pi[j];
    inv_pi2[j].y = (float)(inv_pi[j] - (double)inv_pi2[j].x);
  }
  ALLOC(h->rope_inv_pi, inv_pi2.size() * sizeof(float2));
  {
    cudaError_t e = cudaMemcpyAsync(h->rope_inv_pi, inv_pi2.data(), inv_pi2.size() * sizeof(float2),
                                    cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) { cuda_fail(h, e, "rope table"); return bail(DFLASH_ECUDA); }
  }

  // ---- paged pool
  PoolGeom& g = h->geom;
  g.tile = kPage * hd;
  // a head's V tile right after its K tile: one 8 KB run per (layer, page, head)
  g.kv_stride = g.tile;
  g.head_stride = 2 * g.tile;
  g.page_stride = 2 * nkv * g.tile;
  g.layer_stride = (int64_t)c.num_pages * g.page_stride;
  g.num_pages = c.num_pages;
  g.nkv = (int)nkv;
  g.hd = (int)hd;
  h->pool_bytes = (size_t)(L * g.layer_stride) * es;
  ALLOC(h->pool, h->pool_bytes);
  if (cudaMemsetAsync(h->pool, 0, h->pool_bytes, st) != cudaSuccess) {
    fail(h, DFLASH_ECUDA, "pool memset");
    return bail(DFLASH_ECUDA);
  }

  // ---- scratch
  h->rows_max = c.max_batch * kGamma;
  const int64_t R = h->rows_max, Rw = c.max_write_rows;
  const int64_t ymax = std::max(std::max(qkvd, 2 * F), H);
  ALLOC(h->x, R * H * 4);
  ALLOC(h->xn, R * H * es);
  ALLOC(h->y, R * ymax * 4);
  ALLOC(h->q, R * qd * es);
  ALLOC(h->attn, R * qd * es);
  ALLOC(h->act, R * F * es);
  ALLOC(h->logits32, R * V * 4);
  ALLOC(h->wy, Rw * std::max(H, L * 2 * kvd) * 4);
  ALLOC(h->wf, Rw * H * 4);
  if (h->tc) {
    ALLOC(h->xb, R * H * es);
    ALLOC(h->ss_a, (H / 128) * R * 4);
    ALLOC(h->ss_b, (H / 128) * R * 4);
    ALLOC(h->amax_best, R * sizeof(unsigned long long));
    if (cudaMemsetAsync(h->amax_best, 0, R * sizeof(unsigned long long), st) != cudaSuccess) {
      fail(h, DFLASH_ECUDA, "argmax memset");
      return bail(DFLASH_ECUDA);
    }
    ALLOC(h->counters, kCounters * sizeof(unsigned));
    if (cudaMemsetAsync(h->counters, 0, kCounters * sizeof(unsigned), st) != cudaSuccess) {
      fail(h, DFLASH_ECUDA, "counter memset");
      return bail(DFLASH_ECUDA);
    }
    // split-K workspace: the largest need over every projection and batch size, and over
    // the writer's two GEMMs for every chunk size
    size_t need = 16;
    auto account = [&](int64_t N, int64_t K, int64_t m) {
      const int tn = pick_tn((int)m);
      const int64_t tiles = ((N + 127) / 128) * ((m + tn - 1) / tn);
      const int ns = pick_splits((int)tiles, (int)(K / 64), h->num_sms, tn);
      if (ns > 1) need = std::max(need, (size_t)(tiles * ns * 128 * tn));
      return tiles <= kCounters - 64;
    };
    bool fits = true;
    for (int64_t m = kGamma; m <= R; m += kGamma)
      fits = account(qkvd, H, m) && account(H, qd, m) && account(2 * F, H, m) && account(H, F, m) && fits;
    for (int64_t m = 1; m <= Rw; m = m < 256 ? m + 1 : m + 256)
      fits = account(H, tapd, m) && account(L * 2 * kvd, H, m) && fits;
    fits = account(H, tapd, Rw) && account(L * 2 * kvd, H, Rw) && fits;
    if (!fits || tapd % 64) {
      fail(h, DFLASH_EUNSUPPORTED, "GEMM tiling out of range (too many tiles or n_taps*target_hidden % 64 != 0)");
      return bail(DFLASH_EUNSUPPORTED);
    }
    ALLOC(h->wf2, Rw * 2 * H * es);
    h->tc_attn = (nh / nkv) == 8;
    // single-launch persistent forward for batch 1: needs the tensor-core attention, a bf16
    // lm_head, one resident CTA per SM, and at least one (tile, k-block) unit of every projection
    // per CTA (its split-K finisher counts every CTA between a tile's first and last owner)
    if (h->tc_attn && c.lm_head_dtype != DFLASH_FP8E4M3_ROWSCALE && c.layer_weight_dtype != DFLASH_FP8E4M3_ROWSCALE &&
        c.markov_rank == 0 && H <= persist_max_hidden() &&
        L <= kPersistMaxL && persist_every_cta_has_work(H, F, nh, nkv, V, h->num_sms)) {
      int per_sm = 0;
      if (persist_occupancy(&per_sm) == cudaSuccess && per_sm >= 1) h->persist_ok = true;
      cudaGetLastError();
    }
    if (h->persist_ok) {
      // two halves of split-K partials, used by alternate phases of the single launch
      h->p_ws_half = persist_ws_floats((int)H, (int)F, (int)nh, (int)nkv, (int)V, h->num_sms);
      need = std::max(need, 2 * h->p_ws_half);
      ALLOC(h->xb2, R * H * es);
      std::vector<CUtensorMap> maps(4 * L + 5);
      bool ok = true;
      for (int l = 0; l < L && ok; ++l) {
        const LayerW& d = h->layer[l];
        ok = make_tmap_bf16(&maps[4 * l + 0], d.w_qkv, qkvd, H, H, 128) &&
             make_tmap_bf16(&maps[4 * l + 1], d.w_o, H, qd, qd, 128) &&
             make_tmap_bf16(&maps[4 * l + 2], d.w_gu, 2 * F, H, H, 128) &&
             make_tmap_bf16(&maps[4 * l + 3], d.w_down, H, F, F, 128);
      }
      ok = ok && make_tmap_bf16(&maps[4 * L], h->lm_head, V, H, H, 128) &&
           make_tmap_bf16(&maps[4 * L + 1], h->xb, kGamma, H, H, kGamma) &&
           make_tmap_bf16(&maps[4 * L + 2], h->attn, kGamma, qd, qd, kGamma) &&
           make_tmap_bf16(&maps[4 * L + 3], h->act, kGamma, F, F, kGamma) &&
           make_tmap_bf16(&maps[4 * L + 4], h->xb2, kGamma, H, H, kGamma);
      if (!ok) {
        fail(h, DFLASH_ECUDA, "tensor maps of the persistent forward");
        return bail(DFLASH_ECUDA);
      }
      ALLOC(h->p_maps, maps.size() * sizeof(CUtensorMap));
      h->p_ctl_words = persist_ctl_words((int)L, (int)H, (int)F, (int)nh, (int)nkv, (int)V);
      ALLOC(h->p_ctl, h->p_ctl_words * sizeof(unsigned));
#if DFLASH_PHASE_TRACE
      h->p_trace_words = (size_t)h->num_sms * (2 + 6 * L) * kTraceSlots;
      ALLOC(h->p_trace, h->p_trace_words * sizeof(unsigned long long));
      cudaMemsetAsync(h->p_trace, 0, h->p_trace_words * sizeof(unsigned long long), st);
#endif
      cudaError_t e1 = cudaMemcpy(h->p_maps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
      if (e1 != cudaSuccess) {
        cuda_fail(h, e1, "persistent forward tables");
        return bail(DFLASH_ECUDA);
      }
      h->persist_on = true;
    }
    h->ws_floats = need;
    ALLOC(h->ws, need * 4);
    if (h->tc_attn) {
      const int64_t units = (int64_t)c.max_batch * nkv;
      const int64_t slots = attn_tc_partial_slots(h->num_sms, (int)units);
      ALLOC(h->attn_opart, slots * 128 * 128 * 4);
      ALLOC(h->attn_ml, slots * 128 * 2 * 4);
    }
  }
  if (cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
    fail(h, DFLASH_ECUDA, "capture stream");
    return bail(DFLASH_ECUDA);
  }
  ALLOC(h->d_status, sizeof(unsigned));
  if (cudaMemsetAsync(h->d_status, 0, sizeof(unsigned), st) != cudaSuccess) {
    fail(h, DFLASH_ECUDA, "status memset");
    return bail(DFLASH_ECUDA);
  }

  // ---- FP8 lm_head (from_weights.rs FP8 block; quantised once here)
  if (c.lm_head_dtype == DFLASH_FP8E4M3_ROWSCALE) {
    ALLOC(h->lm_fp8, V * H);
    ALLOC(h->lm_scale, V * 4);
    cudaError_t e = launch_quantize_fp8(w->lm_head, (int)V, (int)H, c.dtype, h->lm_fp8, h->lm_scale, st);
    if (e != cudaSuccess) { cuda_fail(h, e, "fp8 quantise"); return bail(DFLASH_ECUDA); }
  }
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) { cuda_fail(h, e, "create"); return bail(DFLASH_ECUDA); }
  *out = h;
  return DFLASH_OK;
#undef ALLOC
#undef D2D
}

int dflash_destroy(dflash_handle* h) {
  if (!h) return DFLASH_OK;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
  return DFLASH_OK;
}

int dflash_write_ctx_kv(dflash_handle* h, const void* taps, const int32_t* positions, const int32_t* page_table,
                        int32_t first, int32_t n, dflash_stream stream) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  h->err.clear();
  const dflash_cfg& c = h->cfg;
  if (n < 0 || first < 0) return fail(h, DFLASH_EINVAL, "first and n must be >= 0");
  if ((int64_t)first + n > (int64_t)kPage * c.max_pages_per_seq)
    return fail(h, DFLASH_ECAPACITY, "first + n beyond the page-table capacity (16 * max_pages_per_seq)");
  if (n == 0) return DFLASH_OK;
  if (!taps || !positions || !page_table) return fail(h, DFLASH_EINVAL, "null pointer");
  return write_ctx_rows(h, taps, positions, page_table, 1, nullptr, nullptr, first, n,
                        reinterpret_cast<cudaStream_t>(stream));
}

int dflash_write_ctx_kv_batch(dflash_handle* h, const void* taps, const int32_t* positions, const int32_t* row_seq,
                              const int32_t* row_index, const int32_t* page_tables, int32_t nseq, int32_t n,
                              dflash_stream stream) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  h->err.clear();
  if (n < 0 || nseq < 1) return fail(h, DFLASH_EINVAL, "n must be >= 0 and nseq >= 1");
  if (n == 0) return DFLASH_OK;
  if (!taps || !positions || !row_seq || !row_index || !page_tables) return fail(h, DFLASH_EINVAL, "null pointer");
  return write_ctx_rows(h, taps, positions, page_tables, nseq, row_seq, row_index, 0, n,
                        reinterpret_cast<cudaStream_t>(stream));
}

int dflash_propose(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens,
                   const int32_t* page_tables, int32_t nb, int32_t max_ctx_len, int32_t* draft_tokens,
                   void* logits, void* final_hidden, dflash_stream stream) {
  return dflash_propose_ex(h, bonus_tokens, ctx_lens, page_tables, nb, max_ctx_len, nullptr, nullptr, draft_tokens,
                           logits, final_hidden, stream);
}

int dflash_propose_ex(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens,
                      const int32_t* page_tables, int32_t nb, int32_t max_ctx_len, const int32_t* q_rope_pos,
                      const int32_t* widths, int32_t* draft_tokens, void* logits, void* final_hidden,
                      dflash_stream stream) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  h->err.clear();
  const dflash_cfg& c = h->cfg;
  if (nb < 1) return fail(h, DFLASH_EINVAL, "nb must be >= 1");
  if (nb > c.max_batch) return fail(h, DFLASH_ECAPACITY, "nb > max_batch");
  if (max_ctx_len < 0) return fail(h, DFLASH_EINVAL, "max_ctx_len must be >= 0");
  if ((int64_t)max_ctx_len + kGamma > (int64_t)kPage * c.max_pages_per_seq)
    return fail(h, DFLASH_ECAPACITY, "max_ctx_len + gamma beyond the page-table capacity");
  if (!bonus_tokens || !ctx_lens || !page_tables || !draft_tokens) return fail(h, DFLASH_EINVAL, "null pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  h->cur_rope_pos = q_rope_pos;
  h->cur_widths = widths;
  const int rc = propose_graph(h, bonus_tokens, ctx_lens, page_tables, nb, max_ctx_len, draft_tokens, logits,
                               final_hidden, st);
  h->cur_rope_pos = nullptr;
  h->cur_widths = nullptr;
  return rc;
}

}  // extern "C"

namespace {

// The fp32 gamma-block forward on the CUDA-core kernels, launched eagerly on st.
int propose_simple(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens, const int32_t* page_tables,
                   int nb, int max_ctx_len, int32_t* draft_tokens, void* logits, void* final_hidden, cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  const int M = nb * kGamma;
  const int H = c.hidden, F = c.n_ff, qd = c.n_q_heads * c.head_dim;
  const int qkvd = qd + 2 * c.n_kv_heads * c.head_dim;

  KL(K_EMBED, launch_embed(h, bonus_tokens, nb, h->x, st), "embed");
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& w = h->layer[l];
    KL(K_NORM, launch_rmsnorm_f32in(h, h->x, w.ln_in, h->xn, M, H, st), "ln_in");
    KL(K_QKV, launch_gemm(h, h->xn, H, w.w_qkv, M, qkvd, H, h->y, qkvd, false, st), "qkv");
    KL(K_QKV_POST, launch_qkv_post(h, l, h->y, ctx_lens, page_tables, nb, h->q, st), "qkv post");
    KL(K_ATTN, launch_attention(h, l, h->q, ctx_lens, page_tables, nb, max_ctx_len, h->attn, st), "attention");
    KL(K_OPROJ, launch_gemm(h, h->attn, qd, w.w_o, M, H, qd, h->x, H, true, st), "o_proj");
    KL(K_NORM, launch_rmsnorm_f32in(h, h->x, w.ln_post, h->xn, M, H, st), "ln_post");
    KL(K_GATEUP, launch_gemm(h, h->xn, H, w.w_gu, M, 2 * F, H, h->y, 2 * F, false, st), "gate/up");
    KL(K_SILU, launch_silu_mul(h, h->y, M, h->act, st), "silu_mul");
    KL(K_DOWN, launch_gemm(h, h->act, F, w.w_down, M, H, F, h->x, H, true, st), "down");
  }
  KL(K_NORM, launch_rmsnorm_f32in(h, h->x, h->norm, h->xn, M, H, st), "final norm");
  if (final_hidden) KL(K_COPY, launch_copy_hidden(h, h->xn, M, final_hidden, st), "final hidden");
  if (c.lm_head_dtype == DFLASH_FP8E4M3_ROWSCALE)
    KL(K_LMHEAD, launch_gemm_fp8w(h, h->xn, H, h->lm_fp8, h->lm_scale, M, c.vocab, H, h->logits32, c.vocab, st), "lm_head");
  else
    KL(K_LMHEAD, launch_gemm(h, h->xn, H, h->lm_head, M, c.vocab, H, h->logits32, c.vocab, false, st), "lm_head");
  KL(K_ARGMAX, launch_argmax(h, h->logits32, nb, draft_tokens, logits, st), "argmax");
  return DFLASH_OK;
}

// DSpark Markov head after the lm_head (dflash.rs draft step, semi-AR Markov chain): the
// drafts (and logit rows 1..15 of every band, when written) are replaced by the chain's.
int propose_markov(dflash_handle* h, const int32_t* bonus_tokens, int nb, int32_t* draft_tokens, void* logits,
                   cudaStream_t st) {
  const dflash_cfg& c = h->cfg;
  MarkovParams m{};
  m.z = h->logits32;
  m.w1 = h->mk_w1;
  m.w2 = h->mk_w2;
  m.V = c.vocab;
  m.R = c.markov_rank;
  m.nb = nb;
  m.bonus = bonus_tokens;
  m.drafts = draft_tokens;
  m.logits = logits;
  m.status = h->d_status;
  m.widths = h->cur_widths;
  markov_bind_ctl(m, h->mk_ctl, nb);
  CK(cudaMemsetAsync(h->mk_ctl, 0, h->mk_ctl_bytes, st), "Markov control reset");
  KL(K_MARKOV, launch_markov(c.dtype, m, h->num_sms, st), "Markov chain");
  return DFLASH_OK;
}

int propose_eager(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens, const int32_t* page_tables,
                  int nb, int max_ctx_len, int32_t* draft_tokens, void* logits, void* final_hidden, cudaStream_t st) {
  const int rc = h->tc ? propose_tc(h, bonus_tokens, ctx_lens, page_tables, nb, max_ctx_len, draft_tokens, logits,
                                    final_hidden, st)
                       : propose_simple(h, bonus_tokens, ctx_lens, page_tables, nb, max_ctx_len, draft_tokens, logits,
                                        final_hidden, st);
  if (rc != DFLASH_OK || h->cfg.markov_rank == 0) return rc;
  return propose_markov(h, bonus_tokens, nb, draft_tokens, logits, st);
}

// Replay the CUDA graph captured for these arguments (capturing it on first use on a private
// stream); the whole forward is then one graph launch on the caller's stream.
int propose_graph(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens, const int32_t* page_tables,
                  int nb, int max_ctx_len, int32_t* draft_tokens, void* logits, void* final_hidden, cudaStream_t st) {
  const void* args[8] = {bonus_tokens, ctx_lens, page_tables, draft_tokens, logits, final_hidden,
                         h->cur_rope_pos, h->cur_widths};
  GraphEntry* e = nullptr;
  for (GraphEntry* g : h->graphs)
    if (g->nb == nb && g->max_ctx == max_ctx_len && g->prof == h->prof.on && g->persist == h->persist_on &&
        memcmp(g->args, args, sizeof(args)) == 0) {
      e = g;
      break;
    }
  if (!e) {
    if (h->graphs.size() >= 8) {
      auto it = std::min_element(h->graphs.begin(), h->graphs.end(),
                                 [](GraphEntry* a, GraphEntry* b) { return a->stamp < b->stamp; });
      graph_collect(h);
      CK(cudaStreamSynchronize(st), "graph evict sync");
      graph_free(*it);
      h->graphs.erase(it);
    }
    e = new GraphEntry();
    e->nb = nb;
    e->max_ctx = max_ctx_len;
    memcpy(e->args, args, sizeof(args));
    e->prof = h->prof.on;
    e->persist = h->persist_on;
    cudaError_t err = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeRelaxed);
    if (err != cudaSuccess) {
      graph_free(e);
      return cuda_fail(h, err, "begin capture");
    }
    h->cap_entry = e;
    const int rc = propose_eager(h, bonus_tokens, ctx_lens, page_tables, nb, max_ctx_len, draft_tokens, logits,
                                 final_hidden, h->cap_stream);
    h->cap_entry = nullptr;
    cudaGraph_t graph = nullptr;
    err = cudaStreamEndCapture(h->cap_stream, &graph);
    if (rc != DFLASH_OK || err != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      graph_free(e);
      cudaGetLastError();
      return rc != DFLASH_OK ? rc : cuda_fail(h, err, "end capture");
    }
    err = cudaGraphInstantiate(&e->exec, graph, 0);
    cudaGraphDestroy(graph);
    if (err != cudaSuccess) {
      graph_free(e);
      return cuda_fail(h, err, "graph instantiate");
    }
    h->graphs.push_back(e);
  }
  e->stamp = ++h->graph_clock;
  if (h->prof.on) graph_collect(h);
  for (int k = 0; k < K_COUNT; ++k) h->prof.launches[k] += e->kind_counts[k];
  CK(cudaGraphLaunch(e->exec, st), "graph launch");
  if (!e->evs.empty()) e->pending = true;
  return DFLASH_OK;
}

}  // namespace

extern "C" {

int dflash_kv_layout(const dflash_handle* h, void** pool, size_t* bytes, int64_t strides[6]) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  if (pool) *pool = h->pool;
  if (bytes) *bytes = h->pool_bytes;
  if (strides) {
    strides[0] = h->geom.layer_stride;
    strides[1] = h->geom.page_stride;
    strides[2] = h->geom.kv_stride;
    strides[3] = h->geom.head_stride;
    strides[4] = h->geom.tile;
    strides[5] = (int64_t)h->esz;
  }
  return DFLASH_OK;
}

int dflash_profile(dflash_handle* h, int enable) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  prof_drain(h);
  for (int k = 0; k < K_COUNT; ++k) {
    h->prof.launches[k] = 0;
    h->prof.ms[k] = 0.0;
  }
  h->prof.on = enable != 0;
  return DFLASH_OK;
}

int dflash_profile_kinds(void) { return K_COUNT; }

int dflash_set_persistent(dflash_handle* h, int enable) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  if (enable && !h->persist_ok)
    return fail(h, DFLASH_EUNSUPPORTED, "no persistent forward for this configuration or device");
  h->persist_on = enable != 0;
  return DFLASH_OK;
}

int dflash_persistent(const dflash_handle* h) { return h && h->persist_on ? 1 : 0; }

int dflash_profile_read(dflash_handle* h, int kind, const char** name, double* total_ms, int64_t* launches) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  if (kind < 0 || kind >= K_COUNT) return fail(h, DFLASH_EINVAL, "kernel kind out of range");
  prof_drain(h);
  if (name) *name = kKindNames[kind];
  if (total_ms) *total_ms = h->prof.ms[kind];
  if (launches) *launches = h->prof.launches[kind];
  return DFLASH_OK;
}

int dflash_gemm_bf16(const void* W, int32_t N, int32_t K, const void* X, int32_t M, float* out, int32_t nsplit,
                     dflash_stream stream) {
  if (!W || !X || !out) return fail(nullptr, DFLASH_EINVAL, "null pointer");
  if (N < 1 || M < 1 || K < 64 || K % 64) return fail(nullptr, DFLASH_EINVAL, "need N, M >= 1 and K % 64 == 0");
  if (nsplit != 1) return fail(nullptr, DFLASH_EINVAL, "nsplit must be 1 (no workspace)");
  GemmParams p;
  p.out = out;
  p.ldo = N;
  cudaError_t e = launch_gemm_tc(EPI_STORE, W, N, K, X, K, M, p, 1, reinterpret_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return fail(nullptr, DFLASH_ECUDA, std::string("gemm: ") + cudaGetErrorString(e));
  return DFLASH_OK;
}

int dflash_attention_check(dflash_handle* h, int32_t layer, const int32_t* ctx_lens, const int32_t* page_tables,
                           int32_t nb, int32_t max_ctx_len, void* out_cuda_core, void* out_tensor_core,
                           dflash_stream stream) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  const dflash_cfg& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers || nb < 1 || nb > c.max_batch || max_ctx_len < 0 ||
      (int64_t)max_ctx_len + kGamma > (int64_t)kPage * c.max_pages_per_seq || !ctx_lens || !page_tables ||
      !out_cuda_core || !out_tensor_core)
    return fail(h, DFLASH_EINVAL, "bad argument");
  if (!h->tc_attn) return fail(h, DFLASH_EUNSUPPORTED, "no tensor-core attention for this configuration");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CK(launch_attention(h, layer, h->q, ctx_lens, page_tables, nb, max_ctx_len, out_cuda_core, st), "attention");
  AttnParams a;
  a.q = static_cast<const __nv_bfloat16*>(h->q);
  a.pool = static_cast<const __nv_bfloat16*>(h->pool);
  a.g = h->geom;
  a.layer = layer;
  a.ctx_lens = ctx_lens;
  a.page_tables = page_tables;
  a.mpps = c.max_pages_per_seq;
  a.nh = c.n_q_heads;
  a.nkv = c.n_kv_heads;
  a.window = c.layer_sliding[layer] ? c.sliding_window : 0;
  a.o_part = h->attn_opart;
  a.ml_part = h->attn_ml;
  a.out = static_cast<__nv_bfloat16*>(out_tensor_core);
  a.status = h->d_status;
  CK(launch_attn_tc(a, nb, max_ctx_len, h->num_sms, st), "attention tc");
  return DFLASH_OK;
}

int dflash_fp8_lm_head(const dflash_handle* h, const uint8_t** codes, const float** scales) {
  if (!h || !codes || !scales) return fail(nullptr, DFLASH_EINVAL, "null argument");
  if (!h->lm_fp8) return DFLASH_EINVAL;
  *codes = h->lm_fp8;
  *scales = h->lm_scale;
  return DFLASH_OK;
}

int dflash_fp8_layer(const dflash_handle* h, int32_t layer, int32_t proj, const uint8_t** codes,
                     const float** scales) {
  if (!h || !codes || !scales) return DFLASH_EINVAL;
  if (h->cfg.layer_weight_dtype != DFLASH_FP8E4M3_ROWSCALE || layer < 0 || layer >= h->cfg.n_layers || proj < 0 ||
      proj > 3)
    return DFLASH_EINVAL;
  const LayerW& d = h->layer[layer];
  const uint8_t* cs[4] = {d.qkv8, d.o8, d.gu8, d.down8};
  const float* ss[4] = {d.qkv_s, d.o_s, d.gu_s, d.down_s};
  *codes = cs[proj];
  *scales = ss[proj];
  return DFLASH_OK;
}

int dflash_device_status(dflash_handle* h, dflash_stream stream, uint32_t* flags) {
  if (!h) return fail(nullptr, DFLASH_EINVAL, "null handle");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned v = 0;
  CK(cudaMemcpyAsync(&v, h->d_status, sizeof(unsigned), cudaMemcpyDeviceToHost, st), "status read");
  CK(cudaMemsetAsync(h->d_status, 0, sizeof(unsigned), st), "status clear");
  CK(cudaStreamSynchronize(st), "status sync");
  if ((v & DFLASH_DEV_TIMEOUT) && h->counters) {
    // a kernel that gave up a wait may have left split-K and argmax tile counters part-counted:
    // re-arm them so the next call starts from zero
    CK(cudaMemsetAsync(h->counters, 0, kCounters * sizeof(unsigned), st), "counter reset");
    CK(cudaStreamSynchronize(st), "counter reset sync");
  }
#if DFLASH_PHASE_TRACE
  // phase-timeline builds: the last persistent launch's stamps to $DFLASH_TRACE_FILE
  // (int32 CTAs, int32 phases, int32 slots, then the uint64 stamps)
  if (h->p_trace) {
    const char* path = getenv("DFLASH_TRACE_FILE");
    if (path && *path) {
      std::vector<unsigned long long> tr(h->p_trace_words);
      CK(cudaMemcpy(tr.data(), h->p_trace, tr.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost),
         "trace read");
      if (FILE* f = fopen(path, "wb")) {
        const int32_t hdr[3] = {h->num_sms, 2 + 6 * h->cfg.n_layers, kTraceSlots};
        fwrite(hdr, sizeof(hdr), 1, f);
        fwrite(tr.data(), sizeof(unsigned long long), tr.size(), f);
        fclose(f);
      }
    }
  }
#endif
  if (flags) *flags = v;
  if (v) return fail(h, DFLASH_EDEVICE, "device-side check fired (see flags)");
  return DFLASH_OK;
}

}  // extern "C"

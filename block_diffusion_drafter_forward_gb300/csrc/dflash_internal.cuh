// Internal declarations shared by the library's translation units: the handle, the
// paged-pool addressing, small device helpers and the kernel launchers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "dflash.h"

namespace dflash {

constexpr int kPage = 16;     // rows per K/V page (from_weights.rs paged pool: block size 16)
constexpr int kGamma = 16;    // block rows (drafts = gamma - 1)

// ---------------------------------------------------------------- paged pool addressing
// Pool = [layer][page][kv][kv_head] tiles of 16 x hd elements.  Inside a tile the rows
// (page offset j) and head dims d are stored in 8x8 blocks, the operand layout of the
// tensor-core attention kernel (K: keys x dims, dims fastest; V: dims x keys, keys fastest).
__host__ __device__ inline int64_t k_in_tile(int j, int d, int hd) {
  return (int64_t)(((j >> 3) * (hd >> 3) + (d >> 3)) * 64 + (j & 7) * 8 + (d & 7));
}
__host__ __device__ inline int64_t v_in_tile(int j, int d, int /*hd*/) {
  return (int64_t)(((d >> 3) * 2 + (j >> 3)) * 64 + (d & 7) * 8 + (j & 7));
}

struct PoolGeom {
  int64_t tile;        // elements per tile: 16 * hd
  int64_t head_stride; // = tile
  int64_t kv_stride;   // = nkv * tile
  int64_t page_stride; // = 2 * nkv * tile
  int64_t layer_stride;// = num_pages * page_stride
  int num_pages;
  int nkv, hd;
};

__host__ __device__ inline int64_t tile_base(const PoolGeom& g, int layer, int page, int kv, int head) {
  return layer * g.layer_stride + (int64_t)page * g.page_stride + kv * g.kv_stride + head * g.head_stride;
}

// ---------------------------------------------------------------- element conversions
template <typename T> struct Elem;
template <> struct Elem<float> {
  __device__ static float load(const float* p) { return *p; }
  __device__ static float to_f(float v) { return v; }
  __device__ static float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  __device__ static float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// ---------------------------------------------------------------- profiling
enum Kind {
  K_EMBED, K_NORM, K_QKV, K_QKV_POST, K_ATTN, K_OPROJ, K_GATEUP, K_SILU, K_DOWN, K_LMHEAD, K_ARGMAX,
  K_COPY, K_W_FC, K_W_NORM, K_W_KV, K_W_POST, K_PERSIST, K_MARKOV, K_COUNT
};
static const char* const kKindNames[K_COUNT] = {
    "embed", "rmsnorm", "qkv_gemm", "qkv_post", "attention", "o_proj_gemm", "gate_up_gemm", "silu_mul",
    "down_gemm", "lm_head", "argmax", "copy", "writer_fc_gemm", "writer_norm", "writer_kv_gemm", "writer_post",
    "persistent_forward", "markov_chain"};

struct Prof {
  bool on = false;
  int64_t launches[K_COUNT] = {};
  double ms[K_COUNT] = {};
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> pending;
  std::vector<cudaEvent_t> spare;
};

// One captured propose (CUDA graph) and the arguments it was captured with.
struct GraphEntry {
  int nb = 0, max_ctx = 0;
  const void* args[8] = {};           // bonus, ctx_lens, page_tables, drafts, logits, hidden,
                                      // q_rope_pos, widths
  bool prof = false;                  // captured with per-kernel timing events
  bool persist = false;               // captured on the single-launch persistent forward
  cudaGraphExec_t exec = nullptr;
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> evs;  // owned timing events
  int64_t kind_counts[K_COUNT] = {};
  bool pending = false;               // events of the last launch not yet accumulated
  uint64_t stamp = 0;
};

// ---------------------------------------------------------------- the handle
struct LayerW {
  void* ln_in = nullptr;
  void* ln_post = nullptr;
  void* q_norm = nullptr;
  void* k_norm = nullptr;
  void* w_qkv = nullptr;   // [(nh + 2 nkv) hd, H]: q rows, then k rows, then v rows
  void* w_o = nullptr;     // [H, nh hd]
  void* w_gu = nullptr;    // [2F, H]: gate rows then up rows
  void* w_down = nullptr;  // [H, F]
  // FP8 drafter lane: the same four packed projections as e4m3 codes + per-row fp32 scales
  uint8_t* qkv8 = nullptr;
  uint8_t* o8 = nullptr;
  uint8_t* gu8 = nullptr;
  uint8_t* down8 = nullptr;
  float* qkv_s = nullptr;
  float* o_s = nullptr;
  float* gu_s = nullptr;
  float* down_s = nullptr;
};

}  // namespace dflash

struct dflash_handle {
  dflash_cfg cfg{};
  int device = 0;
  int num_sms = 0;
  size_t esz = 2;                      // bytes per element of cfg.dtype
  std::vector<void*> allocs;           // every library-owned device buffer

  // weights
  void* fc = nullptr;                  // [H, n_taps * Ht]
  void* hidden_norm = nullptr;         // [H]
  void* norm = nullptr;                // [H]
  const void* embed = nullptr;         // [V, H] borrowed
  const void* lm_head = nullptr;       // [V, H] borrowed (cfg.dtype)
  uint8_t* lm_fp8 = nullptr;           // [V, H] e4m3 codes (owned) when FP8
  float* lm_scale = nullptr;           // [V]
  void* w_ctxkv = nullptr;             // [L * 2 * kv, H]: K_0, V_0, K_1, V_1, ...
  void* kn_all = nullptr;              // [L, hd] every layer's k_norm (writer epilogue)
  dflash::LayerW layer[64];
  float2* rope_inv_pi = nullptr;       // [hd/2] inv_freq_j / pi split as (hi, lo) floats
  float rope_mscale = 1.f;

  // paged K/V pool
  void* pool = nullptr;
  size_t pool_bytes = 0;
  dflash::PoolGeom geom{};

  // propose scratch (rows = max_batch * gamma)
  int rows_max = 0;
  float* x = nullptr;                  // [rows, H] residual stream, fp32
  void* xn = nullptr;                  // [rows, H] normed activations (cfg.dtype)
  float* y = nullptr;                  // [rows, ymax] fp32 projection outputs
  void* q = nullptr;                   // [rows, nh hd]
  void* attn = nullptr;                // [rows, nh hd]
  void* act = nullptr;                 // [rows, F]
  float* logits32 = nullptr;           // [rows, V] fp32 logits
  // writer scratch (rows = max_write_rows)
  float* wy = nullptr;                 // [Rw, max(H, L*2*kv)] fp32
  float* wf = nullptr;                 // [Rw, H] ctx features (fp32)
  void* wf2 = nullptr;                 // [Rw, 2H] ctx features as bf16 [hi | lo] (tensor-core writer)

  // tensor-core (bf16) path scratch
  void* xb = nullptr;                  // [rows, H] bf16 copy of the residual stream
  float* ss_a = nullptr;               // [H/128, rows] partial sums of x^2 after o_proj
  float* ss_b = nullptr;               // [H/128, rows] partial sums of x^2 after down_proj / embed
  float* ws = nullptr;                 // split-K partials
  size_t ws_floats = 0;
  unsigned* counters = nullptr;        // split-K / argmax counters (zero between launches)
  unsigned long long* amax_best = nullptr;  // [rows] packed running argmax (zero between launches)
  float* attn_opart = nullptr;         // attention split partials (O)
  float* attn_ml = nullptr;            // attention split partials (max, sum)
  bool tc = false;                     // bf16 tensor-core path in use
  bool tc_attn = false;                // tensor-core attention (8 query heads per kv head)
  // single-launch persistent forward (batch 1, bf16 lm_head)
  bool persist_ok = false;             // available for this configuration and device
  bool persist_on = false;             // used by dflash_propose (dflash_set_persistent)
  void* p_maps = nullptr;              // device CUtensorMap table
  void* xb2 = nullptr;                 // [rows, H] bf16 gate/up operand of the single launch
  size_t p_ws_half = 0;                // floats in each half of the single launch's partials
  unsigned* p_ctl = nullptr;           // control words, zeroed before each launch
  size_t p_ctl_words = 0;
  unsigned long long* p_trace = nullptr;  // phase timeline (DFLASH_PHASE_TRACE builds only)
  size_t p_trace_words = 0;
  // DSpark Markov head (cfg.markov_rank > 0)
  void* mk_w1 = nullptr;               // [V, rank] cfg.dtype (owned copy)
  void* mk_w2 = nullptr;               // [V, rank]
  void* mk_ctl = nullptr;              // per-step argmax keys and barriers, zeroed before each launch
  size_t mk_ctl_bytes = 0;

  // per-call optional inputs of dflash_propose_ex (device arrays [nb] or null), read by the
  // launchers of the call being issued or captured
  const int32_t* cur_rope_pos = nullptr;
  const int32_t* cur_widths = nullptr;

  unsigned* d_status = nullptr;        // device status word
  dflash::Prof prof;
  // CUDA graphs of dflash_propose, keyed by its arguments (small LRU)
  std::vector<dflash::GraphEntry*> graphs;
  uint64_t graph_clock = 0;
  cudaStream_t cap_stream = nullptr;   // private stream used only for capture
  dflash::GraphEntry* cap_entry = nullptr;  // non-null while capturing
  std::string err;
};

namespace dflash {

// Active block width of sequence s (dflash_propose_ex): widths[s] clamped to [2, gamma];
// gamma when no widths are given.
__device__ __forceinline__ int block_width(const int32_t* widths, int s) {
  if (!widths) return kGamma;
  const int w = __ldg(widths + s);
  return w < 2 ? 2 : (w > kGamma ? kGamma : w);
}
__device__ __forceinline__ bool width_out_of_range(const int32_t* widths, int s) {
  if (!widths) return false;
  const int w = __ldg(widths + s);
  return w < 2 || w > kGamma;
}
// RoPE position of block row 0 of sequence s: q_rope_pos[s], or the context length.
__device__ __forceinline__ int rope_start(const int32_t* rope_pos, int s, int ctx) {
  return rope_pos ? __ldg(rope_pos + s) : ctx;
}

// One 16-byte piece x (0 <= x < 2048) of the queries of unit (sequence s, kv head g) into sQ,
// the no-swizzle K-major operand of S = Q K^T (row = head hh * 16 + token r in 8-row x 16-byte
// core matrices), as a cp.async copy.  x = 128 r + 16 hh + d8: the 8 query heads of one token
// are 2 KB contiguous in q, so 32 consecutive x read 512 contiguous bytes.  The caller waits
// (cp.async.wait_group), then fences the copies for the async proxy before the MMA reads sQ.
__device__ __forceinline__ void stage_q_piece(uint8_t* sQ, const __nv_bfloat16* q, int s, int g, int nh, int x) {
  const int r = x >> 7, hh = (x >> 4) & 7, d8 = x & 15;
  const int row = hh * 16 + r;
  const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(sQ + ((row >> 3) * 16 + d8) * 128 + (row & 7) * 16));
  const __nv_bfloat16* src = q + ((int64_t)(s * kGamma + r) * nh + g * 8 + hh) * 128 + d8 * 8;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Split-attention partial O (fp32, unnormalised) of slot `slot`: 128 rows x 128 dims as float4
// dim blocks (dims 4 db .. 4 db + 3), stored [slot][row / 4][db][row % 4]: the 4 rows a combine
// block merges are 2 KB contiguous per slot, and a row-per-thread writer's warp stores 64
// contiguous bytes per group of 4 rows.  Returns the float4 of (row r, dim block db).
__host__ __device__ __forceinline__ float4* o_part_at(float* o_part, int64_t slot, int r, int db) {
  return reinterpret_cast<float4*>(o_part) + ((slot * 32 + (r >> 2)) * 32 + db) * 4 + (r & 3);
}

// ---------------------------------------------------------------- launchers (kernels_simple.cu)
// All launchers are stream-ordered and return cudaGetLastError() of the launch.
cudaError_t launch_embed(const dflash_handle* h, const int32_t* bonus, int nb, float* x, cudaStream_t st);
cudaError_t launch_rmsnorm_f32in(const dflash_handle* h, const float* x, const void* w, void* out,
                                 int rows, int n, cudaStream_t st);
// Y[m, n] (+)= sum_k X[m, k] W[n, k]; X, W in cfg.dtype; Y fp32 with row stride ldy.
cudaError_t launch_gemm(const dflash_handle* h, const void* X, int ldx, const void* W, int M, int N,
                        int K, float* Y, int ldy, bool accumulate, cudaStream_t st);
cudaError_t launch_gemm_xf32(const dflash_handle* h, const float* X, int ldx, const void* W, int M, int N, int K,
                             float* Y, int ldy, cudaStream_t st);
cudaError_t launch_rmsnorm_f32out(const dflash_handle* h, const float* x, const void* w, float* out, int rows, int n,
                                  cudaStream_t st);
cudaError_t launch_gemm_fp8w(const dflash_handle* h, const void* X, int ldx, const uint8_t* Wq,
                             const float* scale, int M, int N, int K, float* Y, int ldy,
                             cudaStream_t st);
cudaError_t launch_qkv_post(const dflash_handle* h, int layer, const float* y, const int32_t* ctx_lens,
                            const int32_t* page_tables, int nb, void* q, cudaStream_t st);
cudaError_t launch_attention(const dflash_handle* h, int layer, const void* q, const int32_t* ctx_lens,
                             const int32_t* page_tables, int nb, int max_ctx_len, void* out,
                             cudaStream_t st);
cudaError_t launch_silu_mul(const dflash_handle* h, const float* y, int rows, void* act, cudaStream_t st);
cudaError_t launch_argmax(const dflash_handle* h, const float* logits32, int nb, int32_t* drafts,
                          void* logits_out, cudaStream_t st);
cudaError_t launch_copy_hidden(const dflash_handle* h, const void* src, int rows, void* dst, cudaStream_t st);
// Row i goes to row first + i of the one sequence of page_table, or (row_seq / row_index given,
// the batched writer) to row row_index[i] of sequence row_seq[i] of page_table [nseq, mpps].
cudaError_t launch_ctxkv_post(const dflash_handle* h, const float* ykv, int n, const int32_t* positions,
                              const int32_t* page_table, int first, cudaStream_t st,
                              const int32_t* row_seq = nullptr, const int32_t* row_index = nullptr, int nseq = 1);
cudaError_t launch_embed_tc(const dflash_handle* h, const int32_t* bonus, int nb, cudaStream_t st);
cudaError_t launch_split_hi_lo(const float* x, int rows, int n, void* out, cudaStream_t st);
cudaError_t launch_fold_norm(const void* A, const void* B, int mode, int rows, int cols, const void* ln, void* out,
                             cudaStream_t st);
cudaError_t launch_quantize_fp8(const void* w, int rows, int cols, int dtype, uint8_t* codes,
                                float* scale, cudaStream_t st);

}  // namespace dflash

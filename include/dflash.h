/*
 * dflash.h -- C ABI of the GB300 DFlash drafter library (libdflash.so).
 *
 * The library runs the gamma-block forward of a DFlash block-diffusion drafter: a small
 * Qwen3-class transformer that drafts gamma-1 tokens in ONE non-causal forward over a
 * block [bonus, mask x (gamma-1)], conditioned on a paged K/V cache built from the
 * target model's tapped hidden states.  Sources for the operations (page: section):
 *   - memra-engine `dflash.rs` (docs.rs 0.94.0): ctx_features, ingest_ctx,
 *     forward_round, the draft step of generate_spec_dflash, the YaRN block of load.
 *   - spark_model `dflash_head/from_weights.rs`: paged BF16 pool (16 rows/page),
 *     fused context K/V weight, RoPE/YaRN table, FP8 per-row weight quantisation.
 *   - spark_model `layers/dflash_head.rs`: batched propose (sequences stacked
 *     seq-major, gamma rows each; row 0 of a band is the anchor echo).
 *
 * General rules for every call:
 *   - Tensor arguments are DEVICE pointers unless stated; calls are asynchronous and
 *     stream-ordered on `stream` (a cudaStream_t; NULL = legacy default stream).  No
 *     call synchronises the host except dflash_create (weight packing), dflash_destroy
 *     and dflash_device_status.
 *   - The return value is a dflash_status.  A non-zero status means nothing was
 *     launched by that call (argument and capacity checks run on the host first);
 *     dflash_last_error() then gives a message.
 *   - Device-side checks (a page id outside [0, num_pages), a context length outside
 *     [0, max_ctx_len] or past the page table, a bonus token outside [0, vocab), a bounded
 *     wait that gave up) never trap: the offending row is skipped (a bad token's row is
 *     embedded as zeros) and a bit is set in the handle's device status word, read (and
 *     cleared) by dflash_device_status().
 *   - A handle is not thread-safe: one caller at a time (one draft step at a time, as in
 *     the pages' proposer contract).
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                         /* cudaStream_t is `struct CUstream_st*` */
typedef struct CUstream_st* dflash_stream;
typedef struct dflash_handle dflash_handle;  /* opaque */

typedef enum {
  DFLASH_OK = 0,
  DFLASH_EINVAL = -1,       /* bad argument (null pointer, shape, unsupported combination) */
  DFLASH_ENOMEM = -2,       /* device allocation failed in dflash_create */
  DFLASH_ECUDA = -3,        /* a CUDA runtime call failed (message has the CUDA error) */
  DFLASH_ECAPACITY = -4,    /* nb > max_batch, rows beyond the page-table capacity, ... */
  DFLASH_EUNSUPPORTED = -5, /* configuration outside what the kernels implement */
  DFLASH_EDEVICE = -6       /* dflash_device_status: a device-side check fired */
} dflash_status;

typedef enum {
  DFLASH_F32 = 0,              /* fp32 weights, activations and K/V cache (CUDA-core path) */
  DFLASH_BF16 = 1,             /* bf16 weights, activations and K/V cache (tensor-core path) */
  DFLASH_FP8E4M3_ROWSCALE = 2  /* lm_head_dtype / layer_weight_dtype: e4m3 codes + one fp32 scale
                                  per output row */
} dflash_dtype;

/* Device status bits (dflash_device_status). */
#define DFLASH_DEV_BAD_PAGE 0x1u    /* a page id outside [0, num_pages) was met */
#define DFLASH_DEV_BAD_CTX 0x2u     /* ctx_len < 0 or > max_ctx_len, or ctx_len+gamma > capacity */
#define DFLASH_DEV_BAD_TOKEN 0x4u   /* a bonus token outside [0, vocab) (row embedded as zeros) */
#define DFLASH_DEV_TIMEOUT 0x8u     /* a kernel's bounded wait gave up (its outputs are invalid) */
#define DFLASH_DEV_BAD_WIDTH 0x10u  /* dflash_propose_ex: a block width outside [2, gamma] (clamped) */

/* Drafter configuration.  Names follow the drafter config.json of the pages
 * (hidden_size, num_attention_heads, num_key_value_heads, head_dim, intermediate_size,
 * num_hidden_layers, vocab_size, block_size = gamma, mask_token_id,
 * len(target_layer_ids) = n_taps, rms_norm_eps, rope_theta, rope_scaling (yarn),
 * sliding_window, layer_types). */
typedef struct {
  int32_t hidden;           /* H */
  int32_t n_q_heads;        /* nh */
  int32_t n_kv_heads;       /* nkv; nh % nkv == 0 (GQA: q head h reads kv head h / (nh/nkv)) */
  int32_t head_dim;         /* hd: 64 or 128 (bf16 path: 128) */
  int32_t n_ff;             /* F */
  int32_t n_layers;         /* L <= 64 */
  int32_t vocab;            /* V */
  int32_t gamma;            /* block rows; must be 16 */
  int32_t mask_token_id;
  int32_t n_taps;           /* number of tapped target layers */
  int32_t target_hidden;    /* hidden size of the target (per tap) */
  float rms_eps;            /* e.g. 1e-6 */
  float rope_theta;         /* e.g. 1e6 */
  int32_t rope_yarn;        /* 0: plain RoPE; 1: YaRN (the four fields below) */
  float yarn_factor, yarn_orig_max_pos, yarn_beta_fast, yarn_beta_slow;
  int32_t sliding_window;   /* W > 0 for sliding layers; ignored where layer_sliding is 0 */
  uint8_t layer_sliding[64];/* per layer: 1 = sliding-window attention */
  int32_t dtype;            /* DFLASH_F32 or DFLASH_BF16 */
  int32_t lm_head_dtype;    /* == dtype, or DFLASH_FP8E4M3_ROWSCALE (quantised at create) */
  int32_t page_size;        /* must be 16 */
  int32_t num_pages;        /* K/V pool capacity in pages (library-owned pool) */
  int32_t max_batch;        /* largest nb passed to dflash_propose */
  int32_t max_pages_per_seq;/* row stride of page tables; capacity = 16 * this rows */
  int32_t max_write_rows;   /* rows per internal chunk of dflash_write_ctx_kv (>= 16) */
  int32_t markov_rank;      /* DSpark Markov head rank; 0 = no head.  Otherwise a multiple of 32,
                               <= 1024, with max_batch <= 64 and max_batch * rank <= 40960 */
  int32_t layer_weight_dtype; /* 0 or dtype: as dtype; DFLASH_FP8E4M3_ROWSCALE (bf16 drafters): the FP8
                               drafter lane (from_weights.rs Phase G), q/k/v/o/gate/up/down of every
                               layer quantised at create to e4m3 with a per-output-row fp32 scale
                               (scale = fp32 rowmax|w| / 448) and used by dflash_propose; the
                               context-K/V writer keeps the bf16 K/V weights */
} dflash_cfg;

/* One layer's weights, HF layout (Linear weights [out, in] row-major), all in cfg.dtype,
 * device pointers.  Read during dflash_create only (copied and repacked). */
typedef struct {
  const void* ln_in;    /* [H]            input_layernorm */
  const void* wq;       /* [nh*hd, H]     q_proj */
  const void* wk;       /* [nkv*hd, H]    k_proj */
  const void* wv;       /* [nkv*hd, H]    v_proj */
  const void* q_norm;   /* [hd] */
  const void* k_norm;   /* [hd] */
  const void* wo;       /* [H, nh*hd]     o_proj */
  const void* ln_post;  /* [H]            post_attention_layernorm */
  const void* w_gate;   /* [F, H] */
  const void* w_up;     /* [F, H] */
  const void* w_down;   /* [H, F] */
} dflash_layer_weights;

typedef struct {
  const void* fc;           /* [H, n_taps*target_hidden]   copied */
  const void* hidden_norm;  /* [H]                         copied */
  const void* norm;         /* [H] final norm              copied */
  const void* embed;        /* [V, H] target embedding: BORROWED, must outlive the handle */
  const void* lm_head;      /* [V, H] target lm_head (cfg.dtype): BORROWED when lm_head_dtype
                               == dtype; read once to quantise when it is FP8 */
  const dflash_layer_weights* layers; /* host array of n_layers entries */
  /* DSpark Markov head (read when cfg.markov_rank > 0, copied; dflash.rs draft step, Markov
   * chain block; dflash_head.rs DSpark fields), cfg.dtype, row-major: */
  const void* markov_w1;    /* [V, rank] previous-token table */
  const void* markov_w2;    /* [V, rank] Linear(rank, V) weight */
} dflash_weights;

/* Create a drafter: validates cfg, copies and repacks the layer weights into
 * library-owned device buffers (fused QKV, fused gate/up, fused context-K/V), allocates
 * the paged K/V pool of
 * cfg.num_pages pages and the scratch for cfg.max_batch sequences, builds the RoPE
 * table (from_weights.rs inv_freq / YaRN block, in float64 on the host), and quantises
 * the lm_head to e4m3 when asked (from_weights.rs FP8 block).  Synchronises `stream`.
 * On success *out is a new handle.  Errors: EINVAL / EUNSUPPORTED / ENOMEM / ECUDA. */
int dflash_create(const dflash_cfg* cfg, const dflash_weights* weights, dflash_stream stream,
                  dflash_handle** out);

/* Free every library-owned buffer (after synchronising the device). NULL is a no-op. */
int dflash_destroy(dflash_handle* h);

/* Context-K/V writer for ONE sequence (dflash.rs ctx_features + ingest_ctx;
 * from_weights.rs fused K/V weight + reshape_and_cache):
 *   f_i   = hidden_norm(fc . taps_i)
 *   K_l,i = mscale * RoPE(k_norm_l(Wk_l f_i), positions[i]);  V_l,i = Wv_l f_i
 * stored for every layer l at logical rows first..first+n-1 of the sequence, i.e. slot
 * page_table[(first+i)/16]*16 + (first+i)%16 of the pool.
 *   taps       [n, n_taps*target_hidden] cfg.dtype, taps concatenated in
 *              target_layer_ids order, row-major.
 *   positions  [n] int32 RoPE positions of the rows (usually first..first+n-1).
 *   page_table [max_pages_per_seq] int32, the sequence's pages.
 * Requires 0 <= first, n >= 0, first + n <= 16 * max_pages_per_seq (ECAPACITY).
 * n == 0 is a no-op.  Rows are processed in chunks of cfg.max_write_rows. */
int dflash_write_ctx_kv(dflash_handle* h, const void* taps, const int32_t* positions,
                        const int32_t* page_table, int32_t first, int32_t n,
                        dflash_stream stream);

/* Batched context-K/V writer: one call over the new rows of many sequences (dflash_head.rs
 * batched precompute_ctx_kv over every sequence's uncommitted rows; dflash.rs prime ingest),
 * the same arithmetic as dflash_write_ctx_kv row by row, with the fc and fused K/V weights
 * streamed once per chunk of cfg.max_write_rows rows instead of once per sequence.
 *   taps       [n, n_taps*target_hidden] cfg.dtype, rows of any sequences in any order.
 *   positions  [n] int32 RoPE positions of the rows.
 *   row_seq    [n] int32: sequence of row i (a row of page_tables), in [0, nseq).
 *   row_index  [n] int32: logical row index of row i within its sequence, in
 *              [0, 16 * max_pages_per_seq); row i goes to slot
 *              page_tables[row_seq[i]][row_index[i] / 16] * 16 + row_index[i] % 16.
 *   page_tables [nseq, max_pages_per_seq] int32.
 * Two rows aimed at the same slot race (one of them wins).  A row whose row_seq or row_index
 * is out of range is skipped and sets DFLASH_DEV_BAD_CTX; a bad page id DFLASH_DEV_BAD_PAGE.
 * n == 0 is a no-op; nseq >= 1. */
int dflash_write_ctx_kv_batch(dflash_handle* h, const void* taps, const int32_t* positions,
                              const int32_t* row_seq, const int32_t* row_index,
                              const int32_t* page_tables, int32_t nseq, int32_t n,
                              dflash_stream stream);

/* One gamma-block forward over nb sequences (dflash.rs forward_round + final norm +
 * lm_head + argmax; dflash_head.rs propose_batch band layout).  Sequence s drafts from
 * its block [bonus_tokens[s], mask x (gamma-1)] at positions ctx_lens[s] + r, attends
 * (non-causally, GQA, windowed on sliding layers) over its ctx_lens[s] cached rows plus
 * the block, and writes:
 *   draft_tokens [nb, gamma-1] int32: argmax over the vocabulary of block rows 1..gamma-1
 *                (ties -> lowest id).  Required.
 *   logits       [nb*gamma, V] cfg.dtype (fp32 when dtype is F32, bf16 otherwise),
 *                all gamma rows of every band; NULL = not written.
 *   final_hidden [nb*gamma, H] cfg.dtype, final-normed hidden; NULL = not written.
 * With a Markov head (cfg.markov_rank > 0) the drafts come from the DSpark semi-autoregressive
 * chain instead (dflash.rs draft step): from chain_0 = bonus_tokens[s], for k = 0..gamma-2,
 * logits row k+1 += markov_w2 . markov_w1[chain_k] and chain_{k+1} = its argmax; drafts are
 * chain_1..chain_{gamma-1}, and logit rows 1..gamma-1 (when written) carry the added bias.
 * Inputs: bonus_tokens [nb] int32, ctx_lens [nb] int32, page_tables
 * [nb, max_pages_per_seq] int32 (row s = sequence s's pages; entries past
 * ceil((ctx_lens[s]+gamma)/16) are not read).  max_ctx_len is a HOST upper bound of
 * ctx_lens, used for grid sizing; it must satisfy max_ctx_len + gamma <=
 * 16 * max_pages_per_seq (ECAPACITY).  The block K/V are written transiently into rows
 * ctx_lens[s]..ctx_lens[s]+gamma-1 of each sequence's pages (never committed: the next
 * dflash_write_ctx_kv at first = ctx_len overwrites them).  1 <= nb <= max_batch.
 * The launch sequence is captured as a CUDA graph the first time a given set of pointers,
 * nb and max_ctx_len is seen (a small per-handle cache) and replayed after that; the values
 * in the input buffers may change freely between calls.  A caller that passes new buffer
 * addresses every call pays a graph capture each time: reuse the buffers. */
int dflash_propose(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens,
                   const int32_t* page_tables, int32_t nb, int32_t max_ctx_len,
                   int32_t* draft_tokens, void* logits, void* final_hidden,
                   dflash_stream stream);

/* dflash_propose with two optional per-sequence inputs, both device arrays [nb] int32 read by
 * the kernels at run time (so one captured graph serves every value; NULL = the default):
 *   q_rope_pos  RoPE position of block row 0 of sequence s (block row r at q_rope_pos[s] + r);
 *               default ctx_lens[s] (dflash_head.rs / from_weights.rs indirect arguments
 *               [kv_len, q_offset, q_rope_pos]).  The K/V rows and the sliding window keep the
 *               row indices ctx_lens[s] + r.  Positions must lie in [0, 2^24).
 *   widths      active block width b of sequence s, 2 <= b <= gamma (dflash_head.rs block-width
 *               resolver): the block is [bonus, mask x (b-1)], its b rows attend to the context
 *               and to each other only, and drafts[s, 0..b-2] are the argmaxes of rows 1..b-1;
 *               drafts[s, b-1..gamma-2] are set to -1 and logit / hidden rows b..gamma-1 of the
 *               band hold no meaningful values.  Default gamma.  A width outside [2, gamma] is
 *               clamped and sets DFLASH_DEV_BAD_WIDTH.
 * Everything else as dflash_propose (the graph cache also keys on these two pointers). */
int dflash_propose_ex(dflash_handle* h, const int32_t* bonus_tokens, const int32_t* ctx_lens,
                      const int32_t* page_tables, int32_t nb, int32_t max_ctx_len,
                      const int32_t* q_rope_pos, const int32_t* widths, int32_t* draft_tokens,
                      void* logits, void* final_hidden, dflash_stream stream);

/* Layout of the library-owned K/V pool (for tests and inspection).  *pool = device base,
 * *bytes = size, strides (in ELEMENTS of cfg.dtype) for the tile index
 * [layer][page][kv (0 = K, 1 = V)][kv_head] in strides[0..3]; strides[4] = elements per
 * tile (16 * head_dim); strides[5] = element size in bytes.  A head's V tile directly follows
 * its K tile (strides[2] == strides[4]), so one page of one head is one contiguous run of
 * K then V.  Inside a tile of page rows
 * j (0..15) and head dims d (0..hd-1), the element offset is
 *   K tile:  ((j/8) * (hd/8) + d/8) * 64 + (j%8) * 8 + d%8
 *   V tile:  ((d/8) * 2     + j/8) * 64 + (d%8) * 8 + j%8
 * (8x8 blocks, the operand layout of the tensor-core attention kernel). */
int dflash_kv_layout(const dflash_handle* h, void** pool, size_t* bytes, int64_t strides[6]);

/* The e4m3 lm_head built by dflash_create when lm_head_dtype is FP8 (for tests):
 * *codes = [V, H] uint8 e4m3 codes, *scales = [V] fp32 per-row scales, device pointers
 * owned by the handle.  EINVAL when the lm_head is not FP8. */
int dflash_fp8_lm_head(const dflash_handle* h, const uint8_t** codes, const float** scales);

/* The e4m3 layer weights built by dflash_create when layer_weight_dtype is FP8 (for tests):
 * proj 0 = fused q|k|v [(nh+2nkv)*hd, H] (q rows, then k, then v), 1 = o_proj [H, nh*hd],
 * 2 = gate/up [2F, H] packed in blocks of 64 rows (block b: gate rows 64b..64b+63, then the
 * matching up rows), 3 = down [H, F]; *codes row-major uint8, *scales fp32 per row, device
 * pointers owned by the handle.  EINVAL when the layer weights are not FP8 or the indices are
 * out of range. */
int dflash_fp8_layer(const dflash_handle* h, int32_t layer, int32_t proj, const uint8_t** codes,
                     const float** scales);

/* Per-kernel timing for benchmarks.  dflash_profile(h, 1) clears the counters and from
 * then on brackets every kernel launch of the handle with CUDA events on the launch
 * stream; dflash_profile(h, 0) stops recording.  Launch counts are kept in both modes.
 * dflash_profile_read(h, k, ...) reports kernel kind k (0 <= k < dflash_profile_kinds()):
 * its name, the summed event time in ms of the recorded launches (synchronises on the
 * recorded events) and the number of launches since the last dflash_profile call. */
int dflash_profile(dflash_handle* h, int enable);
int dflash_profile_kinds(void);
int dflash_profile_read(dflash_handle* h, int kind, const char** name, double* total_ms,
                        int64_t* launches);

/* Single-launch forward.  On bf16 handles with a bf16 lm_head and 8 query heads per kv
 * head, dflash_propose with nb == 1 runs the whole gamma-block forward (embedding, every
 * layer, final norm, lm_head and argmax) as ONE persistent kernel with one CTA per SM;
 * larger batches launch one kernel per projection.  Both give the same result up to the
 * summation order of the split-K partial sums.  dflash_set_persistent(h, 0) makes nb == 1
 * use the per-projection kernels too (for comparisons); enabling it where it is not
 * available returns DFLASH_EUNSUPPORTED.  dflash_persistent(h) is 1 when it is in use. */
int dflash_set_persistent(dflash_handle* h, int enable);
int dflash_persistent(const dflash_handle* h);

/* The tensor-core projection GEMM on its own (for tests): out[m, n] = sum_k W[n, k] X[m, k]
 * with W [N, K] and X [M, K] bf16 row-major device arrays, out [M, N] fp32.  K % 64 == 0,
 * nsplit must be 1.  Same kernel as every bf16 projection of dflash_propose. */
int dflash_gemm_bf16(const void* W, int32_t N, int32_t K, const void* X, int32_t M, float* out,
                     int32_t nsplit, dflash_stream stream);

/* Split-K projection GEMM that allocates nothing (no counterpart in the paper: it exists
 * for callers, not for the method).  Same product and kernel as dflash_gemm_bf16,
 * out[m, n] = sum_k W[n, k] X[m, k] (W [N, K], X [M, K] bf16, out [M, N] fp32, K % 64 == 0),
 * with the K dimension split `nsplit` ways (1..16, <= K/64) and summed in split order.
 * For callers that cannot call cudaMalloc while running: a serving loop that reserved all
 * device memory at start-up, a memory pool that owns the device, a runtime that forbids
 * allocation after initialisation.  Its scratch (split-K partials, tile counters) is a
 * fixed array in the library's device image: 8 MiB of partials and 4096 tiles, held on
 * every GPU that loads the library until the process exits.  With TN = 16, 32, 64 or 128
 * token columns per tile (M <= 16, <= 32, <= 64, else 128) and tiles = ceil(N/128) *
 * ceil(M/TN), shapes need tiles <= 4096 and tiles * nsplit * 128 * TN <= 2^21 floats;
 * larger ones return ECAPACITY.  All calls share that array: calls that overlap on the GPU
 * (two streams, two threads) race and give wrong results, so serialise them.  The first
 * call in a CUDA context (per device, and again after cudaDeviceReset or a new primary
 * context) looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  Each call zeroes the counters
 * it uses on `stream`.  A bounded device-side wait that gives up is not reported by this
 * call (it leaves the affected output tiles unwritten). */
int dflash_gemm_bf16_noalloc(const void* W, int32_t N, int32_t K, const void* X, int32_t M,
                             float* out, int32_t nsplit, dflash_stream stream);

/* Attention cross-check (for tests, bf16 handles with 8 query heads per kv head): runs the
 * CUDA-core and the tensor-core block attention of `layer` on the queries left in the
 * handle by the last dflash_propose (its last layer's) and the pool, writing both
 * [nb*gamma, nh*hd] bf16 outputs.  Arguments as in dflash_propose. */
int dflash_attention_check(dflash_handle* h, int32_t layer, const int32_t* ctx_lens,
                           const int32_t* page_tables, int32_t nb, int32_t max_ctx_len,
                           void* out_cuda_core, void* out_tensor_core, dflash_stream stream);

/* Synchronise `stream`, read the device status word into *flags (may be NULL) and clear
 * it.  When DFLASH_DEV_TIMEOUT was set it also re-arms the handle's internal tile counters
 * (a kernel that gave up a wait may have left them part-counted), so the next call starts
 * clean.  Returns DFLASH_EDEVICE when any bit was set, else DFLASH_OK. */
int dflash_device_status(dflash_handle* h, dflash_stream stream, uint32_t* flags);

/* Last error message of the handle ("" if none); with h == NULL the message of the last
 * failed dflash_create on this thread. */
const char* dflash_last_error(const dflash_handle* h);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */

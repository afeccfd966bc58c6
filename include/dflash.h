/*
 * dflash.h - C ABI of the GB300 (sm_103a) DFlash block-diffusion drafting
 * library.  One call per step of the drafting hot path:
 *
 *   dflash_inject_context   target features -> every drafter layer's KV cache
 *   dflash_draft_block      one parallel forward over an S-token block
 *   dflash_select_path      top-16 candidates -> one draft (DFlash-2 Path
 *                           Selector, or top-1 per position)
 *   dflash_verify_greedy    greedy prefix acceptance against target tokens
 * and the sampling modes of the same steps:
 *   dflash_sample_path      a draft drawn over the path scores at a temperature
 *   dflash_verify_rejection rejection sampling against target logits (lossless)
 * Engine options ([DF2] table of inference engines): the block size S may be
 * changed between steps (dflash_set_block_size), and the drafter's weights
 * may be FP8 (dflash_config.weight_fp8, "draft quantization").
 *
 * Pages the operations are defined by (cited below by these tags):
 *   [DF]  "DFlash - Difusion de Bloques para Decodificacion Especulativa en
 *         Flash" (gist.science, paper 2602.06036)
 *   [DF2] "DFlash 2: optimizacion de la decodificacion especulativa para
 *         inferencia paralela de LLMs" (kerneldigest.dev)
 *   [FD]  "FlexDraft" (gist.science, paper 2605.20022)
 *   [BW]  "DFlash: Avance en la inferencia de LLM con decodificacion
 *         especulativa en NVIDIA Blackwell" (emedoteme.es)
 *
 * General conventions
 *   - Every pointer named "device" is CUDA device memory owned by the caller;
 *     the library never allocates device memory and never frees caller memory.
 *   - Every call is asynchronous on the given stream and never synchronises
 *     (dflash_read_status and dflash_profile_end excepted).
 *   - Return value: DFLASH_OK (0) or a negative DFLASH_ERR_* code; on error
 *     nothing was launched and dflash_last_error() holds a message.
 *   - Element type: dflash_config.dtype selects bf16 (DFLASH_BF16) or fp32
 *     (DFLASH_F32) for every matrix, activation, KV cache and hidden state;
 *     norm gains, biases and logits are always fp32; ids are int32.
 *   - All matrices are row-major, W[out][in] (y = W x).  Every matrix base
 *     pointer and every row stride must be 16-byte aligned.
 *   - Workspace: one caller-owned device buffer of dflash_workspace_bytes()
 *     bytes, zero-filled ONCE after allocation.  Calls sharing a workspace
 *     must be ordered on one stream.  The first 256 bytes hold the device
 *     status word (see dflash_read_status).
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

typedef struct CUstream_st *dflash_stream_t;   /* == cudaStream_t */
typedef struct dflash_ctx dflash_ctx;            /* opaque */

enum {
  DFLASH_OK = 0,
  DFLASH_ERR_ARG = -1,          /* null pointer or out-of-range scalar       */
  DFLASH_ERR_SHAPE = -2,        /* sizes inconsistent with the config        */
  DFLASH_ERR_ALIGN = -3,        /* pointer / stride not 16-byte aligned      */
  DFLASH_ERR_UNSUPPORTED = -4,  /* e.g. head_dim not 64/128, block > 16      */
  DFLASH_ERR_CUDA = -5,         /* a CUDA runtime / driver call failed       */
  DFLASH_ERR_TIMEOUT = -6,      /* a bounded device wait ran out             */
  DFLASH_ERR_DEVICE = -7        /* a kernel reported bad data (page index)   */
};

enum { DFLASH_BF16 = 0, DFLASH_F32 = 1 };

/* Largest batch (requests per call) the workspace header is sized for; a
 * larger batch returns DFLASH_ERR_ARG. */
#define DFLASH_MAX_BATCH 4096

/* Drafter shape and flags.  block_size S in 2..16 (J = S - 1 mask positions
 * per request; 16 is the pages' block), top_k 16, page_size 64.  Below, S and
 * J in a shape stand for these two numbers. */
typedef struct dflash_config {
  int dtype;             /* DFLASH_BF16 or DFLASH_F32                        */
  int hidden;            /* H, multiple of 16                                */
  int n_layers;          /* L                                                */
  int n_q_heads;         /* nq                                               */
  int n_kv_heads;        /* nkv, divides nq, nq/nkv <= 8                     */
  int head_dim;          /* d: 128 (bf16) or 64/128 (fp32)                   */
  int ffn;               /* F (SwiGLU width)                                 */
  int vocab;             /* V                                                */
  int target_hidden;     /* H_t                                              */
  int n_target_layers;   /* n_sel; feature input width = n_sel * H_t         */
  int block_size;        /* S in 2..16: anchor + J = S-1 mask positions     */
  int top_k;             /* 16                                               */
  int use_conv;          /* DFlash-2 dynamic short convolution ([DF2] 2)     */
  int use_selector;      /* DFlash-2 Path Selector ([DF2] 1)                 */
  int qk_norm;           /* per-head RMSNorm of q and k                      */
  int fc_norm;           /* RMSNorm after the context-feature projection     */
  int split_act;         /* bf16 path: pass every GEMM activation as bf16
                            high + low halves (two MMAs per k-step): fp32-grade
                            activation precision; no extra weight traffic    */
  int sel_rank;          /* r of the bilinear form (<= 64)                   */
  int sel_dim;           /* selector embedding width (256)                   */
  int mask_id;           /* token id of the mask token                       */
  int page_size;         /* KV page size in tokens: 64                       */
  float rope_base;       /* RoPE base (1e6)                                  */
  float eps;             /* RMSNorm epsilon (1e-6)                           */
  int weight_fp8;        /* [DF2] engine flag "Draft quantization: enabled":
                            every GEMM weight (w_fc, w_qkv, w_o, w_gu, w_down,
                            w_conv, lm_head) is E4M3 codes (OCP FP8, 1 byte,
                            row stride = K bytes, a multiple of 16) with one
                            fp32 scale per output row in the s_* pointers:
                            W[n][k] = s[n] * e4m3(code[n][k]).  NaN codes
                            are invalid.  Activations stay bf16 (bf16 dtype
                            only); the embedding and selector tables stay
                            in dtype.                                       */
} dflash_config;

/* Per-layer weights (device pointers, not owned). */
typedef struct dflash_layer_weights {
  const float *g_attn;   /* [H] pre-attention RMSNorm gain                   */
  const void *w_qkv;     /* [(nq+2nkv)*d, H]: q heads, then k heads, then v  */
  const float *g_q;      /* [d] per-head q RMSNorm gain                      */
  const float *g_k;      /* [d] per-head k RMSNorm gain (also for injection) */
  const void *w_o;       /* [H, nq*d]                                        */
  const float *g_ffn;    /* [H] pre-FFN RMSNorm gain                         */
  const void *w_gu;      /* [2F, H]: row 2i = gate_i, row 2i+1 = up_i        */
  const void *w_down;    /* [H, F]                                           */
  const void *w_conv[4]; /* [H/8, H] conv coefficient projections for the
                            sites pre_attn, post_attn, pre_ffn, post_ffn;
                            rows interleaved per 16-channel group g: row 2g
                            = current-tap coefficient of g, row 2g+1 =
                            previous-tap coefficient of g                    */
  const float *b_conv[4];/* [H/8] their biases, interleaved like the rows    */
  /* weight_fp8 only: fp32 per-output-row scales of the matrices above */
  const float *s_qkv;    /* [(nq+2nkv)*d]                                     */
  const float *s_o;      /* [H]                                               */
  const float *s_gu;     /* [2F], interleaved like w_gu                       */
  const float *s_down;   /* [H]                                               */
  const float *s_conv[4];/* [H/8], interleaved like w_conv                   */
  /* weight_fp8 only, optional: the codes' exact bf16 values
   * (dflash_fp8_weights_to_bf16), same layout, scaled by the same s_* rows.
   * When given, a projection whose token tile is 128 tokens or more
   * (tensor-bound: 128+ tokens per launch) uses the copy; smaller launches,
   * bound by the weight stream, use the E4M3 codes.  NULL: codes everywhere.
   * The results are the same either way up to fp32 summation order. */
  const void *w_qkv_bf16;
  const void *w_o_bf16;
  const void *w_gu_bf16;
  const void *w_down_bf16;
  const void *w_conv_bf16[4];
} dflash_layer_weights;

/* Model weights (device pointers, not owned; the layer array is host memory
 * and is copied by dflash_create). */
typedef struct dflash_weights {
  const void *w_fc;      /* [H, n_sel*H_t] context-feature projection        */
  const float *g_fc;     /* [H] its RMSNorm gain (fc_norm)                   */
  const void *embed;     /* [V, H] token embedding shared with the target    */
  const void *lm_head;   /* [V, H] LM head shared with the target            */
  const float *g_final;  /* [H] final RMSNorm gain                           */
  const dflash_layer_weights *layers;   /* host array [n_layers]            */
  const void *sel_e256;  /* [V, sel_dim] selector token embeddings           */
  const void *sel_a;     /* [r, sel_dim] projection of the previous token    */
  const void *sel_b;     /* [r, sel_dim] projection of the current token     */
  const float *sel_w_g;  /* [H] context-gate weights                         */
  float sel_b_g;         /* context-gate bias                                */
  const float *s_fc;     /* weight_fp8 only: [H] row scales of w_fc          */
  const float *s_lm_head;/* weight_fp8 only: [V] row scales of lm_head       */
  const void *w_fc_bf16;    /* weight_fp8 only, optional: bf16 copies (see  */
  const void *lm_head_bf16; /* dflash_layer_weights)                         */
} dflash_weights;

/* Paged drafter KV cache (device memory, not owned, zero-filled when
 * allocated so that slots past a request's length hold finite values).
 *   k_cache: [L][num_pages][nkv][page_size][d] elements of dtype, stored after
 *            the per-head k-norm and RoPE at its absolute position;
 *   v_cache: [L][num_pages][nkv][d][page_size] (each page slice transposed:
 *            the PV product reads it as a K-major operand).
 *   page_table: device int32 [batch][max_pages]; token position p of request
 *   b lives in page page_table[b*max_pages + p/page_size], slot p%page_size.
 *   Entries past a request's last used page are never read.  A page index
 *   outside [0, num_pages) is skipped and reported as DFLASH_ERR_DEVICE. */
typedef struct dflash_kv {
  void *k_cache;
  void *v_cache;
  const int32_t *page_table;
  int num_pages;
  int max_pages;
} dflash_kv;

/* Per-kernel timing record returned by dflash_profile_end. */
typedef struct dflash_kernel_stat {
  char name[32];         /* kernel family                                    */
  int launches;          /* launches recorded                                */
  double ms;             /* summed CUDA-event durations                      */
  double bytes;          /* summed algorithmic HBM bytes (compulsory traffic)*/
  double flops;          /* summed algorithmic flops                         */
} dflash_kernel_stat;

/* Validate the config and weight pointers, record them (no copy of device
 * data), query the device.  Host-only; allocates no device memory. */
DFLASH_API int dflash_create(const dflash_config *cfg, const dflash_weights *w, dflash_ctx **out);
DFLASH_API void dflash_destroy(dflash_ctx *ctx);

/* Bytes of workspace needed for calls with at most max_batch requests and
 * at most max_new_tokens tokens per dflash_inject_context call. */
DFLASH_API size_t dflash_workspace_bytes(const dflash_ctx *ctx, int max_batch, int max_new_tokens);

/* [DF] §2.2 (context-feature and KV-injection bullets; §3 item 2).
 * The target's hidden states from a fixed set of layers, concatenated, are
 * projected to the context feature f = RMSNorm(W_fc x); every drafter layer
 * projects f with its own W_k, W_v; K gets the per-head k-norm and RoPE at
 * its absolute position and both are written into that layer's pages.
 *   target_hidden: device [total_new, n_sel*H_t] (dtype), rows grouped by
 *                  request in order; concat order = ascending layer.
 *   cu_new:        device int32 [batch+1] prefix sums of new tokens per
 *                  request (cu_new[0] = 0, cu_new[batch] = total_new).
 *   ctx_len_in:    device int32 [batch]: tokens already cached; request b's
 *                  new tokens go to positions ctx_len_in[b] ...
 *   ctx_len_out:   device int32 [batch]: receives ctx_len_in + new (may alias
 *                  ctx_len_in).
 *   The caller must have mapped pages for every written position. */
DFLASH_API int dflash_inject_context(dflash_ctx *ctx, const dflash_kv *kv,
                          const void *target_hidden, const int32_t *cu_new, int total_new,
                          const int32_t *ctx_len_in, int32_t *ctx_len_out, int batch,
                          void *workspace, size_t workspace_bytes, dflash_stream_t stream);

/* [DF] §2.2 (parallel block diffusion), §2.3 (anchor; shared embedding and
 * LM head); mask semantics of [FD] Metodologia 1.  For each request b the
 * block is [anchor_ids[b], mask x J] at positions ctx_len[b] .. +J; one
 * forward pass in which every block query attends to all ctx_len[b] cached
 * tokens and to all S block tokens; the J mask positions' logits give the
 * top-16 candidates (value desc, id asc).  The KV cache is only read.
 *   ctx_len:      device int32 [batch], each <= max_pages*page_size.
 *   anchor_ids:   device int32 [batch] in [0, V).
 *   topk_ids:     device int32 [batch][J][16] out.
 *   topk_logits:  device fp32 [batch][J][16] out (raw logits).
 *   final_hidden: device [batch][S][H] (dtype) out, final-normed hidden
 *                 (needed by dflash_select_path's gate); may be NULL.
 *   logits:       device fp32 [batch][J][V] out; may be NULL (then kept in
 *                 the workspace). */
DFLASH_API int dflash_draft_block(dflash_ctx *ctx, const dflash_kv *kv,
                       const int32_t *ctx_len, const int32_t *anchor_ids, int batch,
                       int32_t *topk_ids, float *topk_logits, void *final_hidden, float *logits,
                       void *workspace, size_t workspace_bytes, dflash_stream_t stream);

/* [DF2] Arquitectura 1 (Path Selector) with use_selector: pair scores
 *   s[j][p][c] = z_j[c] + sigmoid(w_g.h_j + b_g) * (A e256[p]).(B e256[c])
 * for j = 1..J, p over position j-1's candidates (the anchor for j = 1,
 * repeated over the 16 rows), c over position j's; then the greedy path
 * (ties to the lower token id).  Without use_selector: draft = top-1.
 *   final_hidden: device [batch][S][H] from dflash_draft_block.
 *   draft_ids:    device int32 [batch][J] out.
 *   pair_scores:  device fp32 [batch][J][16][16] out, or NULL. */
DFLASH_API int dflash_select_path(dflash_ctx *ctx, const int32_t *anchor_ids, const int32_t *topk_ids,
                       const float *topk_logits, const void *final_hidden, int batch,
                       int32_t *draft_ids, float *pair_scores,
                       void *workspace, size_t workspace_bytes, dflash_stream_t stream);

/* [DF2] Flujo de Inferencia 4-5, [BW] Contexto tecnico: k = length of the
 * longest prefix with draft[i] == target[i] (0..J); bonus = target[k];
 * committed = target[0..k] then -1.  Needs no context; block_size = S in
 * 2..16 (else DFLASH_ERR_ARG).
 *   draft_ids: device int32 [batch][J]; target_ids: device int32 [batch][S]
 *   accept_len, bonus: device int32 [batch]; committed: device int32 [batch][S]. */
DFLASH_API int dflash_verify_greedy(const int32_t *draft_ids, const int32_t *target_ids, int batch,
                         int block_size, int32_t *accept_len, int32_t *bonus, int32_t *committed,
                         dflash_stream_t stream);

/* [DF2] Arquitectura del Sistema item 1 (selection "by sampling over these
 * precomputed scores").  Same scores as dflash_select_path (pair scores with
 * use_selector, else every row = the top-16 logits); at position j the draft
 * distribution over the 16 candidates is q_j = softmax(s_j(c_{j-1}, .) / T),
 * c_0 the anchor row, and c_j is the first candidate (in candidate order)
 * whose running probability exceeds uniforms[j] * total.
 *   temperature:  T > 0.
 *   uniforms:     device fp32 [batch][J] in [0, 1) (the caller's random draws).
 *   draft_ids:    device int32 [batch][J] out.
 *   draft_probs:  device fp32 [batch][J][16] out: q_j over the candidates, as
 *                 needed by dflash_verify_rejection.
 *   pair_scores:  device fp32 [batch][J][16][16] out, or NULL. */
DFLASH_API int dflash_sample_path(dflash_ctx *ctx, const int32_t *anchor_ids, const int32_t *topk_ids,
                       const float *topk_logits, const void *final_hidden, int batch, float temperature,
                       const float *uniforms, int32_t *draft_ids, float *draft_probs, float *pair_scores,
                       void *workspace, size_t workspace_bytes, dflash_stream_t stream);

/* [DF2] Arquitectura del Sistema item 1 ("rejection sampling to restore the
 * exact distribution of the target model").  p_i = softmax(target_logits[i]),
 * the target's distributions over the drafted block (one target pass);
 * draft token d_i is accepted while u_accept[i] * q_i(d_i) < p_i(d_i); at the
 * first rejection k the bonus is drawn from max(0, p_k - q_k) (q_k zero
 * outside position k's candidates), after J acceptances from p_J, both by
 * inverse CDF in vocabulary order with u_bonus; committed = d_0..d_{k-1},
 * bonus, then -1.  The committed tokens follow the target's distribution.
 *   target_logits: device fp32 [batch][S][V], V = the context's vocabulary.
 *   draft_ids, topk_ids, draft_probs: from dflash_sample_path / draft_block.
 *   u_accept: device fp32 [batch][J]; u_bonus: device fp32 [batch], in [0, 1).
 *   accept_len, bonus: device int32 [batch]; committed: device int32 [batch][S]. */
DFLASH_API int dflash_verify_rejection(dflash_ctx *ctx, const float *target_logits, const int32_t *draft_ids,
                       const int32_t *topk_ids, const float *draft_probs, const float *u_accept,
                       const float *u_bonus, int batch, int32_t *accept_len, int32_t *bonus,
                       int32_t *committed, void *workspace, size_t workspace_bytes, dflash_stream_t stream);

/* Synchronise `stream`, read the workspace's device status word into
 * *device_status (0 = clean) and clear it.  Returns DFLASH_ERR_TIMEOUT or
 * DFLASH_ERR_DEVICE when a kernel reported one, else DFLASH_OK. */
DFLASH_API int dflash_read_status(const void *workspace, int *device_status, dflash_stream_t stream);

/* Bound on every device-side wait, in nanoseconds (default 2e9). */
DFLASH_API int dflash_set_wait_timeout(dflash_ctx *ctx, unsigned long long ns);

/* Test hook: cap the CTA count of the persistent GEMM (0 = SM count). */
DFLASH_API int dflash_set_gemm_ctas(dflash_ctx *ctx, int ctas);

/* Projections with 256-token tiles (bf16 weights and activations) run on CTA
 * pairs with the 2-SM tensor-core MMA where the launch's plan favours it
 * (on = 1, the default) or always on single CTAs (on = 0): a switch for
 * comparing the two; results are identical up to fp32 summation order.
 * Host-only. */
DFLASH_API int dflash_set_gemm_pairs(dflash_ctx *ctx, int on);
/* bf16 drafters: the LM head selects the top-16 inside its GEMM epilogue
 * (on = 1: per 128-row vocabulary tile the 16 largest keys of each mask row,
 * then one merge; the fp32 logits are written only when dflash_draft_block
 * is given a logits buffer) or writes the fp32 logits and runs the
 * standalone top-16 over them (on = 0, the default: measured faster on
 * GB300 at every batch size this library was benchmarked on).  On applies
 * only where the LM head is bound by its weight stream (at most 32 mask rows
 * per call); larger calls always take the logits path.  The same top-16
 * either way.  Host-only. */
DFLASH_API int dflash_set_fused_topk(dflash_ctx *ctx, int on);

/* Test hook: 2-CTA clusters of the pair GEMM that fit on the current device
 * at once (from the occupancy calculator), or a negative error code. */
DFLASH_API int dflash_debug_gemm_pair_clusters(void);

/* Test hook: the least number of context tokens (a multiple of the page
 * size) the bf16 block attention gives each CTA of its balanced split; 64
 * splits the chunk list as finely as the SM count allows, 0 = automatic. */
DFLASH_API int dflash_set_attn_split(dflash_ctx *ctx, int tokens);

/* Runtime block size ([DF2] table of inference engines: engine flag "runtime
 * block size", example 5; [DF] §3 item 4 and §4 block size: a drafter trained
 * on larger blocks generalises to smaller inference blocks, so the serving
 * engine may pick the block size per step).  block_size in
 * 2..dflash_config.block_size (else DFLASH_ERR_ARG); every later call on the
 * context uses it (S and J = S - 1 in the shapes above).  The workspace from
 * dflash_workspace_bytes fits every runtime block size.  Host-only; must not
 * change while calls on the context are being enqueued from another thread. */
DFLASH_API int dflash_set_block_size(dflash_ctx *ctx, int block_size);
/* The context's current runtime block size (0 for a null context). */
DFLASH_API int dflash_get_block_size(const dflash_ctx *ctx);

/* Per-launch CUDA-event timing of every kernel the next calls launch (on
 * their own streams), aggregated by kernel family.  profile_end
 * synchronises the recorded events. */
DFLASH_API int dflash_profile_begin(dflash_ctx *ctx);
DFLASH_API int dflash_profile_end(dflash_ctx *ctx, dflash_kernel_stat *out, int max_out, int *n_out);

/* Bounded-wait self test: one block spins on *flag (device int32) until it
 * is non-zero or timeout_ns elapses; on timeout it writes
 * DFLASH_ERR_TIMEOUT into the status word of `workspace`.  Used to check the
 * timeout path without any fault. */
DFLASH_API int dflash_debug_wait_flag(const int32_t *flag, unsigned long long timeout_ns,
                           void *workspace, dflash_stream_t stream);

/* Test hook: the library's tcgen05 GEMM on caller buffers, fp32 result
 *   out[m][n] = scale[n] * sum_k X[m][k] * W[n][k]
 * (scale = 1 for bf16 weights), with the same decomposition the drafting
 * calls use (gemm_ctas > 0 forces persistent stream-K over that many single
 * CTAs; gemm_ctas < 0, where the tile is 256 tokens of bf16 weights, forces
 * -gemm_ctas CTA pairs with the 2-SM MMA).
 *   W: device bf16 [N][K], or with w_fp8 E4M3 codes [N][K] and w_scale fp32 [N];
 *   X: device bf16 [M][K]; out: device fp32 [M][N]; K a multiple of 8 (16 with
 *   w_fp8); every pointer 16-byte aligned.
 *   scratch: device buffer of dflash_debug_gemm_scratch_bytes() bytes,
 *   zero-filled once (its first 256 bytes are a status word).  0 if no device. */
DFLASH_API size_t dflash_debug_gemm_scratch_bytes(void);
DFLASH_API int dflash_debug_gemm(const void *W, const float *w_scale, int w_fp8, const void *X, int M, int N, int K,
                      float *out, void *scratch, size_t scratch_bytes, int gemm_ctas, dflash_stream_t stream);

/* Test hook, host only: the decomposition the tensor-core GEMM chooses for
 * one launch of out[M][N] (n_groups weight matrices of N rows sharing the
 * activations X[M][K]; w_fp8: E4M3 weights; split_act: activations as bf16
 * high + low halves; swiglu: the gate/up epilogue), given per_sm CTAs of the
 * chosen variant resident per SM and num_sms SMs (gemm_ctas as for
 * dflash_debug_gemm).  plan (10 values, out): token tile, 128-row weight
 * tiles per group, token tiles, k-blocks per tile, CTAs, cluster split-K
 * width (1 = none), output tiles, (tile, k-block) iterations, then the fp32
 * partial-scratch floats and tile counters a workspace holds for num_sms
 * SMs.  Launches nothing; DFLASH_ERR_ARG on a null plan or a non-positive
 * size. */
DFLASH_API int dflash_debug_gemm_plan(int M, int N, int K, int n_groups, int w_fp8, int split_act, int swiglu,
                                      int per_sm, int num_sms, int gemm_ctas, long long *plan);

/* bf16 copy of an FP8 weight matrix ("Draft quantization", [DF2] engine
 * table): out[n][k] = e4m3(codes[n][k]), every code's value exactly (bf16
 * holds all of them); the row scales stay in the s_* pointers, which the
 * projections apply to the copies as to the codes.  For the optional *_bf16
 * fields of dflash_weights / dflash_layer_weights, made once at set-up.
 * codes: device uint8 [rows][cols], cols a multiple of 4; out: device bf16
 * [rows][cols].  Asynchronous on `stream`. */
DFLASH_API int dflash_fp8_weights_to_bf16(const void *codes, int rows, int cols, void *out, dflash_stream_t stream);

/* Test hook: the FP8 GEMM's own E4M3 -> bf16 weight conversion (the device
 * function its converter warps run) applied to n codes.
 *   codes: device uint8 [n], n > 0 a multiple of 4; out: device bf16 [n]. */
DFLASH_API int dflash_debug_e4m3_to_bf16(const void *codes, int n, void *out, dflash_stream_t stream);

/* Allocation-free top-16, for callers that cannot allocate device memory:
 * e.g. engine plugin hooks that are handed only their input and output
 * buffers and must stay inside a device-memory budget planned in advance,
 * where a cudaMalloc could fail or stall the device.  It computes what the
 * top-16 stage of dflash_draft_block computes (per row of fp32 logits: the
 * 16 largest values, ties to the lower id, sorted) but keeps its scratch in
 * a fixed array inside the library (4 MB + 4 KB per GPU that loads it, held
 * until the process exits) instead of a caller workspace.  No counterpart in
 * the paper: it is an interface convenience, not part of the method.
 *   logits:      device fp32 [rows][vocab];
 *   topk_ids:    device int32 [rows][16] out; topk_logits: device fp32 [rows][16] out.
 *   rows <= 1024, else DFLASH_ERR_SHAPE (nothing launched).
 * Allocates nothing (no cudaMalloc / cudaFree).  The first call on each
 * device looks up the array's device address and keeps it; make that first
 * call before any stream capture.  The kept address belongs to the device's
 * current CUDA context: after cudaDeviceReset (a new context) it is stale,
 * so a process that resets a device must not call this entry point on that
 * device again.  All calls share the array and clear its counters at the
 * start of each call: calls that overlap on the GPU race. */
DFLASH_API int dflash_topk16_noalloc(const float *logits, int rows, int vocab, int32_t *topk_ids,
                                     float *topk_logits, dflash_stream_t stream);

/* Message for the last non-zero return on this thread. */
DFLASH_API const char *dflash_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */

// Host-side interfaces shared by the translation units of libdflash.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/dflash.h"

namespace dflash {

// GEMM epilogues: out[m][n] = epi(sum_k X[m][k] * W[n][k])
enum Epi : int {
  EPI_BF16 = 0,       // out (bf16)  = acc      (+ out_lo = bf16(acc - out) when given)
  EPI_F32 = 1,        // out (fp32)  = acc
  EPI_ADD_F32 = 2,    // out (fp32) += acc          (residual stream)
  EPI_SWIGLU = 3,     // rows 2i / 2i+1 = gate_i / up_i: out[m][i] = silu(gate) * up (+ out_lo)
  EPI_TANH_BIAS = 4,  // out (fp32)  = tanh(acc + bias[n])   (conv coefficients)
  EPI_STORE_T = 5,    // out (activation dtype) = acc (+ out_lo on the bf16 path)
  EPI_F32_SPLIT = 6,  // out (fp32) = acc, out2 / out2_lo = bf16 hi / lo halves of acc
  // LM head with its top-16 selection: the 16 largest (value, id) keys of
  // each token over each 128-row vocabulary tile -> cand[token][tile][16]
  // (64-bit keys, value descending, id ascending); out (fp32 logits) too
  // when given
  EPI_TOPK = 7
};

// One projection.  Activations may come as two bf16 tensors X (high half)
// and X_lo (low half, X + X_lo ~ the fp32 value): the kernel then issues a
// second MMA per k-step on the same weight tile.
struct GemmOp {
  const void *W = nullptr;
  int ldw = 0;
  const void *X = nullptr;
  const void *X_lo = nullptr;
  int ldx = 0;
  int M = 0, N = 0, K = 0;
  int epi = EPI_F32;
  void *out = nullptr;
  int ldo = 0;
  void *out_lo = nullptr;
  void *out2 = nullptr, *out2_lo = nullptr;
  int ldo2 = 0;
  const float *bias = nullptr;
  uint64_t *cand = nullptr;   // EPI_TOPK: [M][cand_ld][16] keys
  int cand_ld = 0;            // EPI_TOPK: vocabulary tiles per token row
  const char *name = "gemm";
  // grouped launch: n_groups weight matrices Wg[g] of the same shape applied
  // to the same activations, output g at out + g * out_gstride elements
  int n_groups = 1;
  const void *Wg[16] = {};
  size_t out_gstride = 0;
  // FP8 weights: W / Wg hold E4M3 codes (ldw in bytes = elements); row n of
  // the result is scaled by wscale[n] (grouped: wscale_g[g][n])
  bool w_fp8 = false;
  const float *wscale = nullptr;
  const float *wscale_g[16] = {};
};

// Per-launch timing of kernel families (dflash_profile_begin / _end).
struct Profiler {
  struct Rec {
    const char *name;
    cudaEvent_t a, b;
    double bytes, flops;
  };
  bool on = false;
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  cudaEvent_t take();
  void reset();
  ~Profiler();
};

struct Launch {
  cudaStream_t stream = nullptr;
  int num_sms = 148;
  int *status = nullptr;                 // device status word
  unsigned long long timeout_ns = 2000000000ull;
  int gemm_ctas = 0;                     // 0 = SM count; < 0: that many CTA pairs (test hook)
  int gemm_pairs = 1;                    // 256-token tiles on CTA pairs (2-SM MMA) where that pays
  Profiler *prof = nullptr;
};

// RAII: records CUDA events around the launches in its scope when profiling.
struct ProfScope {
  const Launch &lc;
  int idx = -1;
  ProfScope(const Launch &l, const char *name, double bytes, double flops);
  ~ProfScope();
};

struct GemmScratch {
  float *partials = nullptr;   // [ctas][2][128 * 256] fp32
  size_t partial_floats = 0;
  int *counters = nullptr;     // one per output tile, zero between launches
  int n_counters = 0;
};

int set_error(int code, const char *fmt, ...);
int cuda_check(cudaError_t e, const char *what);

// The FP8 GEMM's E4M3 -> bf16 conversion over n codes (test hook).
int e4m3_to_bf16(const Launch &lc, const void *codes, int n, void *out);
// 2-CTA clusters of the pair GEMM resident at once on the current device (< 0: error).
int gemm_pair_clusters();
// Exact bf16 values of n E4M3 weight codes (the row scales stay apart).
int fp8_rows_to_bf16(const Launch &lc, const void *codes, long long n, void *out);

// TMA descriptor of a row-major 2-D tensor [rows][cols] (128-byte swizzle
// unless told otherwise); box = box_cols x box_rows.
int make_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elt_bytes, uint64_t cols,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// Decomposition of one tensor-core GEMM launch (host arithmetic only).
struct GemmPlan {
  int BN;              // token tile (UMMA N)
  int rtpg;            // 128-row weight tiles per group
  int tok_tiles;       // token tiles
  int kbpt;            // k-blocks (ring stages) per tile
  int G;               // CTAs launched
  int csk;             // > 1: cluster split-K, csk CTAs per tile
  long long tiles;     // output tiles over all groups
  long long total;     // tiles * kbpt
};
int gemm_token_tile(int M, bool split, bool f8);
// per_sm: CTAs of the chosen variant resident per SM; gemm_ctas > 0 forces
// that many stream-K CTAs (test hook).
GemmPlan gemm_plan(int M, int N, int K, int n_groups, bool f8, bool split, bool swiglu, int per_sm, int num_sms,
                   int gemm_ctas);

// bf16 operands on tcgen05 tensor cores.
int gemm_bf16(const Launch &lc, const GemmOp &op, const GemmScratch &sc);
// fp32 operands on CUDA cores (tiny fp32 configurations).
int gemm_f32(const Launch &lc, const GemmOp &op);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  const void *q;            // [B*16][nq*d] (dtype)
  const void *k_cache;      // this layer: [num_pages][nkv][page][d]
  const void *v_cache;
  const void *bk, *bv;      // block K [B][nkv][64][d], block V^T [B][nkv][d][64]
  const int32_t *page_table;
  int max_pages, num_pages, page_size;
  const int32_t *ctx_len;   // [B]
  void *out;                // [B*16][nq*d] (dtype)
  void *out_lo;             // low bf16 halves of out, or null
  int B, nq, nkv, d;
  int S;                    // block size (queries per request, block keys), 2..16
  int min_chunks;           // bf16: at least this many 64-token chunks per CTA (0 = default)
  int *counters;            // bf16: [counter_cap] ints, zero between launches (self-resetting)
  size_t counter_cap;       // >= B * nkv
  float *partials;          // bf16: [partial_slots][ATTN_PART_FLOATS] merge scratch
  size_t partial_slots;     // >= 2 * SM count
};
// one split partial of the bf16 attention: O [128 rows][128 d] (row-major), max [128], sum [128]
constexpr int ATTN_PART_FLOATS = 128 * 128 + 2 * 128;
int attention_bf16(const Launch &lc, const AttnArgs &a);
int attention_f32(const Launch &lc, const AttnArgs &a);

// ---------------------------------------------------------------- elementwise
// *_lo outputs: low bf16 halves (value - high half) for split activations;
// null to skip (always null on the fp32 path).
// S = block size (anchor + S-1 mask positions), 2..16
int embed_rmsnorm(const Launch &lc, bool f32, const void *embed, const int32_t *anchor, int mask_id, int vocab,
                  const float *gain, float eps, int B, int S, int H, float *x, void *u, void *u_lo);
// conv_y32 / conv_coef (both or neither): a post-sublayer DFlash-2 short conv
// added into x first (x written back), see rmsnorm_kernel
int rmsnorm_rows(const Launch &lc, bool f32, float *x, int rows, int H, int S, const float *gain, float eps,
                 void *out, void *out_lo, void *out_mask_rows, void *out_mask_lo, const float *conv_y32 = nullptr,
                 const float *conv_coef = nullptr);
int feature_norm(const Launch &lc, bool f32, const float *in, int rows, int H, const float *gain, float eps,
                 bool apply_norm, void *out, void *out_lo, const int32_t *ctx_len_in, int32_t *ctx_len_saved, int B);
int qk_norm_rope(const Launch &lc, bool f32, const float *qkv, int B, int S, int nq, int nkv, int d,
                 const float *g_q, const float *g_k, bool qk_norm, float eps, float rope_base,
                 const int32_t *ctx_len, void *q_out, void *bk, void *bv);
int inject_scatter(const Launch &lc, bool f32, const float *kvproj, int T, int L, int nkv, int d,
                   const float *const *g_k, bool qk_norm, float eps, float rope_base, const int32_t *cu_new,
                   int B, const int32_t *ctx_len_saved, int32_t *ctx_len_out, const dflash_kv &kv,
                   size_t layer_elems);
// y: activation (hi [+ y_lo]) or y32 (fp32); pre sites write out_t (+ out_lo),
// post sites add into x_add.
int conv_apply(const Launch &lc, bool f32, const void *y, const void *y_lo, const float *y32, const float *coef,
               int B, int S, int H, void *out_t, void *out_lo, float *x_add);

// ---------------------------------------------------------------- top-k / select / verify
// J = block size - 1 mask positions per request; S = J + 1 target rows.
int sample_path(const Launch &lc, const float *scores, const float *topk_logits, const int32_t *topk_ids, int B,
                int J, float temperature, const float *uniforms, int32_t *draft, float *qprob);
int verify_rejection_scratch_floats(int B, int S);
int verify_rejection(const Launch &lc, const float *target_logits, int V, float *scratch, const int32_t *draft,
                     const int32_t *topk_ids, const float *qprob, const float *u_accept, const float *u_bonus, int B,
                     int J, int32_t *accept, int32_t *bonus, int32_t *committed);
int topk16(const Launch &lc, const float *logits, int rows, int V, int32_t *ids, float *vals,
           uint64_t *part_keys, int *counters, int max_chunks);
// The top-16 of each row from the LM head's per-tile candidates (EPI_TOPK):
// cand [rows][tiles][16] keys -> ids / vals [rows][16].
int topk16_merge(const Launch &lc, const uint64_t *cand, int rows, int tiles, int32_t *ids, float *vals,
                 uint64_t *part_keys, int *counters, int max_chunks);
int pair_scores(const Launch &lc, bool f32, const int32_t *anchor, const int32_t *topk_ids,
                const float *topk_logits, const void *final_hidden, int B, int J, int H, const void *e256,
                const void *sel_a, const void *sel_b, int r, int E, const float *w_g, float b_g, float *scores);
int greedy_path(const Launch &lc, const float *scores, const int32_t *topk_ids, int B, int J, bool use_scores,
                int32_t *draft);
int verify(const Launch &lc, const int32_t *draft, const int32_t *target, int B, int J, int32_t *accept,
           int32_t *bonus, int32_t *committed);
int wait_flag(const Launch &lc, const int32_t *flag);

}  // namespace dflash

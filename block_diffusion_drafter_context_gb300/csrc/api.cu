// C ABI of libdflash: argument validation, workspace layout, and the launch
// sequence of each call of the drafting hot path (see include/dflash.h).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

struct dflash_ctx {
  dflash_config cfg;
  dflash_weights w;
  std::vector<dflash_layer_weights> layers;
  int device = 0;
  int num_sms = 148;
  unsigned long long timeout_ns = 2000000000ull;
  int gemm_ctas = 0;
  int gemm_pairs = 1;
  int fused_topk = 0;      // bf16: LM head with its top-16 epilogue (no logits round trip)
  int attn_split = 0;
  int block = 16;   // runtime block size S (2..cfg.block_size)
  dflash::Profiler prof;
};

namespace dflash {

static thread_local std::string g_err;

int set_error(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_check(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return DFLASH_OK;
  return set_error(DFLASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int elt_bytes, uint64_t cols,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return set_error(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (reinterpret_cast<uintptr_t>(base) & 15 || row_stride_bytes % 16)
    return set_error(DFLASH_ERR_ALIGN, "TMA operand base / row stride must be 16-byte aligned");
  (void)elt_bytes;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %llux%llu tensor", static_cast<int>(r),
                     static_cast<unsigned long long>(rows), static_cast<unsigned long long>(cols));
  return DFLASH_OK;
}

// ------------------------------------------------------------------ profiler
cudaEvent_t Profiler::take() {
  if (used < pool.size()) return pool[used++];
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  pool.push_back(e);
  ++used;
  return e;
}
void Profiler::reset() {
  recs.clear();
  used = 0;
}
Profiler::~Profiler() {
  for (auto e : pool) cudaEventDestroy(e);
}

// Inside a stream capture the records must be external event nodes, so that
// replaying the graph stamps the events.
static void record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

ProfScope::ProfScope(const Launch &l, const char *name, double bytes, double flops) : lc(l) {
  if (!lc.prof || !lc.prof->on) return;
  Profiler::Rec r;
  r.name = name;
  r.a = lc.prof->take();
  r.b = lc.prof->take();
  r.bytes = bytes;
  r.flops = flops;
  record(r.a, lc.stream);
  lc.prof->recs.push_back(r);
  idx = static_cast<int>(lc.prof->recs.size()) - 1;
}
ProfScope::~ProfScope() {
  if (idx >= 0) record(lc.prof->recs[idx].b, lc.stream);
}

// ------------------------------------------------------------------ workspace layout
namespace {

constexpr int GEMM_COUNTERS = 1 << 16;
constexpr int GEMM_MAX_BN = 256;
constexpr int TOPK_MAX_CHUNKS = 64;

// The header of the workspace (status word, self-resetting counters, split
// scratch) sits at offsets that depend on neither the batch nor the token
// count, so calls with different sizes on one workspace never read another
// call's data as a counter.  Everything after it is rewritten before it is
// read within each call.
struct Layout {
  size_t status, gemm_ctr, gemm_part, topk_ctr, attn_ctr, attn_part, attn_part_slots, topk_part;
  size_t x, u, u2, qkv, q, bk, bv, o, ysub, coef, hmid, hmask, hfinal, logits, scores, lse;
  size_t u_lo, u2_lo, o_lo, ysub_lo, hmid_lo, hmask_lo, ysub32;
  size_t fc, f, f_lo, kvproj, ctx_saved, cand;
  size_t total;
  size_t gemm_part_floats;
};

// Byte offsets of every workspace buffer for batch B, Tn injected tokens and
// block size S (default: the context's runtime block size).
Layout layout(const dflash_ctx *c, int B, int Tn, int S_ = 0) {
  const dflash_config &g = c->cfg;
  const size_t te = g.dtype == DFLASH_F32 ? 4 : 2;
  const size_t H = g.hidden, d = g.head_dim, nq = g.n_q_heads, nkv = g.n_kv_heads, F = g.ffn, V = g.vocab;
  const size_t S = S_ > 0 ? S_ : c->block, J = S - 1;   // positions per request, mask positions
  const size_t R = static_cast<size_t>(B) * S;
  Layout L = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  };
  L.status = take(256);
  L.gemm_ctr = take(sizeof(int) * GEMM_COUNTERS);
  L.gemm_part_floats = static_cast<size_t>(c->num_sms) * 2 * 128 * GEMM_MAX_BN;
  L.gemm_part = take(4 * L.gemm_part_floats);
  L.topk_ctr = take(sizeof(int) * static_cast<size_t>(DFLASH_MAX_BATCH) * 15);
  L.attn_ctr = take(sizeof(int) * static_cast<size_t>(DFLASH_MAX_BATCH) * nkv);
  L.attn_part_slots = 2ull * c->num_sms;
  L.attn_part = take(4ull * L.attn_part_slots * ATTN_PART_FLOATS);
  (void)B;
  L.topk_part = take(8ull * B * J * TOPK_MAX_CHUNKS * 16);
  L.x = take(4 * R * H);
  L.u = take(te * R * H);
  L.u2 = take(te * R * H);
  L.qkv = take(4 * R * (nq + 2 * nkv) * d);
  L.q = take(te * R * nq * d);
  L.bk = take(te * B * nkv * 64 * d);   // block K [B][nkv][64][d], rows S.. unused
  L.bv = take(te * B * nkv * 64 * d);   // block V^T [B][nkv][d][64], cols S.. unused
  L.o = take(te * R * nq * d);
  L.ysub = take(te * R * H);
  L.coef = take(4 * R * (H / 8));
  L.hmid = take(te * R * F);
  L.hmask = take(te * B * J * H);
  // low halves of the GEMM activations (split activations, bf16 path)
  const size_t tl = (g.dtype == DFLASH_F32 || !g.split_act) ? 0 : 2;
  L.u_lo = take(tl * R * H);
  L.u2_lo = take(tl * R * H);
  L.o_lo = take(tl * R * nq * d);
  L.ysub_lo = take(tl * R * H);
  L.hmid_lo = take(tl * R * F);
  L.hmask_lo = take(tl * B * J * H);
  L.ysub32 = take(4 * R * H);
  L.hfinal = take(te * R * H);
  L.logits = take(4ull * B * J * V);
  L.scores = take(4ull * B * J * 256);
  L.lse = take(4ull * verify_rejection_scratch_floats(B, static_cast<int>(S)));   // rejection verification scratch
  L.fc = take(4ull * Tn * H);
  L.f = take(te * Tn * H);
  L.f_lo = take(tl * Tn * H);
  L.kvproj = take(4ull * g.n_layers * Tn * 2 * nkv * d);
  L.ctx_saved = take(sizeof(int) * static_cast<size_t>(B));
  // the LM head's top-16 candidates: 16 keys per mask row per 128-row vocabulary tile
  L.cand = take(8ull * B * J * ((V + 127) / 128) * 16);
  L.total = off;
  return L;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

Launch make_launch(dflash_ctx *c, void *ws, cudaStream_t s) {
  Launch lc;
  lc.stream = s;
  lc.num_sms = c->num_sms;
  lc.status = ws ? at<int>(ws, 0) : nullptr;
  lc.timeout_ns = c->timeout_ns;
  lc.gemm_ctas = c->gemm_ctas;
  lc.gemm_pairs = c->gemm_pairs;
  lc.prof = &c->prof;
  return lc;
}

// One projection of the drafter on the path's GEMM (tcgen05 for bf16, CUDA
// cores for fp32).
int proj(dflash_ctx *c, const Launch &lc, void *ws, const Layout &L, const GemmOp &op) {
  if (c->cfg.dtype == DFLASH_F32) return gemm_f32(lc, op);
  GemmScratch sc;
  sc.partials = at<float>(ws, L.gemm_part);
  sc.partial_floats = L.gemm_part_floats;
  sc.counters = at<int>(ws, L.gemm_ctr);
  sc.n_counters = GEMM_COUNTERS;
  return gemm_bf16(lc, op, sc);
}

GemmOp mk(const void *W, int ldw, const void *X, const void *X_lo, int ldx, int M, int N, int K, int epi, void *out,
          int ldo, const char *name) {
  GemmOp o;
  o.W = W;
  o.ldw = ldw;
  o.X = X;
  o.X_lo = X_lo;
  o.ldx = ldx;
  o.M = M;
  o.N = N;
  o.K = K;
  o.epi = epi;
  o.out = out;
  o.ldo = ldo;
  o.name = name;
  return o;
}

// The weight of a GEMM: bf16 matrix, or (weight_fp8) E4M3 codes with their
// row scales - unless a bf16 copy of the matrix is given and the launch is
// tensor-bound (token tile of 128 or more: the FP8 tiles stop at 128 tokens,
// where the weight stream no longer bounds the launch and the conversion
// only costs), which then takes the copy.
GemmOp wq(const dflash_ctx *c, GemmOp op, const float *scale, const void *bf16_copy = nullptr) {
  if (c->cfg.weight_fp8) {
    const bool split = op.X_lo != nullptr;
    if (bf16_copy && gemm_token_tile(op.M, split, false) >= 128) {
      op.W = bf16_copy;        // exact code values; the row scales apply in the epilogue
      op.wscale = scale;
      return op;
    }
    op.w_fp8 = true;
    op.wscale = scale;
  }
  return op;
}

int check_ws(const dflash_ctx *c, void *ws, size_t bytes, int B, int Tn) {
  if (!ws) return set_error(DFLASH_ERR_ARG, "workspace is null");
  if (!aligned16(ws)) return set_error(DFLASH_ERR_ALIGN, "workspace must be 16-byte aligned");
  if (B > DFLASH_MAX_BATCH) return set_error(DFLASH_ERR_ARG, "batch %d over DFLASH_MAX_BATCH", B);
  const size_t need = layout(c, B, Tn).total;
  if (bytes < need)
    return set_error(DFLASH_ERR_SHAPE, "workspace of %zu bytes is smaller than the %zu needed for batch %d", bytes, need,
                     B);
  return DFLASH_OK;
}

int check_kv(const dflash_ctx *c, const dflash_kv *kv) {
  if (!kv || !kv->k_cache || !kv->v_cache || !kv->page_table) return set_error(DFLASH_ERR_ARG, "null KV cache");
  if (kv->num_pages <= 0 || kv->max_pages <= 0) return set_error(DFLASH_ERR_SHAPE, "empty KV page pool");
  if (!aligned16(kv->k_cache) || !aligned16(kv->v_cache)) return set_error(DFLASH_ERR_ALIGN, "KV cache not aligned");
  (void)c;
  return DFLASH_OK;
}

size_t layer_elems(const dflash_ctx *c, const dflash_kv *kv) {
  return static_cast<size_t>(kv->num_pages) * c->cfg.n_kv_heads * c->cfg.page_size * c->cfg.head_dim;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

// ====================================================================== C ABI
extern "C" {

const char *dflash_last_error(void) { return g_err.c_str(); }

int dflash_create(const dflash_config *cfg, const dflash_weights *w, dflash_ctx **out) {
  if (!cfg || !w || !out) return set_error(DFLASH_ERR_ARG, "dflash_create: null argument");
  *out = nullptr;
  const dflash_config &g = *cfg;
  if (g.dtype != DFLASH_BF16 && g.dtype != DFLASH_F32) return set_error(DFLASH_ERR_ARG, "dtype must be bf16 or fp32");
  if (g.block_size < 2 || g.block_size > 16 || g.top_k != 16 || g.page_size != 64)
    return set_error(DFLASH_ERR_UNSUPPORTED, "block_size must be 2..16, top_k 16, page_size 64");
  if (g.hidden <= 0 || g.hidden % 16 || g.n_layers < 1 || g.n_layers > 16 || g.n_q_heads <= 0 || g.n_kv_heads <= 0 ||
      g.n_q_heads % g.n_kv_heads || g.ffn <= 0 || g.ffn % 8 || g.vocab < 16 || g.target_hidden <= 0 ||
      g.n_target_layers <= 0 || (g.n_target_layers * g.target_hidden) % 8)
    return set_error(DFLASH_ERR_SHAPE, "inconsistent drafter shape");
  if (g.dtype == DFLASH_BF16 && (g.head_dim != 128 || g.n_q_heads / g.n_kv_heads > 8))
    return set_error(DFLASH_ERR_UNSUPPORTED, "bf16 path: head_dim must be 128 and q heads per kv head <= 8");
  if (g.dtype == DFLASH_F32 && g.head_dim != 64 && g.head_dim != 128)
    return set_error(DFLASH_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (g.mask_id < 0 || g.mask_id >= g.vocab) return set_error(DFLASH_ERR_ARG, "mask_id outside the vocabulary");
  if (g.use_selector && (g.sel_rank < 1 || g.sel_rank > 64 || g.sel_dim < 1 || g.sel_dim > 1024))
    return set_error(DFLASH_ERR_UNSUPPORTED, "selector rank must be 1..64 and width 1..1024");
  if (!(g.eps >= 0.f) || !(g.rope_base > 1.f)) return set_error(DFLASH_ERR_ARG, "eps / rope_base out of range");
  const bool f8 = g.weight_fp8 != 0;
  if (f8 && g.dtype != DFLASH_BF16) return set_error(DFLASH_ERR_UNSUPPORTED, "FP8 weights need the bf16 path");
  // FP8 code rows are K bytes: every GEMM's K a multiple of 16
  if (f8 && (g.ffn % 16 || (g.n_target_layers * g.target_hidden) % 16))
    return set_error(DFLASH_ERR_SHAPE, "FP8 weights: ffn and n_sel * H_t must be multiples of 16");
  auto scale_ok = [](const float *s) { return s && (reinterpret_cast<uintptr_t>(s) & 3) == 0; };
  if (f8 && (!scale_ok(w->s_fc) || !scale_ok(w->s_lm_head)))
    return set_error(DFLASH_ERR_ARG, "FP8 weights: s_fc / s_lm_head missing");
  const void *req[] = {w->w_fc, w->embed, w->lm_head, w->g_final};
  for (const void *p : req)
    if (!p || !aligned16(p)) return set_error(DFLASH_ERR_ALIGN, "model weight missing or not 16-byte aligned");
  if (g.fc_norm && !w->g_fc) return set_error(DFLASH_ERR_ARG, "fc_norm needs g_fc");
  if (!w->layers) return set_error(DFLASH_ERR_ARG, "null layer array");
  for (int l = 0; l < g.n_layers; ++l) {
    const dflash_layer_weights &lw = w->layers[l];
    const void *lp[] = {lw.g_attn, lw.w_qkv, lw.w_o, lw.g_ffn, lw.w_gu, lw.w_down};
    for (const void *p : lp)
      if (!p || !aligned16(p)) return set_error(DFLASH_ERR_ALIGN, "layer %d weight missing or misaligned", l);
    if (g.qk_norm && (!lw.g_q || !lw.g_k)) return set_error(DFLASH_ERR_ARG, "layer %d: qk_norm needs g_q, g_k", l);
    if (g.use_conv)
      for (int s = 0; s < 4; ++s)
        if (!lw.w_conv[s] || !lw.b_conv[s] || !aligned16(lw.w_conv[s]) || (f8 && !scale_ok(lw.s_conv[s])))
          return set_error(DFLASH_ERR_ARG, "layer %d: conv site %d weights missing", l, s);
    if (f8 && (!scale_ok(lw.s_qkv) || !scale_ok(lw.s_o) || !scale_ok(lw.s_gu) || !scale_ok(lw.s_down)))
      return set_error(DFLASH_ERR_ARG, "layer %d: FP8 row scales missing", l);
  }
  if (g.use_selector && (!w->sel_e256 || !w->sel_a || !w->sel_b || !w->sel_w_g))
    return set_error(DFLASH_ERR_ARG, "selector weights missing");
  dflash_ctx *c = new dflash_ctx();
  c->cfg = g;
  c->block = g.block_size;
  c->w = *w;
  c->layers.assign(w->layers, w->layers + g.n_layers);
  c->w.layers = c->layers.data();
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return set_error(DFLASH_ERR_CUDA, "no CUDA device");
  }
  *out = c;
  return DFLASH_OK;
}

void dflash_destroy(dflash_ctx *ctx) { delete ctx; }

size_t dflash_workspace_bytes(const dflash_ctx *ctx, int max_batch, int max_new_tokens) {
  if (!ctx || max_batch < 0 || max_new_tokens < 0) return 0;
  // sized for the largest block the context can run, so that any runtime block size fits
  return layout(ctx, max_batch < 1 ? 1 : max_batch, max_new_tokens, ctx->cfg.block_size).total;
}

int dflash_set_wait_timeout(dflash_ctx *ctx, unsigned long long ns) {
  if (!ctx || ns == 0) return set_error(DFLASH_ERR_ARG, "bad timeout");
  ctx->timeout_ns = ns;
  return DFLASH_OK;
}

int dflash_set_gemm_ctas(dflash_ctx *ctx, int ctas) {
  if (!ctx || ctas < 0) return set_error(DFLASH_ERR_ARG, "bad CTA count");
  ctx->gemm_ctas = ctas > ctx->num_sms ? ctx->num_sms : ctas;
  return DFLASH_OK;
}

int dflash_set_fused_topk(dflash_ctx *ctx, int on) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  ctx->fused_topk = on != 0;
  return DFLASH_OK;
}

int dflash_set_gemm_pairs(dflash_ctx *ctx, int on) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  ctx->gemm_pairs = on != 0;
  return DFLASH_OK;
}

int dflash_set_block_size(dflash_ctx *ctx, int block_size) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  if (block_size < 2 || block_size > ctx->cfg.block_size)
    return set_error(DFLASH_ERR_ARG, "runtime block size must be 2..%d", ctx->cfg.block_size);
  ctx->block = block_size;
  return DFLASH_OK;
}

int dflash_get_block_size(const dflash_ctx *ctx) { return ctx ? ctx->block : 0; }

int dflash_set_attn_split(dflash_ctx *ctx, int tokens) {
  if (!ctx || tokens < 0 || tokens % 64) return set_error(DFLASH_ERR_ARG, "split must be a multiple of 64");
  ctx->attn_split = tokens;
  return DFLASH_OK;
}

int dflash_inject_context(dflash_ctx *ctx, const dflash_kv *kv, const void *target_hidden, const int32_t *cu_new,
                          int total_new, const int32_t *ctx_len_in, int32_t *ctx_len_out, int batch, void *workspace,
                          size_t workspace_bytes, dflash_stream_t stream) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  if (batch < 0 || total_new < 0) return set_error(DFLASH_ERR_ARG, "negative batch / token count");
  if (batch == 0 || total_new == 0) return DFLASH_OK;
  if (!target_hidden || !cu_new || !ctx_len_in || !ctx_len_out)
    return set_error(DFLASH_ERR_ARG, "dflash_inject_context: null argument");
  if (!aligned16(target_hidden)) return set_error(DFLASH_ERR_ALIGN, "target_hidden must be 16-byte aligned");
  if (int e = check_kv(ctx, kv)) return e;
  if (int e = check_ws(ctx, workspace, workspace_bytes, batch, total_new)) return e;
  const dflash_config &g = ctx->cfg;
  const bool f32 = g.dtype == DFLASH_F32;
  const Layout L = layout(ctx, batch, total_new);
  Launch lc = make_launch(ctx, workspace, reinterpret_cast<cudaStream_t>(stream));
  const int H = g.hidden, d = g.head_dim, nq = g.n_q_heads, nkv = g.n_kv_heads, K = g.n_target_layers * g.target_hidden;
  const size_t te = f32 ? 4 : 2;
  const bool split = !f32 && g.split_act;
  void *f_lo = split ? at<void>(workspace, L.f_lo) : nullptr;
  // context feature: fc projection, then RMSNorm
  if (int e = proj(ctx, lc, workspace, L,
                   wq(ctx, mk(ctx->w.w_fc, K, target_hidden, nullptr, K, total_new, H, K, EPI_F32,
                              at<float>(workspace, L.fc), H, "fc"),
                      ctx->w.s_fc, ctx->w.w_fc_bf16)))
    return e;
  if (int e = feature_norm(lc, f32, at<float>(workspace, L.fc), total_new, H, ctx->w.g_fc, g.eps, g.fc_norm != 0,
                           at<void>(workspace, L.f), f_lo, ctx_len_in, at<int32_t>(workspace, L.ctx_saved), batch))
    return e;
  // every layer's own K/V projection of the feature (rows nq*d.. of w_qkv);
  // on tensor cores all layers share one grouped launch
  std::vector<const float *> gk(g.n_layers);
  GemmOp kvop = mk(nullptr, H, at<void>(workspace, L.f), f_lo, H, total_new, 2 * nkv * d, H, EPI_F32,
                   at<float>(workspace, L.kvproj), 2 * nkv * d, "kv_inject");
  kvop.out_gstride = static_cast<size_t>(total_new) * 2 * nkv * d;
  // FP8 codes, or the layers' bf16 copies for a tensor-bound launch (as wq)
  bool copies = g.weight_fp8 != 0 && gemm_token_tile(total_new, split, false) >= 128;
  for (int l = 0; l < g.n_layers; ++l) copies = copies && ctx->layers[l].w_qkv_bf16;
  kvop.w_fp8 = g.weight_fp8 != 0 && !copies;
  const size_t tw = kvop.w_fp8 ? 1 : 2;   // bytes per weight element (fp32 path: te)
  for (int l = 0; l < g.n_layers; ++l) {
    const dflash_layer_weights &lw = ctx->layers[l];
    const void *wl = copies ? lw.w_qkv_bf16 : lw.w_qkv;
    kvop.Wg[l] = static_cast<const char *>(wl) + (f32 ? te : tw) * static_cast<size_t>(nq) * d * H;
    if (g.weight_fp8) kvop.wscale_g[l] = lw.s_qkv + static_cast<size_t>(nq) * d;   // codes or their exact copies
    gk[l] = lw.g_k;
  }
  if (!f32 && (2 * nkv * d) % 128 == 0 && g.n_layers > 1) {
    kvop.n_groups = g.n_layers;
    if (int e = proj(ctx, lc, workspace, L, kvop)) return e;
  } else {
    for (int l = 0; l < g.n_layers; ++l) {
      GemmOp one = kvop;
      one.n_groups = 1;
      one.W = kvop.Wg[l];
      one.wscale = kvop.wscale_g[l];
      one.out = at<float>(workspace, L.kvproj) + l * kvop.out_gstride;
      if (int e = proj(ctx, lc, workspace, L, one)) return e;
    }
  }
  return inject_scatter(lc, f32, at<float>(workspace, L.kvproj), total_new, g.n_layers, nkv, d, gk.data(),
                        g.qk_norm != 0, g.eps, g.rope_base, cu_new, batch, at<int32_t>(workspace, L.ctx_saved),
                        ctx_len_out, *kv, layer_elems(ctx, kv));
}

int dflash_draft_block(dflash_ctx *ctx, const dflash_kv *kv, const int32_t *ctx_len, const int32_t *anchor_ids,
                       int batch, int32_t *topk_ids, float *topk_logits, void *final_hidden, float *logits,
                       void *workspace, size_t workspace_bytes, dflash_stream_t stream) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  if (batch < 0) return set_error(DFLASH_ERR_ARG, "negative batch");
  if (batch == 0) return DFLASH_OK;
  if (!ctx_len || !anchor_ids || !topk_ids || !topk_logits)
    return set_error(DFLASH_ERR_ARG, "dflash_draft_block: null argument");
  if (final_hidden && !aligned16(final_hidden)) return set_error(DFLASH_ERR_ALIGN, "final_hidden not aligned");
  if (int e = check_kv(ctx, kv)) return e;
  if (int e = check_ws(ctx, workspace, workspace_bytes, batch, 0)) return e;
  const dflash_config &g = ctx->cfg;
  const bool f32 = g.dtype == DFLASH_F32;
  const Layout L = layout(ctx, batch, 0);
  Launch lc = make_launch(ctx, workspace, reinterpret_cast<cudaStream_t>(stream));
  void *ws = workspace;
  const int S = ctx->block, J = S - 1;
  const int B = batch, R = B * S, H = g.hidden, d = g.head_dim, nq = g.n_q_heads, nkv = g.n_kv_heads;
  const int F = g.ffn, V = g.vocab, nh = nq + 2 * nkv, G8 = H / 8;
  float *x = at<float>(ws, L.x);
  void *u = at<void>(ws, L.u), *u2 = at<void>(ws, L.u2), *ysub = at<void>(ws, L.ysub);
  float *coef = at<float>(ws, L.coef);
  void *hfinal = final_hidden ? final_hidden : at<void>(ws, L.hfinal);
  float *lg = logits ? logits : at<float>(ws, L.logits);

  const bool split = !f32 && g.split_act;
  auto lo = [&](size_t off) -> void * { return split ? at<void>(ws, off) : nullptr; };
  void *u_lo = lo(L.u_lo), *u2_lo = lo(L.u2_lo), *ysub_lo = lo(L.ysub_lo), *hmid_lo = lo(L.hmid_lo);
  float *ysub32 = at<float>(ws, L.ysub32);

  if (int e = embed_rmsnorm(lc, f32, ctx->w.embed, anchor_ids, g.mask_id, V, ctx->layers[0].g_attn, g.eps, B, S, H, x,
                            u, u_lo))
    return e;
  const size_t lelems = layer_elems(ctx, kv);
  const size_t te = f32 ? 4 : 2;
  // conv coefficients of one site: tanh(W_c y + b_c), fp32 [R][H/8]
  auto coef_gemm = [&](int site, const dflash_layer_weights &lw, const void *y, const void *y_lo) {
    GemmOp op = wq(ctx, mk(lw.w_conv[site], H, y, y_lo, H, R, G8, H, EPI_TANH_BIAS, coef, G8, "conv_coef"),
                   lw.s_conv[site], lw.w_conv_bf16[site]);
    op.bias = lw.b_conv[site];
    return proj(ctx, lc, ws, L, op);
  };
  // a sublayer's output projection: straight into the fp32 residual, or (conv)
  // into fp32 + bf16 halves, then the post-site conv adds it to the residual
  // a post-sublayer short conv waiting for the next RMSNorm, which applies
  // it to the residual on the way (one launch fewer per site)
  const float *conv_y = nullptr, *conv_c = nullptr;
  auto out_proj = [&](int site, const dflash_layer_weights &lw, const void *Wm, const float *Ws, const void *Wb,
                      int K, const void *X, const void *X_lo, const char *name) -> int {
    if (!g.use_conv)
      return proj(ctx, lc, ws, L, wq(ctx, mk(Wm, K, X, X_lo, K, R, H, K, EPI_ADD_F32, x, H, name), Ws, Wb));
    GemmOp op = wq(ctx, mk(Wm, K, X, X_lo, K, R, H, K, f32 ? EPI_F32 : EPI_F32_SPLIT, ysub32, H, name), Ws, Wb);
    op.out2 = ysub;
    op.out2_lo = ysub_lo;
    op.ldo2 = H;
    if (int e = proj(ctx, lc, ws, L, op)) return e;
    if (int e = coef_gemm(site, lw, f32 ? static_cast<const void *>(ysub32) : ysub, ysub_lo)) return e;
    conv_y = ysub32;
    conv_c = coef;
    return DFLASH_OK;
  };
  // the next RMSNorm, taking the pending conv if there is one
  auto norm = [&](const float *gain, void *out, void *out_lo, void *mrows, void *mrows_lo) -> int {
    const float *cy = conv_y, *cc = conv_c;
    conv_y = conv_c = nullptr;
    return rmsnorm_rows(lc, f32, x, R, H, S, gain, g.eps, out, out_lo, mrows, mrows_lo, cy, cc);
  };
  for (int l = 0; l < g.n_layers; ++l) {
    const dflash_layer_weights &lw = ctx->layers[l];
    const void *ua = u, *ua_lo = u_lo;
    // ---- attention sublayer
    if (g.use_conv) {
      if (int e = coef_gemm(0, lw, u, u_lo)) return e;
      if (int e = conv_apply(lc, f32, u, u_lo, nullptr, coef, B, S, H, u2, u2_lo, nullptr)) return e;
      ua = u2;
      ua_lo = u2_lo;
    }
    if (int e = proj(ctx, lc, ws, L,
                     wq(ctx, mk(lw.w_qkv, H, ua, ua_lo, H, R, nh * d, H, EPI_F32, at<float>(ws, L.qkv), nh * d, "qkv"),
                        lw.s_qkv, lw.w_qkv_bf16)))
      return e;
    if (int e = qk_norm_rope(lc, f32, at<float>(ws, L.qkv), B, S, nq, nkv, d, lw.g_q, lw.g_k, g.qk_norm != 0, g.eps,
                             g.rope_base, ctx_len, at<void>(ws, L.q), at<void>(ws, L.bk), at<void>(ws, L.bv)))
      return e;
    AttnArgs aa = {};
    aa.q = at<void>(ws, L.q);
    aa.k_cache = static_cast<const char *>(kv->k_cache) + te * lelems * l;
    aa.v_cache = static_cast<const char *>(kv->v_cache) + te * lelems * l;
    aa.bk = at<void>(ws, L.bk);
    aa.bv = at<void>(ws, L.bv);
    aa.page_table = kv->page_table;
    aa.max_pages = kv->max_pages;
    aa.num_pages = kv->num_pages;
    aa.page_size = g.page_size;
    aa.ctx_len = ctx_len;
    aa.out = at<void>(ws, L.o);
    aa.out_lo = lo(L.o_lo);
    aa.B = B;
    aa.S = S;
    aa.nq = nq;
    aa.nkv = nkv;
    aa.d = d;
    aa.min_chunks = ctx->attn_split / 64;
    aa.counters = at<int>(ws, L.attn_ctr);
    aa.counter_cap = static_cast<size_t>(DFLASH_MAX_BATCH) * nkv;
    aa.partials = at<float>(ws, L.attn_part);
    aa.partial_slots = L.attn_part_slots;
    if (int e = f32 ? attention_f32(lc, aa) : attention_bf16(lc, aa)) return e;
    if (int e = out_proj(1, lw, lw.w_o, lw.s_o, lw.w_o_bf16, nq * d, aa.out, aa.out_lo, "o_proj")) return e;
    // ---- FFN sublayer
    if (int e = norm(lw.g_ffn, u, u_lo, nullptr, nullptr)) return e;
    ua = u;
    ua_lo = u_lo;
    if (g.use_conv) {
      if (int e = coef_gemm(2, lw, u, u_lo)) return e;
      if (int e = conv_apply(lc, f32, u, u_lo, nullptr, coef, B, S, H, u2, u2_lo, nullptr)) return e;
      ua = u2;
      ua_lo = u2_lo;
    }
    {
      GemmOp op = wq(ctx, mk(lw.w_gu, H, ua, ua_lo, H, R, 2 * F, H, EPI_SWIGLU, at<void>(ws, L.hmid), F, "gate_up"),
                     lw.s_gu, lw.w_gu_bf16);
      op.out_lo = hmid_lo;
      if (int e = proj(ctx, lc, ws, L, op)) return e;
    }
    if (int e = out_proj(3, lw, lw.w_down, lw.s_down, lw.w_down_bf16, F, at<void>(ws, L.hmid), hmid_lo, "down")) return e;
    if (l + 1 < g.n_layers)
      if (int e = norm(ctx->layers[l + 1].g_attn, u, u_lo, nullptr, nullptr)) return e;
  }
  if (int e = norm(ctx->w.g_final, hfinal, nullptr, at<void>(ws, L.hmask), lo(L.hmask_lo))) return e;
  // the fused epilogue hides under the LM head's weight stream only with
  // small token tiles (at most 32 mask rows per launch); larger launches are
  // tensor-bound and its per-tile selection would lengthen them
  if (!f32 && ctx->fused_topk && gemm_token_tile(B * J, split, g.weight_fp8 != 0) <= 32) {
    // LM head with the top-16 selection in its epilogue: per 128-row
    // vocabulary tile the 16 largest keys of each mask row (the fp32 logits
    // are written only when the caller asks for them), then one merge
    GemmOp op = wq(ctx, mk(ctx->w.lm_head, H, at<void>(ws, L.hmask), lo(L.hmask_lo), H, B * J, V, H, EPI_TOPK,
                           logits, V, "lm_head_topk"),
                   ctx->w.s_lm_head, ctx->w.lm_head_bf16);
    op.cand = at<uint64_t>(ws, L.cand);
    op.cand_ld = (V + 127) / 128;
    if (int e = proj(ctx, lc, ws, L, op)) return e;
    return topk16_merge(lc, op.cand, B * J, op.cand_ld, topk_ids, topk_logits, at<uint64_t>(ws, L.topk_part),
                        at<int>(ws, L.topk_ctr), TOPK_MAX_CHUNKS);
  }
  if (int e = proj(ctx, lc, ws, L,
                   wq(ctx, mk(ctx->w.lm_head, H, at<void>(ws, L.hmask), lo(L.hmask_lo), H, B * J, V, H, EPI_F32, lg, V,
                              "lm_head"),
                      ctx->w.s_lm_head, ctx->w.lm_head_bf16)))
    return e;
  return topk16(lc, lg, B * J, V, topk_ids, topk_logits, at<uint64_t>(ws, L.topk_part), at<int>(ws, L.topk_ctr),
                TOPK_MAX_CHUNKS);
}

int dflash_select_path(dflash_ctx *ctx, const int32_t *anchor_ids, const int32_t *topk_ids, const float *topk_logits,
                       const void *final_hidden, int batch, int32_t *draft_ids, float *pair_scores_out,
                       void *workspace, size_t workspace_bytes, dflash_stream_t stream) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  if (batch < 0) return set_error(DFLASH_ERR_ARG, "negative batch");
  if (batch == 0) return DFLASH_OK;
  if (!topk_ids || !draft_ids) return set_error(DFLASH_ERR_ARG, "dflash_select_path: null argument");
  const dflash_config &g = ctx->cfg;
  Launch lc = make_launch(ctx, workspace, reinterpret_cast<cudaStream_t>(stream));
  const int J = ctx->block - 1;
  if (!g.use_selector) return greedy_path(lc, nullptr, topk_ids, batch, J, false, draft_ids);
  if (!anchor_ids || !topk_logits || !final_hidden)
    return set_error(DFLASH_ERR_ARG, "dflash_select_path: the selector needs anchors, logits and final_hidden");
  float *sc = pair_scores_out;
  if (!sc) {
    if (int e = check_ws(ctx, workspace, workspace_bytes, batch, 0)) return e;
    sc = at<float>(workspace, layout(ctx, batch, 0).scores);
  }
  if (int e = pair_scores(lc, g.dtype == DFLASH_F32, anchor_ids, topk_ids, topk_logits, final_hidden, batch, J,
                          g.hidden, ctx->w.sel_e256, ctx->w.sel_a, ctx->w.sel_b, g.sel_rank, g.sel_dim, ctx->w.sel_w_g,
                          ctx->w.sel_b_g, sc))
    return e;
  return greedy_path(lc, sc, topk_ids, batch, J, true, draft_ids);
}

int dflash_sample_path(dflash_ctx *ctx, const int32_t *anchor_ids, const int32_t *topk_ids, const float *topk_logits,
                       const void *final_hidden, int batch, float temperature, const float *uniforms,
                       int32_t *draft_ids, float *draft_probs, float *pair_scores_out, void *workspace,
                       size_t workspace_bytes, dflash_stream_t stream) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  if (batch < 0) return set_error(DFLASH_ERR_ARG, "negative batch");
  if (batch == 0) return DFLASH_OK;
  if (!(temperature > 0.f)) return set_error(DFLASH_ERR_ARG, "temperature must be positive");
  if (!topk_ids || !topk_logits || !uniforms || !draft_ids || !draft_probs)
    return set_error(DFLASH_ERR_ARG, "dflash_sample_path: null argument");
  const dflash_config &g = ctx->cfg;
  Launch lc = make_launch(ctx, workspace, reinterpret_cast<cudaStream_t>(stream));
  const float *sc = nullptr;
  if (g.use_selector) {
    if (!anchor_ids || !final_hidden)
      return set_error(DFLASH_ERR_ARG, "dflash_sample_path: the selector needs anchors and final_hidden");
    float *s = pair_scores_out;
    if (!s) {
      if (int e = check_ws(ctx, workspace, workspace_bytes, batch, 0)) return e;
      s = at<float>(workspace, layout(ctx, batch, 0).scores);
    }
    if (int e = pair_scores(lc, g.dtype == DFLASH_F32, anchor_ids, topk_ids, topk_logits, final_hidden, batch,
                            ctx->block - 1, g.hidden, ctx->w.sel_e256, ctx->w.sel_a, ctx->w.sel_b, g.sel_rank, g.sel_dim,
                            ctx->w.sel_w_g, ctx->w.sel_b_g, s))
      return e;
    sc = s;
  }
  return sample_path(lc, sc, topk_logits, topk_ids, batch, ctx->block - 1, temperature, uniforms, draft_ids,
                     draft_probs);
}

int dflash_verify_rejection(dflash_ctx *ctx, const float *target_logits, const int32_t *draft_ids,
                            const int32_t *topk_ids, const float *draft_probs, const float *u_accept,
                            const float *u_bonus, int batch, int32_t *accept_len, int32_t *bonus, int32_t *committed,
                            void *workspace, size_t workspace_bytes, dflash_stream_t stream) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  if (batch < 0) return set_error(DFLASH_ERR_ARG, "negative batch");
  if (batch == 0) return DFLASH_OK;
  if (!target_logits || !draft_ids || !topk_ids || !draft_probs || !u_accept || !u_bonus || !accept_len || !bonus ||
      !committed)
    return set_error(DFLASH_ERR_ARG, "dflash_verify_rejection: null argument");
  if (int e = check_ws(ctx, workspace, workspace_bytes, batch, 0)) return e;
  Launch lc = make_launch(ctx, workspace, reinterpret_cast<cudaStream_t>(stream));
  return verify_rejection(lc, target_logits, ctx->cfg.vocab, at<float>(workspace, layout(ctx, batch, 0).lse),
                          draft_ids, topk_ids, draft_probs, u_accept, u_bonus, batch, ctx->block - 1, accept_len,
                          bonus, committed);
}

int dflash_verify_greedy(const int32_t *draft_ids, const int32_t *target_ids, int batch, int block_size,
                         int32_t *accept_len, int32_t *bonus, int32_t *committed, dflash_stream_t stream) {
  if (batch < 0) return set_error(DFLASH_ERR_ARG, "negative batch");
  if (block_size < 2 || block_size > 16) return set_error(DFLASH_ERR_ARG, "block_size must be 2..16");
  if (batch == 0) return DFLASH_OK;
  if (!draft_ids || !target_ids || !accept_len || !bonus || !committed)
    return set_error(DFLASH_ERR_ARG, "dflash_verify_greedy: null argument");
  Launch lc;
  lc.stream = reinterpret_cast<cudaStream_t>(stream);
  return verify(lc, draft_ids, target_ids, batch, block_size - 1, accept_len, bonus, committed);
}

int dflash_read_status(const void *workspace, int *device_status, dflash_stream_t stream) {
  if (!workspace || !device_status) return set_error(DFLASH_ERR_ARG, "null argument");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (int e = cuda_check(cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s), "status read"))
    return e;
  if (int e = cuda_check(cudaStreamSynchronize(s), "status sync")) return e;
  *device_status = v;
  if (v != 0) {
    cudaMemsetAsync(const_cast<void *>(workspace), 0, sizeof(int), s);
    cudaStreamSynchronize(s);
    return set_error(v, "a kernel reported status %d", v);
  }
  return DFLASH_OK;
}

int dflash_profile_begin(dflash_ctx *ctx) {
  if (!ctx) return set_error(DFLASH_ERR_ARG, "null context");
  ctx->prof.reset();
  ctx->prof.on = true;
  return DFLASH_OK;
}

int dflash_profile_end(dflash_ctx *ctx, dflash_kernel_stat *out, int max_out, int *n_out) {
  if (!ctx || !n_out) return set_error(DFLASH_ERR_ARG, "null argument");
  ctx->prof.on = false;
  std::map<std::string, dflash_kernel_stat> agg;
  std::vector<std::string> order;
  for (auto &r : ctx->prof.recs) {
    if (int e = cuda_check(cudaEventSynchronize(r.b), "profile sync")) return e;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    auto it = agg.find(r.name);
    if (it == agg.end()) {
      dflash_kernel_stat s = {};
      snprintf(s.name, sizeof(s.name), "%s", r.name);
      it = agg.emplace(r.name, s).first;
      order.push_back(r.name);
    }
    it->second.launches += 1;
    it->second.ms += ms;
    it->second.bytes += r.bytes > 0 ? r.bytes : 0;
    it->second.flops += r.flops > 0 ? r.flops : 0;
  }
  int n = 0;
  for (auto &nm : order) {
    if (out && n < max_out) out[n] = agg[nm];
    ++n;
  }
  *n_out = n;
  ctx->prof.reset();
  return DFLASH_OK;
}

int dflash_debug_wait_flag(const int32_t *flag, unsigned long long timeout_ns, void *workspace,
                           dflash_stream_t stream) {
  if (!flag || !workspace || timeout_ns == 0) return set_error(DFLASH_ERR_ARG, "null argument");
  Launch lc;
  lc.stream = reinterpret_cast<cudaStream_t>(stream);
  lc.status = at<int>(workspace, 0);
  lc.timeout_ns = timeout_ns;
  return wait_flag(lc, flag);
}

size_t dflash_debug_gemm_scratch_bytes(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return 256 + sizeof(int) * GEMM_COUNTERS + 4ull * sms * 2 * 128 * GEMM_MAX_BN;
}

int dflash_debug_gemm(const void *W, const float *w_scale, int w_fp8, const void *X, int M, int N, int K, float *out,
                      void *scratch, size_t scratch_bytes, int gemm_ctas, dflash_stream_t stream) {
  if (!W || !X || !out || !scratch || (w_fp8 && !w_scale) || M <= 0 || N <= 0 || K <= 0)
    return set_error(DFLASH_ERR_ARG, "debug gemm: bad argument");
  if (K % (w_fp8 ? 16 : 8)) return set_error(DFLASH_ERR_SHAPE, "debug gemm: K must be a multiple of %d", w_fp8 ? 16 : 8);
  if (!aligned16(scratch) || !aligned16(out)) return set_error(DFLASH_ERR_ALIGN, "debug gemm: misaligned buffer");
  const size_t need = dflash_debug_gemm_scratch_bytes();
  if (need == 0 || scratch_bytes < need) return set_error(DFLASH_ERR_SHAPE, "debug gemm: scratch too small");
  int dev = 0;
  Launch lc;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&lc.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return set_error(DFLASH_ERR_CUDA, "no CUDA device");
  lc.stream = reinterpret_cast<cudaStream_t>(stream);
  lc.status = static_cast<int *>(scratch);
  lc.gemm_ctas = gemm_ctas;
  GemmOp op = mk(W, K, X, nullptr, K, M, N, K, EPI_F32, out, N, "debug_gemm");
  if (w_fp8) {
    op.w_fp8 = true;
    op.wscale = w_scale;
  }
  GemmScratch sc;
  sc.counters = reinterpret_cast<int *>(static_cast<char *>(scratch) + 256);
  sc.n_counters = GEMM_COUNTERS;
  sc.partials = reinterpret_cast<float *>(static_cast<char *>(scratch) + 256 + sizeof(int) * GEMM_COUNTERS);
  sc.partial_floats = static_cast<size_t>(lc.num_sms) * 2 * 128 * GEMM_MAX_BN;
  return gemm_bf16(lc, op, sc);
}

int dflash_debug_gemm_plan(int M, int N, int K, int n_groups, int w_fp8, int split_act, int swiglu, int per_sm,
                           int num_sms, int gemm_ctas, long long *plan) {
  if (!plan || M <= 0 || N <= 0 || K <= 0 || n_groups < 1 || per_sm < 1 || num_sms < 1 || gemm_ctas < 0)
    return set_error(DFLASH_ERR_ARG, "debug gemm plan: bad argument");
  const GemmPlan pl = gemm_plan(M, N, K, n_groups, w_fp8 != 0, split_act != 0, swiglu != 0, per_sm, num_sms, gemm_ctas);
  const long long v[10] = {pl.BN, pl.rtpg, pl.tok_tiles, pl.kbpt, pl.G, pl.csk, pl.tiles, pl.total,
                           static_cast<long long>(num_sms) * 2 * 128 * GEMM_MAX_BN, GEMM_COUNTERS};
  for (int i = 0; i < 10; ++i) plan[i] = v[i];
  return DFLASH_OK;
}

int dflash_fp8_weights_to_bf16(const void *codes, int rows, int cols, void *out, dflash_stream_t stream) {
  if (rows <= 0 || cols <= 0 || cols % 4)
    return set_error(DFLASH_ERR_ARG, "fp8 weights to bf16: positive rows, cols a multiple of 4");
  Launch lc;
  lc.stream = reinterpret_cast<cudaStream_t>(stream);
  return fp8_rows_to_bf16(lc, codes, static_cast<long long>(rows) * cols, out);
}

int dflash_debug_gemm_pair_clusters(void) { return gemm_pair_clusters(); }

int dflash_debug_e4m3_to_bf16(const void *codes, int n, void *out, dflash_stream_t stream) {
  Launch lc;
  lc.stream = reinterpret_cast<cudaStream_t>(stream);
  return e4m3_to_bf16(lc, codes, n, out);
}

}  // extern "C"

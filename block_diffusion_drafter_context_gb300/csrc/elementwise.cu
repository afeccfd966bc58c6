// Row-wise kernels of the drafting step: embedding gather + RMSNorm, RMSNorm,
// context-feature norm, per-head q/k RMSNorm + RoPE, KV-injection scatter into
// the paged cache, and the DFlash-2 dynamic short convolution.
//
// Readings used where the pages give no layer internals (Qwen3-shaped
// drafter): RMSNorm y = g * x / sqrt(mean(x^2) + eps); RoPE pairs (i, i+d/2)
// with theta_i = base^(-2i/d), rotation (x, y) -> (x cos - y sin, y cos + x sin).
//
// GB300 notes: fp64 is a slow unit on this part, so theta_i is computed once
// on the host and passed as an fp32 (hi, lo) pair; the device forms the angle
// pos*theta with two fp64 multiply-adds, reduces it by 2*pi in fp64 and
// evaluates sin/cos in fp32.  Row kernels issue all of a row's 128-bit loads
// before the first use (no latency chain).  Outputs that feed a GEMM can be
// written as bf16 high + low halves (split activations).
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace dflash {
namespace {

constexpr int ROW_THREADS = 256;
constexpr int MAXV = 8;            // float4 per thread: rows up to 256*4*8 = 8192

template <typename T>
__host__ __device__ inline T *tp(void *p) {
  return static_cast<T *>(p);
}

// Block-wide sum (blockDim.x a multiple of 32).
__device__ __forceinline__ float block_sum(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16 *p, float4 v) {
  uint2 u;
  u.x = pack_bf16(v.x, v.y);
  u.y = pack_bf16(v.z, v.w);
  *reinterpret_cast<uint2 *>(p) = u;
}
// bf16 high half to p, low half (v - high) to lo (if given)
__device__ __forceinline__ void st4_hl(__nv_bfloat16 *p, __nv_bfloat16 *lo, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t *>(&a);
  u.y = *reinterpret_cast<const uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = u;
  if (lo) {
    uint2 l;
    l.x = pack_bf16(v.x - __low2float(a), v.y - __high2float(a));
    l.y = pack_bf16(v.z - __low2float(b), v.w - __high2float(b));
    *reinterpret_cast<uint2 *>(lo) = l;
  }
}
__device__ __forceinline__ void st4_hl(float *p, float *, float4 v) { st4(p, v); }

__device__ __forceinline__ float4 scale4(float4 a, float r, float4 g) {
  return make_float4(a.x * r * g.x, a.y * r * g.y, a.z * r * g.z, a.w * r * g.w);
}
__device__ __forceinline__ float dot4(float4 a) { return a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w; }

// cos / sin of pos * theta_i, theta_i = hi + lo (host-computed in fp64), all
// in fp32 (this GPU's fp64 rate is a small fraction of fp32's): the product
// pos * hi is split exactly into prod + err by one FMA, whole turns are
// removed from prod with 2 pi in three parts (Cody-Waite: 6.28125 has few
// significant bits; the rest in two fp32 terms), and the small terms are
// added back.  Angle error below 4e-7 rad for positions up to 2^17.
__device__ __forceinline__ void rope_cs(int pos, float th_hi, float th_lo, float &c, float &s) {
  const float p = static_cast<float>(pos);        // exact below 2^24
  const float prod = p * th_hi;
  const float err = fmaf(p, th_hi, -prod);        // p * th_hi = prod + err exactly
  const float tail = fmaf(p, th_lo, err);
  const float k = rintf(prod * 0.15915494309189535f);   // whole turns
  float r = fmaf(-k, 6.28125f, prod);
  r = fmaf(-k, 1.9353072e-3f, r);
  r = fmaf(-k, 1.0253132e-11f, r);
  sincosf(r + tail, &s, &c);
}

// ------------------------------------------------------------------ embed
// x[b*S+j] = E[id] (fp32 residual stream); u = RMSNorm(x) (activation dtype);
// S = block size: the anchor at j = 0, the mask token at j = 1..S-1
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS) embed_rmsnorm_kernel(const T *embed, const int32_t *anchor,
                                                                    int mask_id, int vocab, const float *gain,
                                                                    float eps, int H, int S, float *x, T *u, T *u_lo,
                                                                    int *status) {
  // Every input is the caller's (anchor ids, complete before any kernel of
  // this call starts) or a weight: all loads before the wait for the
  // previous kernel; the stores (x, u) after it.
  __shared__ float red[32];
  const int row = blockIdx.x, b = row / S, j = row % S;
  int id = j == 0 ? anchor[b] : mask_id;
  const bool bad = id < 0 || id >= vocab;
  if (bad) id = 0;
  const T *e = embed + static_cast<size_t>(id) * H;
  const int nv = H >> 2;
  float4 v[MAXV], g[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < nv) {
      v[k] = ld4(e + 4 * i);
      g[k] = ld4(gain + 4 * i);
    }
  }
  pdl_start();
  if (bad && threadIdx.x == 0) report(status, DFLASH_ERR_DEVICE);
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < nv) {
      st4(x + static_cast<size_t>(row) * H + 4 * i, v[k]);
      ss += dot4(v[k]);
    }
  }
  const float r = rsqrtf(block_sum(ss, red) / H + eps);
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < nv)
      st4_hl(u + static_cast<size_t>(row) * H + 4 * i, u_lo ? u_lo + static_cast<size_t>(row) * H + 4 * i : nullptr,
             scale4(v[k], r, g[k]));
  }
}

// ------------------------------------------------------------------ rmsnorm
// out[row] = RMSNorm(x[row]) (+ low halves); rows with j = row % S >= 1 are
// also written compactly to out_mask[b*(S-1) + j-1] (LM-head input of the
// mask rows).  With conv_coef, the DFlash-2 short conv of a post-sublayer
// site is applied first ("DFlash 2", Arquitectura del Sistema item 2):
// x[row] += y + a*y + b*y_prev (y = conv_y32, fp32 [rows][H]; a, b the
// row's two taps of each 16-channel group, interleaved in conv_coef
// [rows][H/8]; nothing before block position 0) and x written back - the
// same arithmetic as conv_kernel, one launch fewer.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS) rmsnorm_kernel(float *x, int H, const float *gain, float eps,
                                                              int S, T *out, T *out_lo, T *out_mask, T *out_mask_lo,
                                                              const float *conv_y32, const float *conv_coef) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const float *xr = x + static_cast<size_t>(row) * H;
  const int nv = H >> 2;
  float4 v[MAXV], g[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < MAXV; ++k)   // the gain is a weight: read before the wait (it may come from HBM)
    if (threadIdx.x + k * ROW_THREADS < nv) g[k] = ld4(gain + 4 * (threadIdx.x + k * ROW_THREADS));
  pdl_start();
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < nv) v[k] = ld4(xr + 4 * i);
  }
  const int b = row / S, j = row % S;
  if (conv_coef) {
    const float *yr = conv_y32 + static_cast<size_t>(row) * H;
    const float *cr = conv_coef + static_cast<size_t>(row) * (H / 8);
    float *xw = x + static_cast<size_t>(row) * H;
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
      const int i = threadIdx.x + k * ROW_THREADS;
      if (i >= nv) continue;
      const float4 yv = ld4(yr + 4 * i);
      const float4 yp = j ? ld4(yr - H + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float ca = cr[2 * (i >> 2)], cb = cr[2 * (i >> 2) + 1];   // group (4i) / 16
      const float cx = yv.x + ca * yv.x + cb * yp.x, cy = yv.y + ca * yv.y + cb * yp.y;
      const float cz = yv.z + ca * yv.z + cb * yp.z, cw = yv.w + ca * yv.w + cb * yp.w;
      v[k] = make_float4(v[k].x + cx, v[k].y + cy, v[k].z + cz, v[k].w + cw);
      *reinterpret_cast<float4 *>(xw + 4 * i) = v[k];
    }
  }
#pragma unroll
  for (int k = 0; k < MAXV; ++k)
    if (threadIdx.x + k * ROW_THREADS < nv) ss += dot4(v[k]);
  const float r = rsqrtf(block_sum(ss, red) / H + eps);
  const size_t mrow = static_cast<size_t>(b * (S - 1) + j - 1) * H;
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i >= nv) continue;
    const float4 y = scale4(v[k], r, g[k]);
    if (out) st4_hl(out + static_cast<size_t>(row) * H + 4 * i, out_lo ? out_lo + static_cast<size_t>(row) * H + 4 * i : nullptr, y);
    if (out_mask && j > 0) st4_hl(out_mask + mrow + 4 * i, out_mask_lo ? out_mask_lo + mrow + 4 * i : nullptr, y);
  }
}

// ------------------------------------------------------------------ feature
// f = RMSNorm(fc output) (or the plain projection); block 0 also saves the
// incoming context lengths so the scatter can read them even when the caller
// updates ctx_len in place.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS) feature_norm_kernel(const float *in, int H, const float *gain,
                                                                   float eps, int apply, T *out, T *out_lo,
                                                                   const int32_t *ctx_in, int32_t *ctx_saved, int B) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int nv = H >> 2;
  float4 v[MAXV], g[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < MAXV; ++k)   // the gain is a weight: read before the wait
    if (threadIdx.x + k * ROW_THREADS < nv)
      g[k] = apply ? ld4(gain + 4 * (threadIdx.x + k * ROW_THREADS)) : make_float4(1.f, 1.f, 1.f, 1.f);
  pdl_start();
  if (row == 0)
    for (int b = threadIdx.x; b < B; b += blockDim.x) ctx_saved[b] = ctx_in[b];
  const float *xr = in + static_cast<size_t>(row) * H;
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < nv) {
      v[k] = ld4(xr + 4 * i);
      ss += dot4(v[k]);
    }
  }
  const float r = apply ? rsqrtf(block_sum(ss, red) / H + eps) : 1.f;
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < nv)
      st4_hl(out + static_cast<size_t>(row) * H + 4 * i, out_lo ? out_lo + static_cast<size_t>(row) * H + 4 * i : nullptr,
             scale4(v[k], r, g[k]));
  }
}

// ------------------------------------------------------------------ q/k norm + rope
struct RopeArgs {
  float th_hi[64], th_lo[64];
};

// This lane's angles theta_{lane + 32 i}, i < N, from the parameter table.
// Kernel parameters indexed by lane serialise the constant bank (one access
// per distinct address, each a possible miss); uniform reads broadcast, so
// the warp walks the table uniformly and each lane keeps its entries.
template <int N>
__device__ __forceinline__ void lane_thetas(const RopeArgs &rp, int lane, float (&hi)[N], float (&lo)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) hi[i] = lo[i] = 0.f;
#pragma unroll 4
  for (int k = 0; k < 32; ++k) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float h = rp.th_hi[k + 32 * i], l = rp.th_lo[k + 32 * i];
      if (lane == k) {
        hi[i] = h;
        lo[i] = l;
      }
    }
  }
}

// 16 consecutive values with vector stores (dst 16-byte aligned).
__device__ __forceinline__ void store16(float *dst, const float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    reinterpret_cast<float4 *>(dst)[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
}
__device__ __forceinline__ void store16(__nv_bfloat16 *dst, const float (&x)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = pack_bf16(x[2 * i], x[2 * i + 1]);
  reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Small batches: the same outputs with one warp per (block row, head) and
// no shared memory, so that the block attention's CTAs (which take nearly
// all of an SM's shared memory) can already become resident - and set up -
// while this kernel runs under programmatic dependent launch.
// qkv: fp32 [B*S][(nq+2nkv)*d] (S = block size).  One warp per (token,
// head).  q heads -> q_out [B*S][nq*d]; k heads -> bk [B][nkv][64][d]
// (normed, rotated); v heads -> bv [B][nkv][d][64], transposed like the V
// pages.  Rows / columns S..63 are padding up to one 64-token page:
// attention masks the scores of rows S.. and skips V columns 16..; V columns
// S..15 share a k-step with the block tokens and are written as zeros.
template <typename T, int DPL>
__global__ void __launch_bounds__(256) qk_rope_rows_kernel(const float *qkv, int nq, int nkv, int S, const float *g_q,
                                                      const float *g_k, int qk_norm, float eps, const RopeArgs rp,
                                                      const int32_t *ctx_len, T *q_out, T *bk, T *bv) {
  constexpr int D = DPL * 32;
  const int tok = blockIdx.x, b = tok / S, j = tok % S;
  const int head = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int nh = nq + 2 * nkv;
  // the norm gain and this lane's angles are weights: read before the wait
  // for the projections, off the dependent chain
  const bool is_q = head < nq, normed = qk_norm && head < nq + nkv;
  float gn[DPL], th_hi[DPL / 2], th_lo[DPL / 2];
#pragma unroll
  for (int i = 0; i < DPL; ++i) gn[i] = normed ? (is_q ? g_q : g_k)[lane + 32 * i] : 1.f;
  lane_thetas(rp, lane, th_hi, th_lo);
  pdl_start();
  if (head >= nh) return;
  const float *src = qkv + static_cast<size_t>(tok) * nh * D + static_cast<size_t>(head) * D;
  float v[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) v[i] = src[lane + 32 * i];
  if (head >= nq + nkv) {   // value head: copy, transposed
    T *dst = bv + (static_cast<size_t>(b) * nkv + (head - nq - nkv)) * D * 64 + j;
#pragma unroll
    for (int i = 0; i < DPL; ++i) Elt<T>::st(dst + static_cast<size_t>(lane + 32 * i) * 64, v[i]);
    // the block's PV k-step reads columns 0..15: below a block of 16 the
    // columns S..15 get zeros (a 0 probability times a stale NaN is NaN),
    // spread over the block's tokens: token j clears j+S, j+2S, ...
    for (int c = j + S; c < 16; c += S)
#pragma unroll
      for (int i = 0; i < DPL; ++i) Elt<T>::st(dst + (c - j) + static_cast<size_t>(lane + 32 * i) * 64, 0.f);
    return;
  }
  const int pos = ctx_len[b] + j;
  if (qk_norm) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) ss += v[i] * v[i];
    const float r = rsqrtf(warp_sum(ss) / D + eps);
#pragma unroll
    for (int i = 0; i < DPL; ++i) v[i] *= r * gn[i];
  }
  float o[DPL];
#pragma unroll
  for (int i = 0; i < DPL / 2; ++i) {   // pairs (lane + 32i, lane + 32i + D/2)
    float c, s;
    rope_cs(pos, th_hi[i], th_lo[i], c, s);
    const float x1 = v[i], x2 = v[i + DPL / 2];
    o[i] = x1 * c - x2 * s;
    o[i + DPL / 2] = x2 * c + x1 * s;
  }
  T *dst = is_q ? q_out + static_cast<size_t>(tok) * nq * D + static_cast<size_t>(head) * D
                : bk + ((static_cast<size_t>(b) * nkv + (head - nq)) * 64 + j) * D;
#pragma unroll
  for (int i = 0; i < DPL; ++i) Elt<T>::st(dst + lane + 32 * i, o[i]);
}

// Per-head RMSNorm and RoPE of one head row held as lane + 32 i (i < DPL),
// pairs (i, i + DPL/2); cs: the row's (cos, sin) per pair, in shared memory.
template <int DPL>
__device__ __forceinline__ void norm_rope_row(float (&v)[DPL], const float (&gn)[DPL], bool norm, float eps,
                                              const float2 *cs, int lane) {
  constexpr int D = DPL * 32;
  if (norm) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) ss += v[i] * v[i];
    const float r = rsqrtf(warp_sum(ss) / D + eps);
#pragma unroll
    for (int i = 0; i < DPL; ++i) v[i] *= r * gn[i];
  }
  float o[DPL];
#pragma unroll
  for (int i = 0; i < DPL / 2; ++i) {
    const float2 c = cs[lane + 32 * i];
    const float x1 = v[i], x2 = v[i + DPL / 2];
    o[i] = x1 * c.x - x2 * c.y;
    o[i + DPL / 2] = x2 * c.x + x1 * c.y;
  }
#pragma unroll
  for (int i = 0; i < DPL; ++i) v[i] = o[i];
}

// Rows of the block's q / k / v projections, CTAs (request b, kv head h,
// split z): the g = nq/nkv query heads of h, the k head h and the v head h
// over the request's S rows (qkv: fp32 [B*S][(nq+2nkv)*d]); with few
// requests the (head, row) items and the v head's d-rows are split over
// gridDim.z CTAs so that the launch still covers the SMs.  The rotation of
// each row (position ctx_len[b] + j) is tabulated once per CTA in shared
// memory and shared by its heads.  q heads -> q_out [B*S][nq*d]; k head -> bk
// [B][nkv][64][d] (normed, rotated); v head -> bv [B][nkv][d][64],
// transposed like the V pages: the CTA stages the S rows in shared memory
// and each thread writes one d-row's 16 columns (32 bytes, whole sectors).
// Rows / columns S..63 are padding up to one 64-token page: attention masks
// the scores of rows S.. and skips V columns 16..; V columns S..15 share a
// k-step with the block tokens and are written as zeros.
template <typename T, int DPL>
__global__ void __launch_bounds__(256) qk_rope_kernel(const float *qkv, int nq, int nkv, int S, const float *g_q,
                                                      const float *g_k, int qk_norm, float eps, const RopeArgs rp,
                                                      const int32_t *ctx_len, T *q_out, T *bk, T *bv) {
  constexpr int D = DPL * 32, HALF = D / 2, U = 4;
  __shared__ float2 cs[16][HALF];
  __shared__ float vt[16][D];
  const int b = blockIdx.x, h = blockIdx.y, g = nq / nkv, nh = nq + 2 * nkv;
  const int z = blockIdx.z, nz = gridDim.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the norm gains and this lane's angles are weights: read before the wait
  float gq[DPL], gk[DPL], th_hi[DPL / 2], th_lo[DPL / 2];
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    gq[i] = qk_norm ? g_q[lane + 32 * i] : 1.f;
    gk[i] = qk_norm ? g_k[lane + 32 * i] : 1.f;
  }
  lane_thetas(rp, lane, th_hi, th_lo);
  pdl_start();
  const int n0 = ctx_len[b];
  for (int j = warp; j < S; j += 8)
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) {
      float c, sn;
      rope_cs(n0 + j, th_hi[i], th_lo[i], c, sn);
      cs[j][lane + 32 * i] = make_float2(c, sn);
    }
  // this CTA's d-rows of the v head: S rows into shared memory
  const int d0 = z * D / nz, d1 = (z + 1) * D / nz, dn = d1 - d0;
  const float *vsrc = qkv + static_cast<size_t>(b) * S * nh * D + static_cast<size_t>(nq + nkv + h) * D + d0;
  for (int e = threadIdx.x; e < S * dn; e += 256) vt[e / dn][e % dn] = vsrc[static_cast<size_t>(e / dn) * nh * D + e % dn];
  __syncthreads();
  // q and k rows: (g + 1) heads x S rows, one warp per (head, row), U rows'
  // loads in flight per warp; this CTA's share of them
  const int items_all = (g + 1) * S;
  const int i_lo = z * items_all / nz, items = (z + 1) * items_all / nz;
  for (int it0 = i_lo + warp * U; it0 < items; it0 += 8 * U) {
    float v[U][DPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = it0 + u;
      if (it < items) {
        const int hh = it / S, j = it % S, head = hh < g ? h * g + hh : nq + h;
        const float *src = qkv + static_cast<size_t>(b * S + j) * nh * D + static_cast<size_t>(head) * D;
#pragma unroll
        for (int i = 0; i < DPL; ++i) v[u][i] = src[lane + 32 * i];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = it0 + u;
      if (it >= items) break;
      const int hh = it / S, j = it % S;
      const bool isq = hh < g;
      norm_rope_row<DPL>(v[u], isq ? gq : gk, qk_norm != 0, eps, cs[j], lane);
      T *dst = isq ? q_out + static_cast<size_t>(b * S + j) * nq * D + static_cast<size_t>(h * g + hh) * D
                   : bk + ((static_cast<size_t>(b) * nkv + h) * 64 + j) * D;
#pragma unroll
      for (int i = 0; i < DPL; ++i) Elt<T>::st(dst + lane + 32 * i, v[u][i]);
    }
  }
  // V^T: one thread per d-row writes its columns 0..15 (zeros from S on) as
  // one 32-byte sector (bf16; 64 bytes fp32)
  if (threadIdx.x < dn) {
    const int d = threadIdx.x;
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = j < S ? vt[j][d] : 0.f;
    store16(bv + ((static_cast<size_t>(b) * nkv + h) * D + d0 + d) * 64, x);
  }
}

// ------------------------------------------------------------------ injection scatter
// kvproj: fp32 [L][T][2*nkv*d] (k heads then v heads of each layer's W_k, W_v
// applied to the context feature).  Token t belongs to the request b with
// cu_new[b] <= t < cu_new[b+1], position ctx_saved[b] + t - cu_new[b].
struct ScatterArgs {
  const float *kvproj;
  int T, L, nkv;
  const float *g_k[16];
  int qk_norm;
  float eps;
  const int32_t *cu_new;
  int B;
  const int32_t *ctx_saved;
  int32_t *ctx_out;
  void *k_cache, *v_cache;
  const int32_t *page_table;
  int num_pages, max_pages, page;
  size_t layer_elems;
  int *status;
};

// One CTA per (16 consecutive new tokens, layer, kv head).
// Each token is placed once (request, position, pool page, slot) and its
// rotation tabulated once in shared memory.  K heads: k-norm + RoPE, one
// warp per (head, token), U tokens' loads in flight; written to the K pages
// ([page][nkv][slot][d]).  V heads: the 16 x d tile is staged in shared
// memory and written transposed into the V pages ([page][nkv][d][slot]) by
// lanes that cover 16 consecutive tokens of two d-rows per store (the
// tokens of a request occupy consecutive slots: whole or two sectors per
// d-row instead of one 2-byte write each).
template <typename T, int DPL>
__global__ void __launch_bounds__(256) inject_scatter_kernel(const ScatterArgs a, const RopeArgs rp) {
  constexpr int D = DPL * 32, HALF = D / 2, U = 4;
  __shared__ float2 cs[16][HALF];
  __shared__ float vt[16][D];
  __shared__ int s_page[16], s_slot[16];
  const int t0 = blockIdx.x * 16, l = blockIdx.y, h = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = min(16, a.T - t0);
  float gk[DPL], th_hi[DPL / 2], th_lo[DPL / 2];
#pragma unroll
  for (int i = 0; i < DPL; ++i) gk[i] = a.qk_norm ? a.g_k[l][lane + 32 * i] : 1.f;
  lane_thetas(rp, lane, th_hi, th_lo);
  pdl_start();
  if (blockIdx.x == 0 && l == 0 && h == 0)
    for (int b = threadIdx.x; b < a.B; b += blockDim.x)
      a.ctx_out[b] = a.ctx_saved[b] + (a.cu_new[b + 1] - a.cu_new[b]);
  __shared__ int s_pos[16];
  if (threadIdx.x < nt) {
    const int t = t0 + threadIdx.x;
    // request of token t: last b with cu_new[b] <= t
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu_new[mid] <= t)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int pos = a.ctx_saved[lo] + t - a.cu_new[lo];
    const int pidx = pos / a.page;
    const int pg = (pos >= 0 && pidx < a.max_pages) ? a.page_table[static_cast<size_t>(lo) * a.max_pages + pidx] : -1;
    const bool ok = pg >= 0 && pg < a.num_pages;
    if (!ok) report(a.status, DFLASH_ERR_DEVICE);
    s_page[threadIdx.x] = ok ? pg : -1;
    s_slot[threadIdx.x] = pos % a.page;
    s_pos[threadIdx.x] = pos;
  }
  __syncthreads();
  for (int j = warp; j < nt; j += 8)
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) {
      float c, sn;
      rope_cs(s_pos[j], th_hi[i], th_lo[i], c, sn);
      cs[j][lane + 32 * i] = make_float2(c, sn);
    }
  __syncthreads();
  const size_t row_stride = static_cast<size_t>(2 * a.nkv) * D;
  const float *base = a.kvproj + (static_cast<size_t>(l) * a.T + t0) * row_stride;
  T *kc = static_cast<T *>(a.k_cache) + l * a.layer_elems;
  T *vc = static_cast<T *>(a.v_cache) + l * a.layer_elems;
  // the V head's 16 x d tile into shared memory (its loads in flight with
  // the K rows' below)
  for (int e = threadIdx.x; e < nt * D; e += 256)
    vt[e / D][e % D] = base[(e / D) * row_stride + static_cast<size_t>(a.nkv + h) * D + e % D];
  // K head: one warp per token, two tokens per warp
  for (int j0 = warp * 2; j0 < nt; j0 += 16) {
    float v[2][DPL];
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (j0 + u < nt) {
        const float *src = base + (j0 + u) * row_stride + static_cast<size_t>(h) * D;
#pragma unroll
        for (int i = 0; i < DPL; ++i) v[u][i] = src[lane + 32 * i];
      }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int j = j0 + u;
      if (j >= nt) break;
      norm_rope_row<DPL>(v[u], gk, a.qk_norm != 0, a.eps, cs[j], lane);
      const int pg = s_page[j];
      if (pg < 0) continue;
      T *dst = kc + ((static_cast<size_t>(pg) * a.nkv + h) * a.page + s_slot[j]) * D;
#pragma unroll
      for (int i = 0; i < DPL; ++i) Elt<T>::st(dst + lane + 32 * i, v[u][i]);
    }
  }
  __syncthreads();
  // V^T: 16 consecutive threads cover one d-row's 16 tokens (consecutive slots)
  for (int e = threadIdx.x; e < 16 * D; e += 256) {
    const int d = e >> 4, j = e & 15;
    const int pg = j < nt ? s_page[j] : -1;
    if (pg >= 0) Elt<T>::st(vc + ((static_cast<size_t>(pg) * a.nkv + h) * D + d) * a.page + s_slot[j], vt[j][d]);
  }
}

// ------------------------------------------------------------------ short conv
// DFlash-2 ("DFlash 2", Arquitectura del Sistema item 2): two taps along the
// block, coefficients per 16-channel group, nothing before position 0.
//   coef: fp32 [B*S][H/8] = tanh(W_c y + b_c), interleaved per group g:
//         column 2g current tap a, 2g+1 previous tap b (S = block size <= 16).
//   out_j = y_j + a_j * y_j + b_j * y_{j-1}
// y is either an activation (hi [+ lo] halves) or fp32 (y32).  Pre sites
// write out (+ low halves), post sites add into the residual x_add.
template <typename T>
__global__ void __launch_bounds__(256) conv_kernel(const T *y, const T *y_lo, const float *y32, const float *coef,
                                                   int H, int S, T *out_t, T *out_lo, float *x_add) {
  pdl_start();
  const int b = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  const int G = H / 16, grp = c >> 4;
  float yv[16], av[16], bv[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j >= S) break;
    const size_t row = static_cast<size_t>(b) * S + j;
    yv[j] = y32 ? y32[row * H + c] : Elt<T>::ld(y + row * H + c) + (y_lo ? Elt<T>::ld(y_lo + row * H + c) : 0.f);
    av[j] = coef[row * (2 * G) + 2 * grp];
    bv[j] = coef[row * (2 * G) + 2 * grp + 1];
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j >= S) break;
    const size_t row = static_cast<size_t>(b) * S + j;
    const float v = yv[j] + av[j] * yv[j] + bv[j] * (j ? yv[j - 1] : 0.f);
    if (out_t) {
      Elt<T>::st(out_t + row * H + c, v);
      if (out_lo) Elt<T>::st(out_lo + row * H + c, v - Elt<T>::ld(out_t + row * H + c));
    } else {
      x_add[row * H + c] += v;
    }
  }
}

template <typename F>
int run(const Launch &lc, const char *name, F f) {
  ProfScope ps(lc, name, -1.0, -1.0);
  f();
  return cuda_check(cudaGetLastError(), name);
}

RopeArgs rope_table(int d, float base) {
  RopeArgs r = {};
  for (int i = 0; i < d / 2 && i < 64; ++i) {
    const double th = pow(static_cast<double>(base), -2.0 * i / d);
    r.th_hi[i] = static_cast<float>(th);
    r.th_lo[i] = static_cast<float>(th - static_cast<double>(r.th_hi[i]));
  }
  return r;
}

int check_row(int H) {
  if (H % 4 || H > ROW_THREADS * 4 * MAXV)
    return set_error(DFLASH_ERR_UNSUPPORTED, "row kernels need hidden %% 4 == 0 and hidden <= %d", ROW_THREADS * 4 * MAXV);
  return DFLASH_OK;
}

}  // namespace

int embed_rmsnorm(const Launch &lc, bool f32, const void *embed, const int32_t *anchor, int mask_id, int vocab,
                  const float *gain, float eps, int B, int S, int H, float *x, void *u, void *u_lo) {
  if (int e = check_row(H)) return e;
  return run(lc, "embed_norm", [&] {
    if (f32)
      launch_pdl(embed_rmsnorm_kernel<float>, dim3(B * S), dim3(ROW_THREADS), 0, lc.stream,
          static_cast<const float *>(embed), anchor, mask_id, vocab, gain, eps, H, S, x, tp<float>(u), nullptr,
          lc.status);
    else
      launch_pdl(embed_rmsnorm_kernel<__nv_bfloat16>, dim3(B * S), dim3(ROW_THREADS), 0, lc.stream,
          static_cast<const __nv_bfloat16 *>(embed), anchor, mask_id, vocab, gain, eps, H, S, x, tp<__nv_bfloat16>(u),
          tp<__nv_bfloat16>(u_lo), lc.status);
  });
}

int rmsnorm_rows(const Launch &lc, bool f32, float *x, int rows, int H, int S, const float *gain, float eps,
                 void *out, void *out_lo, void *out_mask_rows, void *out_mask_lo, const float *conv_y32,
                 const float *conv_coef) {
  if (int e = check_row(H)) return e;
  if (conv_coef && (!conv_y32 || H % 16)) return set_error(DFLASH_ERR_ARG, "rmsnorm: conv needs y and 16-channel groups");
  return run(lc, "rmsnorm", [&] {
    if (f32)
      launch_pdl(rmsnorm_kernel<float>, dim3(rows), dim3(ROW_THREADS), 0, lc.stream, x, H, gain, eps, S,
                 tp<float>(out), nullptr, tp<float>(out_mask_rows), nullptr, conv_y32, conv_coef);
    else
      launch_pdl(rmsnorm_kernel<__nv_bfloat16>, dim3(rows), dim3(ROW_THREADS), 0, lc.stream,
          x, H, gain, eps, S, tp<__nv_bfloat16>(out), tp<__nv_bfloat16>(out_lo), tp<__nv_bfloat16>(out_mask_rows),
          tp<__nv_bfloat16>(out_mask_lo), conv_y32, conv_coef);
  });
}

int feature_norm(const Launch &lc, bool f32, const float *in, int rows, int H, const float *gain, float eps,
                 bool apply_norm, void *out, void *out_lo, const int32_t *ctx_len_in, int32_t *ctx_len_saved, int B) {
  if (rows <= 0) return DFLASH_OK;
  if (int e = check_row(H)) return e;
  return run(lc, "feature_norm", [&] {
    if (f32)
      launch_pdl(feature_norm_kernel<float>, dim3(rows), dim3(ROW_THREADS), 0, lc.stream, in, H, gain, eps, apply_norm, tp<float>(out),
                                                                      nullptr, ctx_len_in, ctx_len_saved, B);
    else
      launch_pdl(feature_norm_kernel<__nv_bfloat16>, dim3(rows), dim3(ROW_THREADS), 0, lc.stream,
          in, H, gain, eps, apply_norm, tp<__nv_bfloat16>(out), tp<__nv_bfloat16>(out_lo), ctx_len_in, ctx_len_saved,
          B);
  });
}

int qk_norm_rope(const Launch &lc, bool f32, const float *qkv, int B, int S, int nq, int nkv, int d,
                 const float *g_q, const float *g_k, bool qk_norm, float eps, float rope_base, const int32_t *ctx_len,
                 void *q_out, void *bk, void *bv) {
  if (S > 16) return set_error(DFLASH_ERR_UNSUPPORTED, "q/k norm + RoPE: block size above 16");
  const RopeArgs rp = rope_table(d, rope_base);
  if (2 * B * nkv < lc.num_sms) {
    // few (request, kv head) lists: the shared-memory-free row kernel
    dim3 grid_rows(B * S, (nq + 2 * nkv + 7) / 8);
    return run(lc, "qk_norm_rope", [&] {
#define QKR(T, DPL)                                                                                        \
  launch_pdl(qk_rope_rows_kernel<T, DPL>, dim3(grid_rows), dim3(256), 0, lc.stream, qkv, nq, nkv, S, g_q, g_k, qk_norm, \
             eps, rp, ctx_len, tp<T>(q_out), tp<T>(bk), tp<T>(bv))
      if (f32 && d == 64)
        QKR(float, 2);
      else if (f32)
        QKR(float, 4);
      else if (d == 64)
        QKR(__nv_bfloat16, 2);
      else
        QKR(__nv_bfloat16, 4);
#undef QKR
    });
  }
  // split each (request, kv head) over nz CTAs until the launch covers the
  // SMs, keeping at least 8 (head, row) items per CTA
  const int items = (nq / nkv + 1) * S;
  int nz = (lc.num_sms + B * nkv - 1) / (B * nkv);
  nz = nz < 1 ? 1 : (nz > items / 8 ? (items / 8 > 0 ? items / 8 : 1) : nz);
  nz = nz > d ? d : nz;
  dim3 grid(B, nkv, nz);
  return run(lc, "qk_norm_rope", [&] {
#define QK(T, DPL)                                                                                         \
  launch_pdl(qk_rope_kernel<T, DPL>, dim3(grid), dim3(256), 0, lc.stream, qkv, nq, nkv, S, g_q, g_k, qk_norm, eps, rp, ctx_len, \
                                                      tp<T>(q_out), tp<T>(bk), tp<T>(bv))
    if (f32 && d == 64)
      QK(float, 2);
    else if (f32)
      QK(float, 4);
    else if (d == 64)
      QK(__nv_bfloat16, 2);
    else
      QK(__nv_bfloat16, 4);
#undef QK
  });
}

int inject_scatter(const Launch &lc, bool f32, const float *kvproj, int T, int L, int nkv, int d,
                   const float *const *g_k, bool qk_norm, float eps, float rope_base, const int32_t *cu_new, int B,
                   const int32_t *ctx_len_saved, int32_t *ctx_len_out, const dflash_kv &kv, size_t layer_elems) {
  if (T <= 0) return DFLASH_OK;
  if (L > 16) return set_error(DFLASH_ERR_UNSUPPORTED, "at most 16 drafter layers");
  ScatterArgs a = {};
  a.kvproj = kvproj;
  a.T = T;
  a.L = L;
  a.nkv = nkv;
  for (int l = 0; l < L; ++l) a.g_k[l] = g_k[l];
  a.qk_norm = qk_norm;
  a.eps = eps;
  a.cu_new = cu_new;
  a.B = B;
  a.ctx_saved = ctx_len_saved;
  a.ctx_out = ctx_len_out;
  a.k_cache = kv.k_cache;
  a.v_cache = kv.v_cache;
  a.page_table = kv.page_table;
  a.num_pages = kv.num_pages;
  a.max_pages = kv.max_pages;
  a.page = 64;
  a.layer_elems = layer_elems;
  a.status = lc.status;
  const RopeArgs rp = rope_table(d, rope_base);
  dim3 grid((T + 15) / 16, L, nkv);
  return run(lc, "inject_scatter", [&] {
    if (f32 && d == 64)
      launch_pdl(inject_scatter_kernel<float, 2>, dim3(grid), dim3(256), 0, lc.stream, a, rp);
    else if (f32)
      launch_pdl(inject_scatter_kernel<float, 4>, dim3(grid), dim3(256), 0, lc.stream, a, rp);
    else if (d == 64)
      launch_pdl(inject_scatter_kernel<__nv_bfloat16, 2>, dim3(grid), dim3(256), 0, lc.stream, a, rp);
    else
      launch_pdl(inject_scatter_kernel<__nv_bfloat16, 4>, dim3(grid), dim3(256), 0, lc.stream, a, rp);
  });
}

int conv_apply(const Launch &lc, bool f32, const void *y, const void *y_lo, const float *y32, const float *coef, int B,
               int S, int H, void *out_t, void *out_lo, float *x_add) {
  dim3 grid((H + 255) / 256, B);
  return run(lc, "short_conv", [&] {
    if (f32)
      launch_pdl(conv_kernel<float>, dim3(grid), dim3(256), 0, lc.stream, static_cast<const float *>(y), nullptr, y32, coef, H,
                 S, tp<float>(out_t), nullptr, x_add);
    else
      launch_pdl(conv_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, lc.stream,
          static_cast<const __nv_bfloat16 *>(y), static_cast<const __nv_bfloat16 *>(y_lo), y32, coef, H, S,
          tp<__nv_bfloat16>(out_t), tp<__nv_bfloat16>(out_lo), x_add);
  });
}

}  // namespace dflash

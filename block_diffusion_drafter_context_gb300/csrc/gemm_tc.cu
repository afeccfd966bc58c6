// Persistent stream-K GEMM on the 5th-generation tensor cores (tcgen05).
//
//   out[m][n] = epi( sum_k X[m][k] * W[n][k] )      W: [N][K] weights, X: [M][K]
//
// Every drafter projection (context feature, per-layer K/V injection, QKV, O,
// gate/up, down, conv coefficients, LM head) is this contraction.  During a
// drafting step M is tiny (16 tokens per request) while W is up to 1.2 GB, so
// the kernel is built around streaming W at HBM speed:
//   * swap-AB: the weight tile is the 128-row UMMA "M" operand, the token
//     tile (BN = 16..256 rows) the "N" operand; the accumulator sits in TMEM
//     as [weight row = lane][token = column];
//   * decomposition, chosen per launch on the host: cluster split-K when the
//     GEMM has at most half as many tiles as CTA slots (the CTAs of one
//     thread-block cluster split a tile's k-range and reduce on chip through
//     distributed shared memory); one whole tile per CTA when there are more
//     tiles than SMs but no more than slots; otherwise stream-K: the (tile,
//     k-block) iteration space is cut into one contiguous range per CTA, and
//     a tile split across CTAs is finished by whichever CTA completes it last
//     (per-tile counter), which sums the fp32 partials in CTA order -
//     deterministic, no spin-waits;
//   * tile order: token tile outer, weight row tile inner (tile = tok * RT +
//     rt).  With several token tiles the CTAs that own the same weight rows
//     for different token tiles sit G / tok_tiles apart and advance in step,
//     so each weight tile leaves DRAM once and the other readers hit L2; the
//     evict-first hint on the weight stream is used only with one token tile;
//   * warp roles: warp 0 issues TMA loads into a STAGES-deep ring of
//     128-byte-swizzled tiles, warp 1 owns TMEM and issues tcgen05.mma from
//     one thread, warps 2-5 drain TMEM (double-buffered) into the epilogue;
//   * split activations (SPLIT): the activation operand arrives as two bf16
//     tensors, high and low halves of the fp32 value; each k-step issues a
//     second MMA on the same weight tile, so the product carries ~16 mantissa
//     bits of the activation at no extra HBM traffic (the weight stream, not
//     the tensor pipe, bounds these GEMMs);
//   * FP8 weights (F8): the weight stream is E4M3 codes with one fp32 scale
//     per output row.  TMA lands a [128 rows][128 codes] tile (16 KB,
//     128-byte swizzle); four converter warps, one TMEM lane quarter each,
//     turn their rows into the exact bf16 values and store them into tensor
//     memory (three tiles), from where the MMA reads its A operand.  Staging
//     the bf16 tile in shared memory instead would move ~6.5 bytes of shared
//     memory per HBM byte, past the SM's shared-memory bandwidth at full HBM
//     rate; this way it is ~2.5, as for bf16 weights.  Activations stay bf16,
//     so the precision is that of the bf16 path; the row scale is applied in
//     the epilogue.  Half the HBM bytes per weight; up to two CTAs per SM so
//     that two threads issue MMAs on each SM.
// Every mbarrier wait is bounded (status word + unwind on timeout).
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <atomic>

namespace dflash {
namespace {

constexpr int BM = 128;   // weight rows per tile (UMMA M)
constexpr int BK = 64;    // bf16 elements per stage row = 128 bytes = one swizzle row
constexpr int UK = 16;    // K per tcgen05.mma (kind::f16)
constexpr int MAX_GROUPS = 16;   // weight matrices sharing one launch (same shape, same activations)
constexpr int SMEM_PER_SM = 228 * 1024;   // shared memory of one SM (1 KB of it reserved per resident CTA)

struct WMaps {
  CUtensorMap m[MAX_GROUPS];
};

constexpr int pow2_at_least(int x) { return x <= 32 ? 32 : 2 * pow2_at_least((x + 1) / 2); }

template <int BN, bool SPLIT, bool F8>
struct Cfg {
  // warps: 0 TMA, 1 MMA, 2-5 epilogue, (F8) 6-9 weight converters
  static constexpr int CONV_WARPS = F8 ? 4 : 0;
  static constexpr int NT = 192 + 32 * CONV_WARPS;
  static constexpr int BKI = F8 ? 2 * BK : BK;         // k per ring stage (one k-block)
  static constexpr int BT = BKI / BK;                  // 64-k activation tiles per stage
  static constexpr int A_BYTES = F8 ? 0 : BM * BK * 2; // bf16 weight tile in shared memory
  static constexpr int RAW_BYTES = F8 ? BM * BKI : 0;  // E4M3 code tile, 128-byte rows
  static constexpr int B_BYTES = BN * BK * 2;          // one 64-k activation tile
  static constexpr int B_STAGE = B_BYTES * BT;
  // one ring stage as TMA fills it: the weight tile (bf16, or codes) and the activation tiles
  static constexpr int STAGE_BYTES = (F8 ? RAW_BYTES : A_BYTES) + B_STAGE * (SPLIT ? 2 : 1);
  static constexpr int CSTAGES = F8 ? 3 : 0;           // bf16 weight tiles in tensor memory
  static constexpr int A_TCOLS = BKI / 2;              // TMEM columns of one (two bf16 per column)
  static constexpr int A_COL = 2 * BN < 32 ? 32 : 2 * BN;   // first of them, after the accumulators
  // cluster split-K with small token tiles pushes each row's fp32 share into
  // the owning CTA: at most (csk - 1) * ceil(128 / csk) <= 120 rows arrive
  static constexpr bool PUSH = BN <= 32;
  static constexpr int PUSH_BYTES = PUSH ? 120 * BN * 4 : 0;
  // the head epilogue's exchange (16 tokens x 128 features + per-warp sums);
  // it never runs with the push path, so the two share one region
  static constexpr int XCH_BYTES = 128 * 16 * 4 + 4 * 16 * 4;
  static constexpr int XREG = PUSH_BYTES > XCH_BYTES ? PUSH_BYTES : XCH_BYTES;
  static constexpr int CTRL = 512;                     // mbarriers and flags
  // Small token tiles (weight streaming): ~100 KB of ring, so two GEMM CTAs
  // fit on one SM and, under programmatic dependent launch, the next GEMM's
  // CTAs become resident and stream their weights while this one drains
  // (152 x 5 stages in flight still exceed what HBM needs in flight).  F8
  // keeps the whole CTA within half an SM.  Large token tiles (tensor-bound):
  // one CTA per SM with a deeper ring.
  static constexpr int BUDGET = BN <= 32 ? (F8 ? (SMEM_PER_SM / 2 - 1024 - 1024 - CTRL - XREG) : 100 * 1024)
                                         : 200 * 1024;
  static constexpr int STAGES_RAW = BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : (STAGES_RAW < 2 ? 2 : STAGES_RAW);
  static constexpr int TMEM_COLS = F8 ? pow2_at_least(A_COL + CSTAGES * A_TCOLS) : (2 * BN < 32 ? 32 : 2 * BN);
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int SMEM = 1024 + RING + CTRL + XREG;
  static_assert((2 * STAGES + 2 * CSTAGES + 6) * 8 + 12 <= CTRL, "GEMM control block overflows");
  static_assert(RING >= BM * BN * 4, "the ring must hold one fp32 tile (cluster split-K share)");
  static_assert(!F8 || BN > 32 || 2 * (SMEM + 1024) <= SMEM_PER_SM, "two F8 CTAs must fit on one SM");
  // (two CTAs per SM only for small token tiles: the others take over 113 KB of shared memory)
  static_assert(TMEM_COLS <= 512 && (BN > 32 || 2 * TMEM_COLS <= 512), "tensor memory of the CTAs resident on one SM");
  static_assert(BN <= 32 || SMEM > SMEM_PER_SM / 2, "a large-tile CTA must not share its SM");
};

struct Params {
  int M, N, K;          // N: output rows of one group
  int n_groups, rtpg;   // groups, 128-row tiles per group
  size_t out_gstride;   // output elements between groups
  int tok_tiles, kbpt;
  int rt_total;         // weight row tiles of all groups (n_groups * rtpg): tile = tok * rt_total + rt
  long long total;     // tiles * kbpt
  int G;               // CTAs
  int csk;             // >1: cluster split-K, csk CTAs (one cluster) per tile
  int epi;
  void *out;
  int ldo;
  void *out_lo;        // low bf16 halves of a bf16 output, or null
  void *out2, *out2_lo;
  int ldo2;
  const float *bias;
  const void *cy, *cy_lo;   // EPI_CONV_PRE: convolved activation (bf16 hi / lo), row stride ldy
  const float *cy32;        // EPI_CONV_POST: convolved activation (fp32)
  int ldy, cS;              // EPI_CONV_*: row stride of y, block size
  HeadArgs head;            // EPI_HEADS
  const float *wscale[MAX_GROUPS];   // F8: per-row weight scales of each group
  float *partials;     // [G][2][BM][BN] row-major shares
  int *counters;       // [tiles]
  int *status;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ long long range_begin(long long total, int G, int c) {
  return static_cast<long long>(c) * total / G;
}
// CTA whose range contains iteration i (ranges [c*T/G, (c+1)*T/G)).
__device__ __forceinline__ int cta_of(long long i, long long total, int G) {
  return static_cast<int>(((i + 1) * G + total - 1) / total) - 1;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ void store_hl(__nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t i, float v) {
  const __nv_bfloat16 h = f2bf(v);
  hi[i] = h;
  if (lo) lo[i] = f2bf(v - bf2f(h));
}

// 8 consecutive channels of row r of the convolved activation (fp32 value).
__device__ __forceinline__ void conv_load8(const Params &p, bool post, int r, int c0, float (&y)[8]) {
  const size_t o = static_cast<size_t>(r) * p.ldy + c0;
  if (post) {
    const float4 a = *reinterpret_cast<const float4 *>(p.cy32 + o), b = *reinterpret_cast<const float4 *>(p.cy32 + o + 4);
    y[0] = a.x, y[1] = a.y, y[2] = a.z, y[3] = a.w, y[4] = b.x, y[5] = b.y, y[6] = b.z, y[7] = b.w;
  } else {
    const uint4 h = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.cy) + o);
    const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
    uint32_t lw[4] = {0u, 0u, 0u, 0u};
    if (p.cy_lo) {
      const uint4 l = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.cy_lo) + o);
      lw[0] = l.x, lw[1] = l.y, lw[2] = l.z, lw[3] = l.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      y[2 * i] = __uint_as_float(hw[i] << 16) + __uint_as_float(lw[i] << 16);
      y[2 * i + 1] = __uint_as_float(hw[i] & 0xFFFF0000u) + __uint_as_float(lw[i] & 0xFFFF0000u);
    }
  }
}

// DFlash-2 short convolution ("DFlash 2", Arquitectura del Sistema item 2)
// of 8 channels c0.. of one 16-channel group over the 16 token rows tok0..:
// out_j = y_j + a_j * y_j + b_j * y_{j-1}, y_{-1} = 0 at every block's first
// position (rows are consecutive positions of S-token blocks).  Pre sites
// store the bf16 hi / lo halves, post sites add into the fp32 residual.
// CB rows at a time: their loads (y, and the residual at post sites) are
// all issued before the first store, so the stores, which the compiler must
// assume may alias the loads, do not serialise them (CB = 1 in the variants
// capped at 96 registers).
template <int CB>
__device__ __noinline__ void conv_rows(const Params &p, bool post, const float (&a)[16], const float (&b)[16],
                                       int c0, int tok0) {
  float prev[8];
  if (tok0 < p.M && tok0 % p.cS != 0) {
    conv_load8(p, post, tok0 - 1, c0, prev);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) prev[k] = 0.f;
  }
#pragma unroll
  for (int i0 = 0; i0 < 16; i0 += CB) {
    float y[CB][8];
    float4 xr[CB][2];
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int r = tok0 + i0 + u;
      if (r < p.M) {
        conv_load8(p, post, r, c0, y[u]);
        if (post) {
          const float4 *x = reinterpret_cast<const float4 *>(static_cast<const float *>(p.out) +
                                                             static_cast<size_t>(r) * p.ldo + c0);
          xr[u][0] = __ldcg(x);
          xr[u][1] = __ldcg(x + 1);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int i = i0 + u, r = tok0 + i;
      if (r >= p.M) break;
      if (r % p.cS == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) prev[k] = 0.f;
      }
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = y[u][k] + a[i] * y[u][k] + b[i] * prev[k];
      const size_t off = static_cast<size_t>(r) * p.ldo + c0;
      if (post) {
        float4 *x = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + off);
        x[0] = make_float4(xr[u][0].x + o[0], xr[u][0].y + o[1], xr[u][0].z + o[2], xr[u][0].w + o[3]);
        x[1] = make_float4(xr[u][1].x + o[4], xr[u][1].y + o[5], xr[u][1].z + o[6], xr[u][1].w + o[7]);
      } else {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat16 h0 = f2bf(o[2 * k]), h1 = f2bf(o[2 * k + 1]);
          const __nv_bfloat16 l0 = f2bf(o[2 * k] - bf2f(h0)), l1 = f2bf(o[2 * k + 1] - bf2f(h1));
          hw[k] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                  (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
          lw[k] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                  (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
        }
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if (p.out_lo)
          *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out_lo) + off) =
              make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) prev[k] = y[u][k];
    }
  }
}

// EPI_HEADS: the tile is one attention head, row n = feature i (0..127) of
// head n / 128 of group g; v holds that feature for the 16 token rows tok0...
// Called by all 128 epilogue threads together, each with a different i (they
// meet at the epilogue's named barrier).  q / k heads: per-token RMSNorm over
// the head's 128 features ("DFlash" layer internals: Qwen3-style q/k norm),
// then RoPE on the pairs (i, i + 64) with the row's (cos, sin); the partner
// feature comes through shared memory.  The head is stored where the block
// attention reads it.  V^T destinations (columns = tokens) are written by
// lanes that cover 16 consecutive tokens of two features per instruction, so
// each warp store fills whole 32-byte sectors instead of 32 scattered bytes.
__device__ __noinline__ void heads_epi(const Params &p, float (&v)[16], int n, int g, int tok0, float *xch) {
  const HeadArgs &a = p.head;
  const int i = n & 127, head = n >> 7, lane = i & 31, q4 = i >> 5;
  const int kind = head < a.nq ? 0 : (head < a.nq + a.nkv ? 1 : 2);   // q, k, v
  const int h = kind == 0 ? head : (kind == 1 ? head - a.nq : head - a.nq - a.nkv);
  float *red = xch + 16 * 128;
  if (kind < 2) {
    if (a.norm) {
      const float gn = (kind == 0 ? a.gq : a.gk[g])[i];
      float ss[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) ss[t] = warp_sum(v[t] * v[t]);
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < 16; ++t) red[q4 * 16 + t] = ss[t];
      }
      epi_bar();
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float tot = red[t] + red[16 + t] + red[32 + t] + red[48 + t];
        v[t] *= rsqrtf(tot * (1.f / 128.f) + a.eps) * gn;
      }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) xch[t * 128 + i] = v[t];
    epi_bar();
    const bool lo = i < 64;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int row = tok0 + t < p.M ? tok0 + t : p.M - 1;
      const float2 cs = a.cs[static_cast<size_t>(row) * 64 + (i & 63)];
      const float o = xch[t * 128 + (i ^ 64)];
      v[t] = lo ? v[t] * cs.x - o * cs.y : v[t] * cs.x + o * cs.y;
    }
    epi_bar();   // the exchange is free again
  }
  __nv_bfloat16 *dst = nullptr;
  if (kind == 2) {
    // V^T: this warp's 32 features, 16 tokens, via shared memory; lane l
    // takes feature 32*q4 + 2k + l/16 of token l%16 in step k
#pragma unroll
    for (int t = 0; t < 16; ++t) xch[t * 128 + i] = v[t];
    __syncwarp();
    const int t = lane & 15, row = tok0 + t;
    if (row < p.M) {
      if (a.mode == 1) {
        const int b = row / a.S, j = row % a.S;
        dst = static_cast<__nv_bfloat16 *>(a.bv) + (static_cast<size_t>(b) * a.nkv + h) * 128 * 64 + j;
      } else {
        const int pg = a.tok_page[row];
        if (pg >= 0)
          dst = static_cast<__nv_bfloat16 *>(a.v_cache) + static_cast<size_t>(g) * a.layer_elems +
                (static_cast<size_t>(pg) * a.nkv + h) * 128 * 64 + a.tok_slot[row];
      }
    }
#pragma unroll 4
    for (int k = 0; k < 16; ++k) {
      const int f = q4 * 32 + 2 * k + (lane >> 4);
      const float x = xch[t * 128 + f];
      if (dst) dst[static_cast<size_t>(f) * 64] = f2bf(x);
    }
    __syncwarp();
    // block V^T below a block of 16: the PV k-step reads columns 0..15, so
    // the columns S..15 of each request get zeros (written by its first row)
    if (a.mode == 1 && a.S < 16) {
#pragma unroll
      for (int t2 = 0; t2 < 16; ++t2) {
        const int r2 = tok0 + t2;
        if (r2 < p.M && r2 % a.S == 0) {
          __nv_bfloat16 *z = static_cast<__nv_bfloat16 *>(a.bv) +
                             (static_cast<size_t>(r2 / a.S) * a.nkv + h) * 128 * 64 + static_cast<size_t>(i) * 64;
          for (int c = a.S; c < 16; ++c) z[c] = f2bf(0.f);
        }
      }
    }
    return;
  }
  // q rows and K rows: lanes cover consecutive features of one token
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int row = tok0 + t;
    if (row >= p.M) break;
    __nv_bfloat16 *o;
    if (a.mode == 1) {
      const int b = row / a.S, j = row % a.S;
      o = kind == 0 ? static_cast<__nv_bfloat16 *>(a.q) + static_cast<size_t>(row) * a.nq * 128 + h * 128 + i
                    : static_cast<__nv_bfloat16 *>(a.bk) + ((static_cast<size_t>(b) * a.nkv + h) * 64 + j) * 128 + i;
    } else {
      const int pg = a.tok_page[row];
      if (pg < 0) continue;
      o = static_cast<__nv_bfloat16 *>(a.k_cache) + static_cast<size_t>(g) * a.layer_elems +
          ((static_cast<size_t>(pg) * a.nkv + h) * 64 + a.tok_slot[row]) * 128 + i;
    }
    *o = f2bf(v[t]);
  }
}

// Apply the epilogue to 16 consecutive token columns of weight row n (ws:
// the group's FP8 row scales, or null).  CB: rows per load batch of the
// short-conv epilogue.
template <int CB>
__device__ __forceinline__ void finalize(const Params &p, float (&v)[16], int n, int tok0, size_t goff,
                                         const float *ws, int grp, float *xch) {
  const bool nok = n < p.N;
  if (ws) {
    const float sc = nok ? ws[n] : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] *= sc;
  }
  switch (p.epi) {
    case EPI_HEADS:
      heads_epi(p, v, n, grp, tok0, xch);
      break;
    case EPI_BF16: {
      __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out), *ol = static_cast<__nv_bfloat16 *>(p.out_lo);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (nok && tok0 + i < p.M) store_hl(o, ol, goff + static_cast<size_t>(tok0 + i) * p.ldo + n, v[i]);
    } break;
    case EPI_F32: {
      float *o = static_cast<float *>(p.out);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (nok && tok0 + i < p.M) o[goff + static_cast<size_t>(tok0 + i) * p.ldo + n] = v[i];
    } break;
    case EPI_ADD_F32: {
      // all 16 residual loads first (independent), then the adds and stores:
      // no chain of read-modify-write round trips
      float *o = static_cast<float *>(p.out);
      float r[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        r[i] = (nok && tok0 + i < p.M) ? __ldcg(o + goff + static_cast<size_t>(tok0 + i) * p.ldo + n) : 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (nok && tok0 + i < p.M) o[goff + static_cast<size_t>(tok0 + i) * p.ldo + n] = r[i] + v[i];
    } break;
    case EPI_SWIGLU: {
      __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out), *ol = static_cast<__nv_bfloat16 *>(p.out_lo);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float up = __shfl_xor_sync(0xffffffffu, v[i], 1);
        if (nok && !(n & 1) && tok0 + i < p.M)
          store_hl(o, ol, goff + static_cast<size_t>(tok0 + i) * p.ldo + (n >> 1), silu(v[i]) * up);
      }
    } break;
    case EPI_TANH_BIAS: {
      float *o = static_cast<float *>(p.out);
      const float b = nok ? p.bias[n] : 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (nok && tok0 + i < p.M) o[goff + static_cast<size_t>(tok0 + i) * p.ldo + n] = tanhf(v[i] + b);
    } break;
    case EPI_CONV_PRE:
    case EPI_CONV_POST: {
      // rows 2g / 2g+1 = tap a / tap b of channel group g, in neighbouring
      // lanes: exchange them, then each lane of the pair takes 8 of the
      // group's 16 channels
      const float bn = nok ? p.bias[n] : 0.f;
      float c[16], o[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i] = tanhf(v[i] + bn);
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = __shfl_xor_sync(0xffffffffu, c[i], 1);
      if (!nok) break;
      const bool odd = n & 1;
      const int c0 = (n >> 1) * 16 + (odd ? 8 : 0);
      if (odd)
        conv_rows<CB>(p, p.epi == EPI_CONV_POST, o, c, c0, tok0);
      else
        conv_rows<CB>(p, p.epi == EPI_CONV_POST, c, o, c0, tok0);
    } break;
    case EPI_F32_SPLIT: {
      float *o = static_cast<float *>(p.out);
      __nv_bfloat16 *o2 = static_cast<__nv_bfloat16 *>(p.out2), *o2l = static_cast<__nv_bfloat16 *>(p.out2_lo);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (nok && tok0 + i < p.M) {
          o[goff + static_cast<size_t>(tok0 + i) * p.ldo + n] = v[i];
          store_hl(o2, o2l, static_cast<size_t>(tok0 + i) * p.ldo2 + n, v[i]);
        }
    } break;
    default:
      break;
  }
}

// Four E4M3 codes -> four bf16 values, exact.  The code's bits, moved into
// bf16 fields (sign to bit 15, exponent and mantissa to bits 4..10), encode
// code * 2^-120 for every code (normal, subnormal, zero: bf16's exponent
// bias is 120 more than E4M3's and both fields line up); one bf16 multiply by
// 2^120 (0x7B80) restores the value.  Each 16-bit half is built by one byte
// permute - the code byte low, its sign replicated into the high byte
// (selector bit 3) - one shift by 4 and one mask keeping bits 4..10 and 15.
// NaN codes (S.1111.111) are not weights.  Returns the two bf16x2 words of
// bytes (0,1) and (2,3).
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  uint32_t lo, hi;
  asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(lo) : "r"(w));   // [sign(b1), b1, sign(b0), b0]
  asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(hi) : "r"(w));   // [sign(b3), b3, sign(b2), b2]
  lo = (lo << 4) & 0x87F087F0u;
  hi = (hi << 4) & 0x87F087F0u;
  uint2 r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r.x) : "r"(lo), "r"(0x7B807B80u));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r.y) : "r"(hi), "r"(0x7B807B80u));
  return r;
}

// EPI_ADD_F32 for 16 token columns whose residual values r were loaded
// earlier (before the accumulator was ready): out = r + scale * v.
__device__ __forceinline__ void finalize_add_pre(const Params &p, float (&v)[16], const float (&r)[16], int n,
                                                 int tok0, size_t goff, const float *ws) {
  const bool nok = n < p.N;
  const float sc = ws && nok ? ws[n] : 1.f;
  float *o = static_cast<float *>(p.out);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (nok && tok0 + i < p.M) o[goff + static_cast<size_t>(tok0 + i) * p.ldo + n] = r[i] + sc * v[i];
}

__global__ void e4m3_to_bf16_kernel(const uint32_t *codes, int n4, uint2 *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n4) out[i] = e4m3x4_to_bf16x4(codes[i]);
}

template <int BN, bool SPLIT, bool F8>
__global__ void __launch_bounds__(Cfg<BN, SPLIT, F8>::NT, BN <= 32 ? 2 : 1)   // small tiles: two CTAs per SM
    gemm_tc_kernel(const __grid_constant__ WMaps wm, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmXlo, const Params p) {
  using C = Cfg<BN, SPLIT, F8>;
  constexpr int CB_ = (F8 && BN <= 32) ? 1 : 4;   // short-conv load batch (96-register variants: 1)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *base = smem_raw + pad;
  // [bf16 weight tiles (not F8)] [activation tiles] [low halves (SPLIT)] [code tiles (F8)]
  uint8_t *sA = base;
  uint8_t *sB = base + C::STAGES * C::A_BYTES;
  uint8_t *sBl = sB + C::STAGES * C::B_STAGE;   // low halves (SPLIT only)
  uint8_t *sRaw = sBl + (SPLIT ? C::STAGES * C::B_STAGE : 0);
  uint64_t *full = reinterpret_cast<uint64_t *>(base + C::RING);
  uint64_t *empty = full + C::STAGES;
  uint64_t *tfull = empty + C::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint64_t *rbar = drain + 1;   // cluster split-K (push): shares of the other CTAs have arrived
  uint64_t *cfull = rbar + 1;   // F8: converted weight tile ready
  uint64_t *cempty = cfull + C::CSTAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cempty + C::CSTAGES);
  float *spush = reinterpret_cast<float *>(base + C::RING + C::CTRL);   // push shares, or ...
  float *xch = spush;                                                      // ... the head epilogue's exchange
  // the head epilogue needs a whole tile in one CTA: no pushing of rows to
  // the other CTAs of a cluster (its shares are pulled by rank 0 instead)
  const bool push = C::PUSH && p.epi != EPI_HEADS;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *bcast = reinterpret_cast<int *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::CSTAGES; ++s) {
      mbar_init(&cfull[s], C::CONV_WARPS);   // every converter warp
      mbar_init(&cempty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 4);
    mbar_init(&tempty[1], 4);
    mbar_init(drain, 1);
    mbar_init(rbar, p.csk > 1 ? p.csk - 1 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.n_groups; ++g) tma_prefetch_desc(&wm.m[g]);
    tma_prefetch_desc(&tmX);
    if (SPLIT) tma_prefetch_desc(&tmXlo);
  }
  grid_dep_launch();   // the next kernel may be scheduled now; it waits for this grid itself
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (push && p.csk > 1) cluster_sync();   // every CTA's barriers exist before any remote arrive

  // The activations, outputs and stream-K scratch are produced / consumed by
  // the neighbouring kernels of the step: only the weight stream may start
  // before the previous grid has completed (programmatic dependent launch).
  // stream-K: one contiguous range of the (tile, k-block) space per CTA;
  // cluster split-K: the csk CTAs of a cluster split one tile's k-blocks
  long long begin, end;
  if (p.csk > 1) {
    const long long tile = blockIdx.x / p.csk, r = blockIdx.x % p.csk;
    begin = tile * p.kbpt + r * p.kbpt / p.csk;
    end = tile * p.kbpt + (r + 1) * p.kbpt / p.csk;
  } else {
    begin = range_begin(p.total, p.G, blockIdx.x);
    end = range_begin(p.total, p.G, blockIdx.x + 1);
  }
  const int first_tile = static_cast<int>(begin / p.kbpt);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // one token tile: every weight tile is read once, evict it first; with
      // several, the readers of the other token tiles follow within the ring
      // depth, so no hint
      const uint64_t pol_w = policy_evict_first();
      const bool hint_w = p.tok_tiles == 1;
      auto load_w = [&](void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y) {
        if (hint_w)
          tma_load_2d_hint(dst, m, bar, x, y, pol_w);
        else
          tma_load_2d(dst, m, bar, x, y);
      };
      const long long n_my = end - begin;
      // iteration -> (group, weight row, token row, k-block), advanced
      // incrementally: no integer division in the issue loop
      struct Iter {
        int kb, tok, rtin, g;
      };
      Iter it0;
      {
        const int tile = static_cast<int>(begin / p.kbpt);
        it0.kb = static_cast<int>(begin - static_cast<long long>(tile) * p.kbpt);
        it0.tok = tile / p.rt_total;
        const int rt = tile - it0.tok * p.rt_total;
        it0.g = rt / p.rtpg;
        it0.rtin = rt - it0.g * p.rtpg;
      }
      auto advance = [&](Iter &q) {
        if (++q.kb == p.kbpt) {
          q.kb = 0;
          if (++q.rtin == p.rtpg) {
            q.rtin = 0;
            if (++q.g == p.n_groups) {
              q.g = 0;
              ++q.tok;
            }
          }
        }
      };
      auto coords = [&](const Iter &q, int &g, int &row0, int &tok0, int &kb) {
        g = q.g;
        row0 = q.rtin * BM;
        tok0 = q.tok * BN;
        kb = q.kb;
      };
      // weights of the first ring slots depend on nothing: stream them while
      // the previous kernel finishes, then wait for it before the activations
      const int n_pre = static_cast<int>(n_my < C::STAGES ? n_my : C::STAGES);
      Iter q = it0;
      for (int i = 0; i < n_pre; ++i, advance(q)) {
        int g, row0, tok0, kb;
        coords(q, g, row0, tok0, kb);
        mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
        load_w(F8 ? sRaw + i * C::RAW_BYTES : sA + i * C::A_BYTES, &wm.m[g], &full[i], kb * C::BKI, row0);
      }
      grid_dep_wait();
      q = it0;
      for (int i = 0; i < n_pre; ++i, advance(q)) {
        int g, row0, tok0, kb;
        coords(q, g, row0, tok0, kb);
#pragma unroll
        for (int t = 0; t < C::BT; ++t) {
          tma_load_2d(sB + i * C::B_STAGE + t * C::B_BYTES, &tmX, &full[i], kb * C::BKI + t * BK, tok0);
          if (SPLIT) tma_load_2d(sBl + i * C::B_STAGE + t * C::B_BYTES, &tmXlo, &full[i], kb * C::BKI + t * BK, tok0);
        }
      }
      uint32_t stage = n_pre % C::STAGES, phase = (n_pre == C::STAGES) ? 1u : 0u;
      long long issued = n_pre;
      bool ok = true;
      for (long long i = n_pre; i < n_my; ++i, advance(q)) {
        int g, row0, tok0, kb;
        coords(q, g, row0, tok0, kb);
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
        load_w(F8 ? sRaw + stage * C::RAW_BYTES : sA + stage * C::A_BYTES, &wm.m[g], &full[stage], kb * C::BKI, row0);
#pragma unroll
        for (int t = 0; t < C::BT; ++t) {
          tma_load_2d(sB + stage * C::B_STAGE + t * C::B_BYTES, &tmX, &full[stage], kb * C::BKI + t * BK, tok0);
          if (SPLIT)
            tma_load_2d(sBl + stage * C::B_STAGE + t * C::B_BYTES, &tmXlo, &full[stage], kb * C::BKI + t * BK, tok0);
        }
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        // let every issued copy land before the CTA's shared memory goes away
        for (int s = 0; s < C::STAGES; ++s) {
          if (issued <= s) break;
          const long long last = s + C::STAGES * ((issued - 1 - s) / C::STAGES);
          mbar_wait(&full[s], static_cast<uint32_t>((last / C::STAGES) & 1), nullptr, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      uint32_t stage = 0, phase = 0;
      uint32_t cst = 0, cph = 0;   // F8: converted-tile ring
      int seg = 0;
      bool ok = true;
      for (long long it = begin; it < end && ok; ++seg) {
        const int kb0 = static_cast<int>(it % p.kbpt);
        const int kb1 = static_cast<int>((kb0 + (end - it) < p.kbpt ? kb0 + (end - it) : p.kbpt));
        const int buf = seg & 1;
        if (!mbar_wait(&tempty[buf], static_cast<uint32_t>(((seg >> 1) & 1) ^ 1), abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns) ||
              (F8 && !mbar_wait(&cfull[cst], cph, abort_flag, p.timeout_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b0 = smem_u32(sB + stage * C::B_STAGE);
          const uint32_t bl = smem_u32(sBl + stage * C::B_STAGE);
          if (F8) {
            // A: the converted tile in tensor memory, 8 columns per K = 16 step
            const uint32_t at = tmem + static_cast<uint32_t>(C::A_COL + cst * C::A_TCOLS);
#pragma unroll
            for (int k = 0; k < C::BKI / UK; ++k) {
              const uint32_t boff = (k / (BK / UK)) * C::B_BYTES + (k % (BK / UK)) * UK * 2;
              umma_bf16_ts(d, at + k * (UK / 2), sdesc_k_sw128(b0 + boff), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
              if (SPLIT) umma_bf16_ts(d, at + k * (UK / 2), sdesc_k_sw128(bl + boff), idesc, 1u);
            }
          } else {
            const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
#pragma unroll
            for (int k = 0; k < BK / UK; ++k) {
              const uint64_t ad = sdesc_k_sw128(a0 + k * UK * 2);
              umma_bf16(d, ad, sdesc_k_sw128(b0 + k * UK * 2), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
              if (SPLIT) umma_bf16(d, ad, sdesc_k_sw128(bl + k * UK * 2), idesc, 1u);
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (F8) {
            umma_commit(&cempty[cst]);
            if (++cst == C::CSTAGES) {
              cst = 0;
              cph ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
        it += kb1 - kb0;
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        umma_commit(drain);   // all issued MMAs retire before TMEM is freed
        mbar_wait(drain, 0, nullptr, p.timeout_ns);
      }
    }
  } else if (F8 && warp >= 6) {
    // ------------------------------------------------------------ FP8 weight converters
    // Code tile: [128 rows][128 codes], 128-byte rows whose 16-byte chunk j
    // sits at j ^ (row & 7) (TMA's 128-byte swizzle: eight consecutive rows
    // read at one chunk column touch every bank once).  Warp w owns TMEM lane
    // quarter w & 3: lane i converts row 32 (w & 3) + i and stores its 128
    // bf16 values into 64 consecutive columns of its lane (lower k in the low
    // half of each column), the A layout of the MMA.
    const int qd = warp & 3, r = qd * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32) << 16) + static_cast<uint32_t>(C::A_COL);
    uint32_t stage = 0, phase = 0, cst = 0, cph = 0;
    bool ok = true;
    for (long long i = begin; i < end && ok; ++i) {
      if (!mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns) ||
          !mbar_wait(&cempty[cst], cph ^ 1u, abort_flag, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();   // the MMAs that read this TMEM tile have completed
      const uint8_t *row = sRaw + stage * C::RAW_BYTES + r * 128;
      const uint32_t tcol = lane_base + static_cast<uint32_t>(cst * C::A_TCOLS);
#pragma unroll
      for (int j = 0; j < C::BKI / 16; ++j) {
        const uint4 c = *reinterpret_cast<const uint4 *>(row + ((j ^ (r & 7)) << 4));
        const uint2 a = e4m3x4_to_bf16x4(c.x), b = e4m3x4_to_bf16x4(c.y), e = e4m3x4_to_bf16x4(c.z),
                    f = e4m3x4_to_bf16x4(c.w);
        const uint32_t o[8] = {a.x, a.y, b.x, b.y, e.x, e.y, f.x, f.y};
        tmem_st8_nw(tcol + j * 8, o);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&cfull[cst]);
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      if (++cst == C::CSTAGES) {
        cst = 0;
        cph ^= 1u;
      }
    }
    if (!ok) {
      if (lane == 0) report(p.status, DFLASH_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int r = q * 32 + lane;         // weight row within the tile
    const int et = threadIdx.x - 64;     // 0..127
    grid_dep_wait();                     // outputs / scratch are shared with the previous kernel
    if (p.epi == EPI_HEADS && p.head.mode == 2 && blockIdx.x == 0)
      // context injection: the requests' new lengths (the feature kernel saved
      // the old ones; nothing reads ctx_len_in after it)
      for (int b = et; b < p.head.B; b += 128)
        p.head.ctx_out[b] = p.head.ctx_saved[b] + (p.head.cu_new[b + 1] - p.head.cu_new[b]);
    int seg = 0;
    for (long long it = begin; it < end; ++seg) {
      const int tile = static_cast<int>(it / p.kbpt);
      const int kb0 = static_cast<int>(it % p.kbpt);
      const int kb1 = static_cast<int>((kb0 + (end - it) < p.kbpt ? kb0 + (end - it) : p.kbpt));
      const int buf = seg & 1;
      // One 16-token column group with a residual add: load the residual of
      // the row this thread will finalise (whole tile, or its own rows of a
      // cluster split-K tile) while the MMAs still run - one L2 round trip
      // off the GEMM's tail.
      float rpre[16];
      bool have_pre = false;
      if (BN == 16 && p.epi == EPI_ADD_F32) {
        const bool whole_t = kb0 == 0 && kb1 == p.kbpt;
        const bool owner = push && p.csk > 1 && ((r + 1) * p.csk - 1) / BM == static_cast<int>(cluster_ctarank());
        if (whole_t || owner) {
          const int rt0 = tile % p.rt_total;
          const int n0 = (rt0 % p.rtpg) * BM + r, t0 = (tile / p.rt_total) * BN;
          const size_t g0 = static_cast<size_t>(rt0 / p.rtpg) * p.out_gstride;
          const float *o = static_cast<const float *>(p.out);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            rpre[i] = (n0 < p.N && t0 + i < p.M) ? __ldcg(o + g0 + static_cast<size_t>(t0 + i) * p.ldo + n0) : 0.f;
          have_pre = true;
        }
      }
      const bool got = mbar_wait(&tfull[buf], static_cast<uint32_t>((seg >> 1) & 1), abort_flag, p.timeout_ns);
      // one uniform decision for all 128 epilogue threads (they meet at named barriers below)
      if (bar_or(1, 128, !got || *abort_flag)) {
        if (et == 0) report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int rt = tile % p.rt_total;
      const int n = (rt % p.rtpg) * BM + r;                       // row within its group
      const size_t goff = static_cast<size_t>(rt / p.rtpg) * p.out_gstride;
      const float *wsg = F8 ? p.wscale[rt / p.rtpg] : nullptr;
      const int tok0 = (tile / p.rt_total) * BN;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      float v[16];
      if (kb0 == 0 && kb1 == p.kbpt) {
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
          if (have_pre)
            finalize_add_pre(p, v, rpre, n, tok0 + c * 16, goff, wsg);
          else
            finalize<CB_>(p, v, n, tok0 + c * 16, goff, wsg, rt / p.rtpg, xch);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      } else if (push && p.csk > 1) {
        // cluster split-K, small token tile: each row's fp32 share goes straight
        // into the shared memory of the CTA that finalises that row (rows
        // [k*BM/csk, (k+1)*BM/csk) belong to rank k); one release arrive per
        // peer, then the owner sums the csk shares in rank order
        const int S = p.csk, rank = static_cast<int>(cluster_ctarank());
        const int o = ((r + 1) * S - 1) / BM;
        const int o_r0 = o * BM / S, o_rows = (o + 1) * BM / S - o_r0;
        float own[BN];
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) own[c * 16 + i] = v[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (o != rank) {
          const int slot = rank < o ? rank : rank - 1;
          const uint32_t a = dsmem_addr(spush + (static_cast<size_t>(slot) * o_rows + (r - o_r0)) * BN,
                                        static_cast<uint32_t>(o));
#pragma unroll
          for (int j = 0; j < BN / 4; ++j)
            st_dsmem_f4(a + 16 * j, make_float4(own[4 * j], own[4 * j + 1], own[4 * j + 2], own[4 * j + 3]));
        }
        fence_acq_rel_cluster();
        epi_bar();   // every push of this CTA is issued and fenced
        if (et < S && et != rank) mbar_arrive_remote(dsmem_addr(rbar, static_cast<uint32_t>(et)));
        const bool got_all = mbar_wait_cluster(rbar, 0, abort_flag, p.timeout_ns);
        if (!got_all) {
          if (et == 0) report(p.status, DFLASH_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        const bool mine = o == rank;
        const int my_rows = (rank + 1) * BM / S - rank * BM / S, my_r0 = rank * BM / S;
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
          for (int k = 0; k < S; ++k) {   // rank order: deterministic
            if (k == rank) {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] += own[c * 16 + i];
            } else if (mine) {
              const int slot = k < rank ? k : k - 1;
              const float4 *src = reinterpret_cast<const float4 *>(
                  spush + (static_cast<size_t>(slot) * my_rows + (r - my_r0)) * BN + c * 16);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 x = src[i];
                v[4 * i] += x.x;
                v[4 * i + 1] += x.y;
                v[4 * i + 2] += x.z;
                v[4 * i + 3] += x.w;
              }
            }
          }
          if (have_pre && mine)
            finalize_add_pre(p, v, rpre, n, tok0 + c * 16, goff, wsg);
          else
            finalize<CB_>(p, v, mine ? n : p.N, tok0 + c * 16, goff, wsg, rt / p.rtpg, xch);   // n >= N: not this CTA's row
        }
      } else if (p.csk > 1) {
        // cluster split-K: this CTA's fp32 share into its own smem, row-major
        // (the ring is idle: every stage has been consumed); the cluster
        // reduces it on chip after the main loop
        float *sp = reinterpret_cast<float *>(sA) + static_cast<size_t>(r) * BN;
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
          float4 *s4 = reinterpret_cast<float4 *>(sp + c * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) s4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      } else {
        // partial tile: this CTA's fp32 share goes to its slot, row-major
        // (each thread writes its row's BN columns as float4); the CTA that
        // completes the tile's k-range sums all shares in CTA order
        const int slot = (tile == first_tile) ? 0 : 1;
        float *P = p.partials + (static_cast<size_t>(blockIdx.x) * 2 + slot) * (BM * BN) + static_cast<size_t>(r) * BN;
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
          float4 *P4 = reinterpret_cast<float4 *>(P + c * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) __stcg(P4 + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        epi_bar();   // every share of this CTA is written ...
        if (et == 0) {
          __threadfence();   // ... and, through the barrier, visible before the count moves
          const int nk = kb1 - kb0;
          const int old = atomicAdd(&p.counters[tile], nk);
          const int last = (old + nk == p.kbpt) ? 1 : 0;
          if (last) {
            p.counters[tile] = 0;   // self-cleaning for the next launch
            __threadfence();
          }
          *bcast = last;
        }
        epi_bar();
        if (*bcast) {
          const long long t_beg = static_cast<long long>(tile) * p.kbpt;
          const int c_lo = cta_of(t_beg, p.total, p.G);
          const int c_hi = cta_of(t_beg + p.kbpt - 1, p.total, p.G);
          // only the first contributor can have started in an earlier tile
          const int slot_lo = range_begin(p.total, p.G, c_lo) < t_beg ? 1 : 0;
          for (int c = 0; c < BN / 16; ++c) {
            float4 acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cc0 = c_lo; cc0 <= c_hi; cc0 += 4) {
              float4 t[4][4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {   // up to 4 contributors' loads in flight
                const int cc = cc0 + u;
                const float4 *Q4 = reinterpret_cast<const float4 *>(
                    p.partials + (static_cast<size_t>(cc) * 2 + (cc == c_lo ? slot_lo : 0)) * (BM * BN) +
                    static_cast<size_t>(r) * BN + c * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i) t[u][i] = cc <= c_hi ? __ldcg(Q4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u)   // summed in contributor order: deterministic
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  acc[i].x += t[u][i].x;
                  acc[i].y += t[u][i].y;
                  acc[i].z += t[u][i].z;
                  acc[i].w += t[u][i].w;
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[4 * i] = acc[i].x;
              v[4 * i + 1] = acc[i].y;
              v[4 * i + 2] = acc[i].z;
              v[4 * i + 3] = acc[i].w;
            }
            finalize<CB_>(p, v, n, tok0 + c * 16, goff, wsg, rt / p.rtpg, xch);
          }
        }
        epi_bar();
      }
      it += kb1 - kb0;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);

  if (!push && p.csk > 1) {
    // ---- cluster split-K reduction through distributed shared memory: CTA
    // r finalises tile rows [r*BM/csk, (r+1)*BM/csk) summing the csk shares in
    // rank order (deterministic); lanes hold consecutive rows (coalesced
    // stores, SwiGLU row pairs in neighbouring lanes)
    cluster_sync();
    if (warp >= 2 && warp < 6) {   // the epilogue warps
      const int et = threadIdx.x - 64;
      const int rank = static_cast<int>(cluster_ctarank());
      // head epilogue: rank 0 finalises the whole tile (one head)
      const bool heads = p.epi == EPI_HEADS;
      const int r0 = heads ? 0 : rank * BM / p.csk;
      const int rows = heads ? (rank == 0 ? BM : 0) : (rank + 1) * BM / p.csk - r0;
      const int tasks = rows * (BN / 16);
      const int tile = first_tile;
      const int rt = tile % p.rt_total;
      const size_t goff = static_cast<size_t>(rt / p.rtpg) * p.out_gstride;
      const float *wsg = F8 ? p.wscale[rt / p.rtpg] : nullptr;
      const int tokt = (tile / p.rt_total) * BN;
      const float *sp = reinterpret_cast<const float *>(sA);
      for (int t0 = 0; t0 < tasks; t0 += 128) {   // every thread takes each round (shuffles in SwiGLU)
        const int task = t0 + et;
        const bool valid = task < tasks;
        const int row = r0 + (valid ? task % rows : 0), grp = valid ? task / rows : 0;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        if (valid) {
          for (int k = 0; k < p.csk; ++k) {
            const uint32_t a = dsmem_addr(sp + static_cast<size_t>(row) * BN + grp * 16, static_cast<uint32_t>(k));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 x = ld_dsmem_f4(a + 16 * i);
              v[4 * i] += x.x;
              v[4 * i + 1] += x.y;
              v[4 * i + 2] += x.z;
              v[4 * i + 3] += x.w;
            }
          }
        }
        const int n = valid ? (rt % p.rtpg) * BM + row : p.N;   // n >= N: nothing stored
        finalize<CB_>(p, v, n, tokt + grp * 16, goff, wsg, rt / p.rtpg, xch);
      }
    }
    cluster_sync();   // nobody leaves while others still read its share
  }
}

// Kernel attributes (dynamic shared memory; for small tiles the whole
// unified L1 / shared array as shared memory so that two CTAs can be
// resident per SM) set once; returns the CTAs of the variant resident per SM
// by registers and shared memory, or a negative error code.
template <int BN, bool SPLIT, bool F8>
int setup_device(int dev) {
  using C = Cfg<BN, SPLIT, F8>;
  if (int e = cuda_check(cudaFuncSetAttribute(gemm_tc_kernel<BN, SPLIT, F8>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM),
                         "gemm smem attribute"))
    return e;
  if (BN <= 32)   // small tiles: two CTAs per SM need the whole array as shared memory
    if (int e = cuda_check(cudaFuncSetAttribute(gemm_tc_kernel<BN, SPLIT, F8>,
                                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                                cudaSharedmemCarveoutMaxShared),
                           "gemm carveout attribute"))
      return e;
  // resident CTAs per SM from the kernel's registers and shared memory
  cudaFuncAttributes fa = {};
  int smem_sm = 0, resv = 0;
  if (int e = cuda_check(cudaFuncGetAttributes(&fa, gemm_tc_kernel<BN, SPLIT, F8>), "gemm attributes")) return e;
  if (int e = cuda_check(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev),
                         "shared memory per SM"))
    return e;
  if (int e = cuda_check(cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev),
                         "reserved shared memory"))
    return e;
  const int warp_regs = ((fa.numRegs * 32 + 255) / 256) * 256;   // allocated per warp in 256-register units
  const int by_regs = 65536 / (warp_regs * (C::NT / 32));
  const int by_smem = smem_sm / (C::SMEM + resv);
  const int n = std::min(std::min(by_regs, by_smem), 2048 / C::NT);
  return n > 0 ? n : 1;
}

// Per device, once (attributes are per device; concurrent first calls only
// repeat the same idempotent setup): CTAs of the variant resident per SM, or
// a negative error code.
template <int BN, bool SPLIT, bool F8>
int setup() {
  constexpr int MAX_DEV = 64;
  static std::atomic<int> per_dev[MAX_DEV];
  int dev = 0;
  if (int e = cuda_check(cudaGetDevice(&dev), "device")) return e;
  if (dev < 0 || dev >= MAX_DEV) return set_error(DFLASH_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, MAX_DEV);
  int v = per_dev[dev].load(std::memory_order_acquire);
  if (v == 0) {
    v = setup_device<BN, SPLIT, F8>(dev);
    if (v < 0) return v;
    per_dev[dev].store(v, std::memory_order_release);
  }
  return v;
}

template <int BN, bool SPLIT, bool F8>
int launch(const Launch &lc, const WMaps &tW, const CUtensorMap &tX, const CUtensorMap &tXl, const Params &p) {
  using C = Cfg<BN, SPLIT, F8>;
  if (int e = setup<BN, SPLIT, F8>(); e < 0) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(C::NT);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(p.csk > 1 ? p.csk : 1);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cuda_check(cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, SPLIT, F8>, tW, tX, tXl, p), "gemm launch");
}

template <bool SPLIT, bool F8>
int launch_bn(int BN, const Launch &lc, const WMaps &tW, const CUtensorMap &tX, const CUtensorMap &tXl,
              const Params &p) {
  switch (BN) {
    case 16: return launch<16, SPLIT, F8>(lc, tW, tX, tXl, p);
    case 32: return launch<32, SPLIT, F8>(lc, tW, tX, tXl, p);
    case 64: return launch<64, SPLIT, F8>(lc, tW, tX, tXl, p);
    case 128: return launch<128, SPLIT, F8>(lc, tW, tX, tXl, p);
    default: return launch<F8 ? 128 : 256, SPLIT, F8>(lc, tW, tX, tXl, p);   // FP8 tiles stop at 128
  }
}

// CTAs of the variant resident per SM (for the decomposition), or < 0.
template <bool SPLIT, bool F8>
int per_sm_of(int BN) {
  switch (BN) {
    case 16: return setup<16, SPLIT, F8>();
    case 32: return setup<32, SPLIT, F8>();
    case 64: return setup<64, SPLIT, F8>();
    case 128: return setup<128, SPLIT, F8>();
    default: return setup<F8 ? 128 : 256, SPLIT, F8>();
  }
}

}  // namespace

int e4m3_to_bf16(const Launch &lc, const void *codes, int n, void *out) {
  if (n <= 0 || n % 4 || !codes || !out || (reinterpret_cast<uintptr_t>(codes) & 3) ||
      (reinterpret_cast<uintptr_t>(out) & 7))
    return set_error(DFLASH_ERR_ARG, "e4m3_to_bf16: n must be a positive multiple of 4, buffers aligned");
  const int n4 = n / 4;
  e4m3_to_bf16_kernel<<<(n4 + 255) / 256, 256, 0, lc.stream>>>(static_cast<const uint32_t *>(codes), n4,
                                                               static_cast<uint2 *>(out));
  return cuda_check(cudaGetLastError(), "e4m3_to_bf16 launch");
}

// Token tile: the smallest that covers M; with split activations at most 128
// so that a stage (weights + two activation tiles) still leaves a 4-deep
// ring in shared memory, and with FP8 weights at most 128 so that the bf16
// weight tiles fit in tensor memory beside the accumulators.
int gemm_token_tile(int M, bool split, bool f8) {
  return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : (M <= 128 || split || f8) ? 128 : 256;
}

GemmPlan gemm_plan(int M, int N, int K, int n_groups, bool f8, bool split, bool paired, int per_sm, int num_sms,
                   int gemm_ctas) {
  GemmPlan pl = {};
  pl.BN = gemm_token_tile(M, split, f8);
  pl.rtpg = (N + BM - 1) / BM;
  pl.tok_tiles = (M + pl.BN - 1) / pl.BN;
  const int bki = f8 ? 2 * BK : BK;   // k per ring stage
  pl.kbpt = (K + bki - 1) / bki;
  pl.tiles = static_cast<long long>(pl.rtpg) * (n_groups > 1 ? n_groups : 1) * pl.tok_tiles;
  pl.total = pl.tiles * pl.kbpt;
  // Resident CTA slots (the variant's occupancy, at most two per SM).  CTAs:
  // one per SM (FP8 weights: one per slot, so that two threads issue MMAs
  // on each SM), at least 4 k-blocks each, and no tile cut into so many
  // pieces that its fixup (the last piece sums the others' fp32 partials
  // from L2) reads more than 256 KB: 32 partials at BN = 16, 4 at BN = 128
  const int slots = std::min(per_sm, 2) * num_sms;
  const int cap = gemm_ctas > 0 ? gemm_ctas : (f8 ? slots : num_sms);
  const int max_parts = std::max(2, (256 * 1024) / (BM * pl.BN * 4));
  const int min_kb = std::max(4, (pl.kbpt + max_parts - 1) / max_parts);
  pl.G = static_cast<int>(std::max<long long>(1, std::min<long long>(cap, (pl.total + min_kb - 1) / min_kb)));
  // More tiles than SMs but no more than the resident slots: one whole tile
  // per CTA, some SMs running two.  Cutting them over the CTAs would split
  // nearly every tile and put a global fixup on the tail of a
  // weight-streaming GEMM.
  if (gemm_ctas == 0 && pl.tiles > num_sms && pl.tiles <= slots) pl.G = static_cast<int>(pl.tiles);
  // Few tiles (at most half the SMs): cluster split-K instead, csk CTAs per
  // tile reducing through distributed shared memory - no global round trips
  // (fence, counter atomic, partial loads: ~2 us each here) on the GEMM's
  // tail.  The test hook (gemm_ctas) keeps stream-K.
  pl.csk = 1;
  if (gemm_ctas == 0 && pl.tiles * 2 <= cap) {
    // at most 8 CTAs, and about 8 k-blocks or more each (short ranges are
    // all pipeline fill; at least 2-way where the k-range allows)
    long long s = std::min<long long>(std::min<long long>(8, cap / pl.tiles),
                                      std::min<long long>(pl.kbpt, std::max<long long>(2, pl.kbpt / 8)));
    // SwiGLU and the short conv pair rows 2i / 2i+1 in neighbouring lanes:
    // row ranges must be even-aligned, so a power-of-two cluster there
    if (paired)
      while (s & (s - 1)) --s;
    if (s >= 2) {
      pl.csk = static_cast<int>(s);
      pl.G = static_cast<int>(pl.tiles * s);
    }
  }
  return pl;
}

int gemm_bf16(const Launch &lc, const GemmOp &op, const GemmScratch &sc) {
  const int M = op.M, N = op.N, K = op.K;
  const char *name = op.name;
  if (M <= 0 || N <= 0 || K <= 0) return DFLASH_OK;
  if ((!op.W && op.n_groups <= 1) || !op.X || (!op.out && op.epi != EPI_HEADS))
    return set_error(DFLASH_ERR_ARG, "gemm %s: null operand", name);
  const uintptr_t al = reinterpret_cast<uintptr_t>(op.W) | reinterpret_cast<uintptr_t>(op.X) |
                       reinterpret_cast<uintptr_t>(op.X_lo);
  const bool f8 = op.w_fp8;
  const int wbytes = f8 ? 1 : 2;   // bytes per weight element
  if ((al & 15) || (op.ldw * wbytes) % 16 || (op.ldx * 2) % 16)
    return set_error(DFLASH_ERR_ALIGN, "gemm %s: operands / row strides must be 16-byte aligned", name);
  int epi = op.epi == EPI_STORE_T ? EPI_BF16 : op.epi;
  if (epi == EPI_F32_SPLIT && !op.out2) return set_error(DFLASH_ERR_ARG, "gemm %s: split output missing", name);
  const bool split = op.X_lo != nullptr;
  const int n_groups = op.n_groups > 1 ? op.n_groups : 1;
  const int BN = gemm_token_tile(M, split, f8);
  if (n_groups > MAX_GROUPS || (n_groups > 1 && N % BM))
    return set_error(DFLASH_ERR_UNSUPPORTED, "gemm %s: at most %d groups of a multiple of %d rows", name, MAX_GROUPS, BM);
  const int per_sm = f8 ? (split ? per_sm_of<true, true>(BN) : per_sm_of<false, true>(BN))
                        : (split ? per_sm_of<true, false>(BN) : per_sm_of<false, false>(BN));
  if (per_sm < 0) return per_sm;
  const bool conv = epi == EPI_CONV_PRE || epi == EPI_CONV_POST;
  if (conv) {
    const uintptr_t ya = reinterpret_cast<uintptr_t>(op.conv_y) | reinterpret_cast<uintptr_t>(op.conv_y_lo) |
                         reinterpret_cast<uintptr_t>(op.conv_y32) | reinterpret_cast<uintptr_t>(op.out) |
                         reinterpret_cast<uintptr_t>(op.out_lo);
    if (N % 2 || !op.bias || op.conv_S < 1 || op.ldy % 8 || op.ldo % 8 || (ya & 31) ||
        (epi == EPI_CONV_PRE ? !op.conv_y : !op.conv_y32))
      return set_error(DFLASH_ERR_ARG, "gemm %s: short-conv epilogue operands", name);
  }
  if (epi == EPI_HEADS) {
    const HeadArgs &h = op.head;
    const int heads = h.mode == 1 ? h.nq + 2 * h.nkv : 2 * h.nkv;
    const bool ok = (h.mode == 1 || h.mode == 2) && h.nkv > 0 && N == heads * BM && h.cs &&
                    (h.mode == 2 ? (h.k_cache && h.v_cache && h.tok_page && h.tok_slot && h.cu_new && h.ctx_saved &&
                                    h.ctx_out && n_groups <= MAX_GROUPS)
                                 : (h.q && h.bk && h.bv && h.S >= 1 && h.S <= 16 && n_groups == 1)) &&
                    (!h.norm || (h.mode == 2 || h.gq) && h.gk[0]);
    if (!ok) return set_error(DFLASH_ERR_ARG, "gemm %s: head epilogue operands", name);
  }
  const GemmPlan pl = gemm_plan(M, N, K, n_groups, f8, split, epi == EPI_SWIGLU || conv, per_sm, lc.num_sms,
                                lc.gemm_ctas);
  const long long tiles = pl.tiles;
  Params p = {};
  p.M = M;
  p.N = N;
  p.K = K;
  p.n_groups = n_groups;
  p.rtpg = pl.rtpg;
  p.out_gstride = op.out_gstride;
  p.tok_tiles = pl.tok_tiles;
  p.rt_total = pl.rtpg * n_groups;
  p.kbpt = pl.kbpt;
  p.total = pl.total;
  p.G = pl.G;
  p.csk = pl.csk;
  p.epi = epi;
  p.out = op.out;
  p.ldo = op.ldo;
  p.out_lo = op.out_lo;
  p.out2 = op.out2;
  p.out2_lo = op.out2_lo;
  p.ldo2 = op.ldo2;
  p.bias = op.bias;
  p.cy = op.conv_y;
  p.cy_lo = op.conv_y_lo;
  p.cy32 = op.conv_y32;
  p.ldy = op.ldy;
  p.cS = op.conv_S;
  p.head = op.head;
  if (f8) {
    for (int g = 0; g < p.n_groups; ++g) {
      p.wscale[g] = p.n_groups > 1 ? op.wscale_g[g] : op.wscale;
      if (!p.wscale[g]) return set_error(DFLASH_ERR_ARG, "gemm %s: FP8 weights without row scales", name);
    }
  }
  p.partials = sc.partials;
  p.counters = sc.counters;
  p.status = lc.status;
  p.timeout_ns = lc.timeout_ns;
  if (tiles > sc.n_counters || static_cast<size_t>(p.G) * 2 * BM * BN > sc.partial_floats)
    return set_error(DFLASH_ERR_SHAPE, "gemm %s: workspace too small for %lld tiles", name, tiles);
  WMaps tW;
  CUtensorMap tX, tXl;
  for (int g = 0; g < p.n_groups; ++g) {
    const void *Wg = p.n_groups > 1 ? op.Wg[g] : op.W;
    if (!Wg) return set_error(DFLASH_ERR_ARG, "gemm %s: null weight group %d", name, g);
    // FP8 codes: [128 rows][128 codes] tiles, 128-byte swizzle
    if (int e = f8 ? make_tmap_2d(&tW.m[g], Wg, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, N, static_cast<uint64_t>(op.ldw),
                                  2 * BK, BM)
                   : make_tmap_2d(&tW.m[g], Wg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N,
                                  static_cast<uint64_t>(op.ldw) * 2, BK, BM))
      return e;
  }
  if (int e = make_tmap_2d(&tX, op.X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, M, static_cast<uint64_t>(op.ldx) * 2,
                           BK, BN))
    return e;
  if (split) {
    if (int e = make_tmap_2d(&tXl, op.X_lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, M,
                             static_cast<uint64_t>(op.ldx) * 2, BK, BN))
      return e;
  } else {
    tXl = tX;
  }
  const double xb = (split ? 4.0 : 2.0) * M * K;
  // short conv: y read and the result written for 8N channels (pre: bf16 y
  // hi / lo in, hi / lo out; post: fp32 y in, fp32 residual read and written)
  const double out_bytes = epi == EPI_HEADS       ? 2.0 * M * N
                           : epi == EPI_CONV_PRE  ? (split ? 64.0 : 32.0) * M * N
                           : epi == EPI_CONV_POST ? 96.0 * M * N
                           : (epi == EPI_F32 || epi == EPI_TANH_BIAS) ? 4.0 * M * N
                           : epi == EPI_ADD_F32                      ? 8.0 * M * N
                           : epi == EPI_F32_SPLIT                    ? 8.0 * M * N
                           : epi == EPI_SWIGLU                       ? (op.out_lo ? 2.0 : 1.0) * M * N
                                                                     : (op.out_lo ? 4.0 : 2.0) * M * N;
  const double ng = p.n_groups;
  ProfScope ps(lc, name, ng * (wbytes * static_cast<double>(N) * K + (f8 ? 4.0 * N : 0.0) + out_bytes) + xb,
               ng * (split ? 4.0 : 2.0) * M * N * K);
  if (f8) return split ? launch_bn<true, true>(BN, lc, tW, tX, tXl, p) : launch_bn<false, true>(BN, lc, tW, tX, tXl, p);
  return split ? launch_bn<true, false>(BN, lc, tW, tX, tXl, p) : launch_bn<false, false>(BN, lc, tW, tX, tXl, p);
}

}  // namespace dflash

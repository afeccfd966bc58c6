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
//     deterministic, no spin-waits.  Its own share it takes from TMEM, the
//     others (on its last segment, when the ring is idle) by bulk copy into
//     the ring; shares are stored transposed (tile_f4) so that every warp
//     access is 512 contiguous bytes;
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
#include <cstring>

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
// Output tensors for the bulk-store epilogue (Params::tma_out): the output
// and, for bf16 outputs split into high and low halves, the low halves.
struct OMaps {
  CUtensorMap o, olo;
};

constexpr int pow2_at_least(int x) { return x <= 32 ? 32 : 2 * pow2_at_least((x + 1) / 2); }

// The most fp32 share rows one CTA of a push-mode split-K cluster receives:
// max over widths s = 2..16 of (s - 1) * ceil(128 / s).
constexpr int max_push_rows(int s = 2) {
  return s > 16 ? 0
                : ((s - 1) * ((128 + s - 1) / s) > max_push_rows(s + 1) ? (s - 1) * ((128 + s - 1) / s)
                                                                        : max_push_rows(s + 1));
}
static_assert(max_push_rows() == 130, "push-mode share rows");

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
  // the owning CTA: at most (csk - 1) * ceil(128 / csk) rows arrive, 130 for
  // some cluster width up to 16 (14 CTAs)
  static constexpr bool PUSH = BN <= 32;
  static constexpr int PUSH_BYTES = PUSH ? max_push_rows() * BN * 4 : 0;
  // the top-16 epilogue's exchange (4 warps x 16 tokens x 16 keys); it never
  // runs with the push path, so the two share one region
  static constexpr int XCH_BYTES = 4 * 16 * 16 * 8;
  // the bulk-store epilogue (token tiles of 64+): per epilogue warp two 2 KB
  // buffers of 16 tokens x 32 rows (fp32, or bf16 high + low halves)
  static constexpr int OSTG_WARP = 4096;
  static constexpr int OSTG_BYTES = BN >= 64 ? 4 * OSTG_WARP : 0;
  static constexpr int XREG0 = PUSH_BYTES > XCH_BYTES ? PUSH_BYTES : XCH_BYTES;
  static constexpr int XREG = XREG0 > OSTG_BYTES ? XREG0 : OSTG_BYTES;
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
  static_assert((2 * STAGES + 2 * CSTAGES + 8) * 8 + 12 <= CTRL, "GEMM control block overflows");
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
  // 1: outputs leave through bulk tensor stores (reduce-add for EPI_ADD_F32)
  // staged per epilogue warp; token tiles of 64+, one group, the plain
  // epilogues (F32, ADD_F32, TANH_BIAS, BF16, SWIGLU)
  int tma_out;
  void *out;
  int ldo;
  void *out_lo;        // low bf16 halves of a bf16 output, or null
  void *out2, *out2_lo;
  int ldo2;
  const float *bias;
  uint64_t *cand;           // EPI_TOPK: [M][cand_ld][16]
  int cand_ld;
  const float *wscale[MAX_GROUPS];   // F8: per-row weight scales of each group
  // [G][2] fp32 shares of BM x BN tiles, each in the transposed layout of
  // tile_f4() (16-byte aligned: the fixup bulk-copies whole shares)
  float *partials;
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

// One fp32 share of `rows` rows x BN columns (the rows a CTA of a cluster
// split-K pushes to another) as float4 units [c][i][r]: row r's columns
// 16c + 4i .. 16c + 4i + 3 sit at float4 index (4c + i) * rows + r.  Lanes
// hold consecutive rows, so every warp access moves 512 contiguous bytes:
// coalesced in global memory, free of bank conflicts in shared memory
// (row-major rows of 1 KB put all 32 lanes of an access on the same banks).
__device__ __forceinline__ int share_f4(int c, int i, int r, int rows) { return (4 * c + i) * rows + r; }
// A whole BM-row share (stream-K partial, cluster split-K stage) orders the
// same units [c][warp][i][lane]: each epilogue warp's part of a 16-column
// group (rows 32w .. 32w + 31) is one contiguous 2 KB run, which the
// bulk-store epilogue reuses as that warp's staging buffer once read.
__device__ __forceinline__ int tile_f4(int c, int i, int r) { return ((c * 4 + (r >> 5)) * 4 + i) * 32 + (r & 31); }

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// silu with the fast exponential and division (relative error ~1e-7,
// far below the bf16 rounding of the output)
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// SwiGLU of one lane pair's 16 token columns (rows 2j = gate and 2j + 1 = up
// sit in neighbouring lanes): one shuffle per output, the transcendental
// work split evenly - the even lane returns tokens 0..7, the odd lane tokens
// 8..15 (o[j] is token j + 8 * odd).  Every lane of the warp calls it.
__device__ __forceinline__ void swiglu_pair(const float (&v)[16], bool odd, float (&o)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float p = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[8 + j], 1);
    const float g = odd ? p : v[j], u = odd ? v[8 + j] : p;
    o[j] = silu(g) * u;
  }
}

__device__ __forceinline__ void store_hl(__nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t i, float v) {
  const __nv_bfloat16 h = f2bf(v);
  hi[i] = h;
  if (lo) lo[i] = f2bf(v - bf2f(h));
}

// Lanes 0..15 sorted descending, lanes 16..31 ascending (a bitonic
// sequence) -> all 32 sorted descending.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t key, int lane) {
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, key, j);
    key = (lane & j) == 0 ? (key > o ? key : o) : (key < o ? key : o);
  }
  return key;
}

// EPI_TOPK ("DFlash 2", Arquitectura del Sistema item 1: 16 candidates per
// position from the shared LM head): the 16 largest (logit, vocabulary id)
// keys of each of the 16 token columns over this 128-row vocabulary tile,
// without the logits leaving the chip.  Row n = vocabulary id (the LM head
// is one group; n / 128 is the tile).  All 128 epilogue threads call it
// together: every warp sorts its 32 rows per token (bitonic; the keys of the
// 32 lanes end descending, lane 0 largest; four tokens at a time), the four warp
// lists of each token meet in shared memory, and one warp per four tokens
// merges them (two bitonic merges of 16 + 16, then one more).
__device__ __noinline__ void topk_tile(const Params &p, const float (&v)[16], int n, int tok0, uint64_t *xch) {
  const int r = n & 127, lane = r & 31, q4 = r >> 5, rt = n >> 7;
  const bool nok = n < p.N;
  for (int t0 = 0; t0 < 16; t0 += 4) {   // four independent sorting networks in flight
    uint64_t key[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) key[u] = nok ? make_key(v[t0 + u], n) : 0ull;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const bool keep_max = ((lane & k) == 0) == ((lane & j) == 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, key[u], j);
          key[u] = keep_max ? (key[u] > o ? key[u] : o) : (key[u] < o ? key[u] : o);
        }
      }
    if (lane < 16) {
#pragma unroll
      for (int u = 0; u < 4; ++u) xch[(q4 * 16 + t0 + u) * 16 + lane] = key[u];
    }
  }
  epi_bar();
  for (int tt = 0; tt < 4; ++tt) {
    const int t = q4 * 4 + tt;
    const uint64_t *l0 = xch + (0 * 16 + t) * 16, *l1 = xch + (1 * 16 + t) * 16;
    const uint64_t *l2 = xch + (2 * 16 + t) * 16, *l3 = xch + (3 * 16 + t) * 16;
    uint64_t a = warp_merge_desc(lane < 16 ? l0[lane] : l1[31 - lane], lane);
    uint64_t b = warp_merge_desc(lane < 16 ? l2[lane] : l3[31 - lane], lane);
    const uint64_t b_rev = __shfl_sync(0xffffffffu, b, 31 - lane);
    const uint64_t c = warp_merge_desc(lane < 16 ? a : b_rev, lane);
    const int row = tok0 + t;
    if (row < p.M && lane < 16) p.cand[(static_cast<size_t>(row) * p.cand_ld + rt) * 16 + lane] = c;
  }
  epi_bar();   // the exchange is free again
}

// Apply the epilogue to 16 consecutive token columns of weight row n (ws:
// the group's FP8 row scales, or null).
// The row scale of weight row n (FP8 codes or their bf16 copies): 1 without
// scales, 0 past the rows.  Read once per tile by the callers, not per
// 16-column group (its load latency would sit on every group's path).
__device__ __forceinline__ float row_scale(const Params &p, const float *ws, int n) {
  return ws ? (n < p.N ? ws[n] : 0.f) : 1.f;
}

__device__ __forceinline__ void finalize(const Params &p, float (&v)[16], int n, int tok0, size_t goff, float sc,
                                         uint64_t *xch) {
  const bool nok = n < p.N;
  if (sc != 1.f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] *= sc;
  }
  switch (p.epi) {
    case EPI_TOPK: {
      if (p.out) {   // the logits too, when asked for
        float *o = static_cast<float *>(p.out);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (nok && tok0 + i < p.M) o[goff + static_cast<size_t>(tok0 + i) * p.ldo + n] = v[i];
      }
      topk_tile(p, v, n, tok0, xch);
    } break;
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
      // lane parity = row parity in every caller (pairs share an owner)
      __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out), *ol = static_cast<__nv_bfloat16 *>(p.out_lo);
      const bool odd = threadIdx.x & 1;
      float sw[8];
      swiglu_pair(v, odd, sw);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = j + (odd ? 8 : 0);
        if (nok && tok0 + i < p.M) store_hl(o, ol, goff + static_cast<size_t>(tok0 + i) * p.ldo + (n >> 1), sw[j]);
      }
    } break;
    case EPI_TANH_BIAS: {
      float *o = static_cast<float *>(p.out);
      const float b = nok ? p.bias[n] : 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (nok && tok0 + i < p.M) o[goff + static_cast<size_t>(tok0 + i) * p.ldo + n] = tanhf(v[i] + b);
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

// finalize() through the bulk-store epilogue: the 16 token columns of this
// warp's 32 weight rows (row n = first row + lane) go to the warp's staging
// slice as [token][row] (conflict-free: lanes write consecutive words), and
// lane 0 writes them with one tiled bulk store, or reduce-add for the
// residual epilogue (out += v, rounded as the plain path's r + v; every
// output element has one finishing CTA).  b: the warp's 2 KB staging buffer
// for this chunk, free to overwrite (the caller has waited for any earlier
// store from it and for the warp's reads of it); lane 0 commits one bulk
// group per chunk.  The same arithmetic as finalize(): identical results.
__device__ __forceinline__ void finalize_tma(const Params &p, const OMaps &om, float (&v)[16], int n, int tok0,
                                             float sc, uint8_t *b, int lane) {
  const bool nok = n < p.N;
  if (sc != 1.f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] *= sc;
  }
  const int row0 = n - lane;                      // the warp's first weight row
  const bool live = row0 < p.N && tok0 < p.M;     // anything of the box inside the output
  switch (p.epi) {
    case EPI_BF16: {
      __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(b), *l = h + 16 * 32;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const __nv_bfloat16 hv = f2bf(v[i]);
        h[i * 32 + lane] = hv;
        l[i * 32 + lane] = f2bf(v[i] - bf2f(hv));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && live) {
        tma_store_2d(&om.o, h, row0, tok0);
        if (p.out_lo) tma_store_2d(&om.olo, l, row0, tok0);
      }
    } break;
    case EPI_SWIGLU: {
      // rows 2j / 2j + 1 (neighbouring lanes) give output column j
      __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(b), *l = h + 16 * 16;
      const bool odd = lane & 1;
      float sw[8];
      swiglu_pair(v, odd, sw);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = j + (odd ? 8 : 0);
        const __nv_bfloat16 hv = f2bf(sw[j]);
        h[i * 16 + (lane >> 1)] = hv;
        l[i * 16 + (lane >> 1)] = f2bf(sw[j] - bf2f(hv));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && live) {
        tma_store_2d(&om.o, h, row0 >> 1, tok0);
        if (p.out_lo) tma_store_2d(&om.olo, l, row0 >> 1, tok0);
      }
    } break;
    default: {   // EPI_F32, EPI_ADD_F32, EPI_TANH_BIAS
      float *f = reinterpret_cast<float *>(b);
      if (p.epi == EPI_TANH_BIAS) {
        const float bb = nok ? p.bias[n] : 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i * 32 + lane] = tanhf(v[i] + bb);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i * 32 + lane] = v[i];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && live) {
        if (p.epi == EPI_ADD_F32)
          tma_reduce_add_2d(&om.o, f, row0, tok0);
        else
          tma_store_2d(&om.o, f, row0, tok0);
      }
    } break;
  }
  if (lane == 0) bulk_commit();
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
                                                 int tok0, size_t goff, float sc) {
  const bool nok = n < p.N;
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
__global__ void __launch_bounds__(Cfg<BN, SPLIT, F8>::NT, (F8 && BN <= 32) ? 2 : 1)
    gemm_tc_kernel(const __grid_constant__ WMaps wm, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmXlo, const __grid_constant__ OMaps om, const Params p) {
  using C = Cfg<BN, SPLIT, F8>;
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
  uint64_t *fbar = cempty + C::CSTAGES;   // stream-K fixup: other CTAs' shares staged in the ring
  uint64_t *xbar = fbar + 1;              // cluster split-K exchange: the other ranks' rows have arrived
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xbar + 1);
  float *spush = reinterpret_cast<float *>(base + C::RING + C::CTRL);   // push shares, or ...
  uint64_t *xch = reinterpret_cast<uint64_t *>(spush);                     // ... the top-16 exchange
  // the top-16 epilogue needs a whole tile in one CTA: no pushing of rows to
  // the other CTAs of a cluster (rank 0 pulls every share instead)
  const bool push = C::PUSH && p.epi != EPI_TOPK;
  // Cluster split-K with 64+-token tiles: exchange by bulk copies.  Each CTA
  // stages its whole share grouped by owner (share_f4 layout per owner
  // block) and one thread sends every other owner its block with one
  // cp.async.bulk; each owner's four epilogue warps sum its rows in rank
  // order from local shared memory and finalise them.  The staging plus the
  // csk - 1 receive slots must fit the idle ring (else, and for the top-16
  // epilogue, whose rank 0 takes the whole tile, the owners pull every
  // share through distributed shared memory).
  const int x_rows = (BM + p.csk - 1) / p.csk;   // most rows any rank owns
  const bool xchg = !C::PUSH && p.csk > 1 && p.epi != EPI_TOPK &&
                    static_cast<long long>(BM + (p.csk - 1) * x_rows) * BN * 4 <= C::RING;
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
    mbar_init(fbar, 1);
    mbar_init(xbar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.n_groups; ++g) tma_prefetch_desc(&wm.m[g]);
    tma_prefetch_desc(&tmX);
    if (SPLIT) tma_prefetch_desc(&tmXlo);
    if (BN >= 64 && p.tma_out) {
      tma_prefetch_desc(&om.o);
      tma_prefetch_desc(&om.olo);
    }
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
    // bulk-store epilogue: this warp's staging slice and chunk count
    uint8_t *ostg = base + C::RING + C::CTRL + (BN >= 64 ? q * C::OSTG_WARP : 0);
    uint32_t ocnt = 0;
    // a chunk's staging buffer from the warp's two alternating ones (after
    // the store issued from it two chunks earlier has read it); on the CTA's
    // last segment the idle ring serves instead, one 2 KB run per warp and
    // chunk, with no waits
    auto xbuf = [&]() -> uint8_t * {
      uint8_t *b = ostg + (ocnt & 1u) * 2048;
      if (ocnt >= 2) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
      }
      ++ocnt;
      return b;
    };
    grid_dep_wait();                     // outputs / scratch are shared with the previous kernel
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
      const float *wsg = p.wscale[rt / p.rtpg];   // FP8 codes, or bf16 copies of them
      const int tok0 = (tile / p.rt_total) * BN;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      float v[16];
      if (kb0 == 0 && kb1 == p.kbpt) {
        const bool ring_out = it + (kb1 - kb0) == end;   // last segment: the ring is idle
        const float wsc = row_scale(p, wsg, n);
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
          if (have_pre)
            finalize_add_pre(p, v, rpre, n, tok0 + c * 16, goff, wsc);
          else if (BN >= 64 && p.tma_out)
            finalize_tma(p, om, v, n, tok0 + c * 16, wsc, ring_out ? base + (c * 4 + q) * 2048 : xbuf(), lane);
          else
            finalize(p, v, n, tok0 + c * 16, goff, wsc, xch);
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
          // slot of this CTA in the owner's push area: one share of o_rows
          // rows in the share_f4 layout (lanes on consecutive rows)
          const int slot = rank < o ? rank : rank - 1;
          const uint32_t a = dsmem_addr(reinterpret_cast<float4 *>(spush) + static_cast<size_t>(slot) * (BN / 4) * o_rows +
                                            (r - o_r0),
                                        static_cast<uint32_t>(o));
#pragma unroll
          for (int j = 0; j < BN / 4; ++j)
            st_dsmem_f4(a + 16u * static_cast<uint32_t>(j * o_rows),
                        make_float4(own[4 * j], own[4 * j + 1], own[4 * j + 2], own[4 * j + 3]));
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
        const float wsc = row_scale(p, wsg, n);
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
              const float4 *src = reinterpret_cast<const float4 *>(spush) + static_cast<size_t>(slot) * (BN / 4) * my_rows;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 x = src[share_f4(c, i, r - my_r0, my_rows)];
                v[4 * i] += x.x;
                v[4 * i + 1] += x.y;
                v[4 * i + 2] += x.z;
                v[4 * i + 3] += x.w;
              }
            }
          }
          if (have_pre && mine)
            finalize_add_pre(p, v, rpre, n, tok0 + c * 16, goff, wsc);
          else
            finalize(p, v, mine ? n : p.N, tok0 + c * 16, goff, wsc, xch);   // n >= N: not this CTA's row
        }
      } else if (xchg) {
        // cluster split-K, exchange: every row goes to its owner's staging
        // block in the idle ring (owner o's block at row o_r0, its rows in
        // the share_f4 layout); the other owners' blocks are sent, this
        // CTA's own stays for its sums
        const int S = p.csk;
        const int o = ((r + 1) * S - 1) / BM;   // the rank that owns row r
        const int o_r0 = o * BM / S, o_rows = (o + 1) * BM / S - o_r0;
        float4 *blk = reinterpret_cast<float4 *>(base) + static_cast<size_t>(o_r0) * (BN / 4);
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            blk[share_f4(c, i, r - o_r0, o_rows)] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        fence_proxy_async_smem();   // the bulk copies read the staging through the async proxy
        tc_fence_before();
        __syncwarp();
      } else if (p.csk > 1) {
        // cluster split-K: this CTA's fp32 share into its own smem in the
        // tile_f4 layout (the ring is idle: every stage has been consumed);
        // the cluster reduces it on chip after the main loop
        float4 *s4 = reinterpret_cast<float4 *>(base);
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            s4[tile_f4(c, i, r)] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      } else {
        // partial tile: this CTA's fp32 share goes to its slot in the
        // tile_f4 layout; the CTA that completes the tile's k-range sums all
        // shares in CTA order (deterministic), its own straight from tensor
        // memory (the accumulator is released only after the fixup)
        constexpr int SHARE = BM * BN;   // floats
        const int slot = (tile == first_tile) ? 0 : 1;
        float4 *P4 = reinterpret_cast<float4 *>(p.partials + (static_cast<size_t>(blockIdx.x) * 2 + slot) * SHARE);
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcg(P4 + tile_f4(c, i, r), make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
        }
        fence_proxy_async_global();   // the completing CTA may bulk-copy these shares
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
          auto share_of = [&](int cc) -> const float4 * {
            return reinterpret_cast<const float4 *>(p.partials +
                                                    (static_cast<size_t>(cc) * 2 + (cc == c_lo ? slot_lo : 0)) * SHARE);
          };
          // On this CTA's last segment no copy is in flight and every ring
          // stage has been consumed: the other contributors' shares (as many
          // as the ring holds, in CTA order) arrive there by bulk copy, one
          // L2 round trip for all of them; the rest are read from L2 directly.
          const int others = c_hi - c_lo;
          const int staged = (it + (kb1 - kb0) == end) ? (others < C::RING / (SHARE * 4) ? others : C::RING / (SHARE * 4))
                                                       : 0;
          if (staged > 0) {
            if (et == 0) {
              fence_proxy_async_global();   // after the acquiring atomic: the copies read the published shares
              mbar_arrive_expect_tx(fbar, static_cast<uint32_t>(staged) * SHARE * 4);
              for (int cc = c_lo, k = 0; k < staged; ++cc) {
                if (cc == static_cast<int>(blockIdx.x)) continue;
                bulk_load(base + static_cast<size_t>(k) * SHARE * 4, share_of(cc), SHARE * 4, fbar);
                ++k;
              }
            }
            const bool got_sh = mbar_wait(fbar, 0, abort_flag, p.timeout_ns);
            if (bar_or(1, 128, !got_sh || *abort_flag)) {
              if (et == 0) report(p.status, DFLASH_ERR_TIMEOUT);
              *abort_flag = 1;
              // the copies still land in the ring: wait for them (bounded) before the CTA exits
              if (et == 0) mbar_wait(fbar, 0, nullptr, p.timeout_ns);
              break;
            }
          }
          const float4 *ring4 = reinterpret_cast<const float4 *>(base);
          const float wsc = row_scale(p, wsg, n);
          for (int c = 0; c < BN / 16; ++c) {
            float4 acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            int k = 0;   // staged shares met so far
            for (int cc = c_lo; cc <= c_hi; ++cc) {   // summed in contributor order: deterministic
              float4 t[4];
              if (cc == static_cast<int>(blockIdx.x)) {
                tmem_ld16(taddr + c * 16, v);
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
              } else if (k < staged) {
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = ring4[static_cast<size_t>(k) * (SHARE / 4) + tile_f4(c, i, r)];
                ++k;
              } else {
                const float4 *Q4 = share_of(cc);
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = __ldcg(Q4 + tile_f4(c, i, r));
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                acc[i].x += t[i].x;
                acc[i].y += t[i].y;
                acc[i].z += t[i].z;
                acc[i].w += t[i].w;
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[4 * i] = acc[i].x;
              v[4 * i + 1] = acc[i].y;
              v[4 * i + 2] = acc[i].z;
              v[4 * i + 3] = acc[i].w;
            }
            if (BN >= 64 && p.tma_out) {
              // with staged shares the output of this group goes where the
              // first staged share's run for it lay (read by this warp)
              uint8_t *b;
              if (staged > 0) {
                __syncwarp();
                b = base + (c * 4 + q) * 2048;
              } else {
                b = xbuf();
              }
              finalize_tma(p, om, v, n, tok0 + c * 16, wsc, b, lane);
            } else
              finalize(p, v, n, tok0 + c * 16, goff, wsc, xch);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        epi_bar();
      }
      it += kb1 - kb0;
    }
    if (BN >= 64 && p.tma_out && lane == 0) bulk_wait_read<0>();   // staging read before the CTA may exit
  }

  if (xchg) {
    // ---- cluster split-K exchange (see xchg above): receive slots armed,
    // every CTA's staging written and its ring idle, then one thread sends
    // each owner its block; the owner's four epilogue warps share its rows'
    // sums (every share, its own staged block included, in local shared
    // memory in the same layout), rank order per element
    const int S = p.csk, rank = static_cast<int>(cluster_ctarank());
    const int my_r0 = rank * BM / S, my_rows = (rank + 1) * BM / S - my_r0;
    const uint32_t recv = static_cast<uint32_t>(BM * BN * 4);   // receive slots after the staging
    if (threadIdx.x == 64) mbar_arrive_expect_tx(xbar, static_cast<uint32_t>((S - 1) * my_rows * BN * 4));
    cluster_sync();
    if (threadIdx.x == 64) {
      for (int o = 0; o < S; ++o) {
        if (o == rank) continue;
        const int o_r0 = o * BM / S, o_rows = (o + 1) * BM / S - o_r0;
        const int slot = rank < o ? rank : rank - 1;   // this sender's slot at the owner
        const uint32_t bytes = static_cast<uint32_t>(o_rows * BN * 4);
        bulk_copy_to_peer(dsmem_addr(base + recv + static_cast<uint32_t>(slot) * bytes, static_cast<uint32_t>(o)),
                          base + static_cast<size_t>(o_r0) * BN * 4, bytes, dsmem_addr(xbar, static_cast<uint32_t>(o)));
      }
    }
    if (warp >= 2 && warp < 6) {   // the epilogue warps
      const int et = threadIdx.x - 64;
      const bool got = mbar_wait(xbar, 0, abort_flag, p.timeout_ns);
      if (bar_or(1, 128, !got)) {
        if (et == 0) report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
      } else {
        const int tile = first_tile;
        const int rt = tile % p.rt_total;
        const size_t goff = static_cast<size_t>(rt / p.rtpg) * p.out_gstride;
        const float *wsg = p.wscale[rt / p.rtpg];   // FP8 codes, or bf16 copies of them
        const int tokt = (tile / p.rt_total) * BN;
        const float4 *own = reinterpret_cast<const float4 *>(base) + static_cast<size_t>(my_r0) * (BN / 4);
        const float4 *rv = reinterpret_cast<const float4 *>(base + recv);
        const int tasks = my_rows * (BN / 16);
        // whole warps of consecutive rows: the bulk-store epilogue
        const bool tma_w = BN >= 64 && p.tma_out && my_rows % 32 == 0;
        uint8_t *ostg = base + C::RING + C::CTRL + (BN >= 64 ? (warp & 3) * C::OSTG_WARP : 0);
        uint32_t ocnt = 0;
        for (int t0 = 0; t0 < tasks; t0 += 128) {   // every thread takes each round (shuffles in SwiGLU)
          const int task = t0 + et;
          const bool valid = task < tasks;
          const int row = valid ? task % my_rows : 0, grp = valid ? task / my_rows : 0;
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
          if (valid)
            for (int k = 0; k < S; ++k) {   // rank order: deterministic
              const float4 *src =
                  k == rank ? own : rv + static_cast<size_t>(k < rank ? k : k - 1) * my_rows * (BN / 4);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 x = src[share_f4(grp, i, row, my_rows)];
                v[4 * i] += x.x;
                v[4 * i + 1] += x.y;
                v[4 * i + 2] += x.z;
                v[4 * i + 3] += x.w;
              }
            }
          const int n = valid ? (rt % p.rtpg) * BM + my_r0 + row : p.N;   // n >= N: nothing stored
          if (tma_w) {
            uint8_t *b = ostg + (ocnt & 1u) * 2048;
            if (ocnt >= 2) {
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
            ++ocnt;
            finalize_tma(p, om, v, n, tokt + grp * 16, row_scale(p, wsg, n), b, lane);
          } else {
            finalize(p, v, n, tokt + grp * 16, goff, row_scale(p, wsg, n), xch);
          }
        }
        if (tma_w && lane == 0) bulk_wait_read<0>();
      }
    }
    cluster_sync();   // every copy has landed (its owner waited) before a sender's smem goes away
  }

  if (!xchg && !push && p.csk > 1) {
    // ---- cluster split-K reduction through distributed shared memory: CTA
    // r finalises tile rows [r*BM/csk, (r+1)*BM/csk) summing the csk shares in
    // rank order (deterministic); lanes hold consecutive rows (coalesced
    // stores, SwiGLU row pairs in neighbouring lanes)
    cluster_sync();
    if (warp >= 2 && warp < 6) {   // the epilogue warps
      const int et = threadIdx.x - 64;
      const int rank = static_cast<int>(cluster_ctarank());
      // the top-16 epilogue: rank 0 finalises the whole tile
      const bool whole = p.epi == EPI_TOPK;
      const int r0 = whole ? 0 : rank * BM / p.csk;
      const int rows = whole ? (rank == 0 ? BM : 0) : (rank + 1) * BM / p.csk - r0;
      const int tasks = rows * (BN / 16);
      const int tile = first_tile;
      const int rt = tile % p.rt_total;
      const size_t goff = static_cast<size_t>(rt / p.rtpg) * p.out_gstride;
      const float *wsg = p.wscale[rt / p.rtpg];   // FP8 codes, or bf16 copies of them
      const int tokt = (tile / p.rt_total) * BN;
      const float4 *s4 = reinterpret_cast<const float4 *>(base);   // every CTA's share, tile_f4 layout
      for (int t0 = 0; t0 < tasks; t0 += 128) {   // every thread takes each round (shuffles in SwiGLU)
        const int task = t0 + et;
        const bool valid = task < tasks;
        const int row = r0 + (valid ? task % rows : 0), grp = valid ? task / rows : 0;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        if (valid) {
          // KB ranks' loads in flight at once (one where registers are
          // scarce: the small-tile variants), then summed in rank order
          constexpr int KB = C::PUSH ? 1 : 4;
          for (int k0 = 0; k0 < p.csk; k0 += KB) {
            float4 xs[KB][4];
#pragma unroll
            for (int u = 0; u < KB; ++u)
              if (k0 + u < p.csk) {
                const uint32_t a = dsmem_addr(s4 + tile_f4(grp, 0, row), static_cast<uint32_t>(k0 + u));
#pragma unroll
                for (int i = 0; i < 4; ++i) xs[u][i] = ld_dsmem_f4(a + 512u * static_cast<uint32_t>(i));
              }
#pragma unroll
            for (int u = 0; u < KB; ++u)
              if (k0 + u < p.csk)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  v[4 * i] += xs[u][i].x;
                  v[4 * i + 1] += xs[u][i].y;
                  v[4 * i + 2] += xs[u][i].z;
                  v[4 * i + 3] += xs[u][i].w;
                }
          }
        }
        const int n = valid ? (rt % p.rtpg) * BM + row : p.N;   // n >= N: nothing stored
        finalize(p, v, n, tokt + grp * 16, goff, row_scale(p, wsg, n), xch);
      }
    }
    cluster_sync();   // nobody leaves while others still read its share
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------------ CTA pairs
// The tensor-bound projections (256-token tiles, bf16 weights and
// activations) on CTA pairs with the 2-SM tcgen05.mma (cta_group::2,
// M = 256 weight rows x N = BN tokens): each CTA of a 2-CTA cluster stages
// its own 128 weight rows and its half of the token tile, so a 64-k stage is
// 32 KB per SM instead of 48 KB for the same MMA work; the same shared
// memory holds a six-deep ring instead of four, which is what the pipeline
// needs to cover the L2 / DRAM latency at this operand rate.  Work: stream-K
// over pair tiles (token tile, pair of weight row tiles), with the same
// last-arriver fixup per CTA half as the single-CTA kernel; an odd last row
// tile pairs with a phantom half whose weight rows TMA fills with zeros and
// whose output nobody stores.
//   even CTA (rank 0): warp 0 TMA, warp 1 MMA issue for the pair, warps 2-5
//   epilogue of rows 0..127;  odd CTA: warp 0 TMA, warps 2-5 epilogue of its
//   rows.  Full barriers live in the even CTA (both CTAs' TMA complete on
//   them); the MMA completion arrives on both CTAs' empty / accumulator-full
//   barriers (multicast commit); both CTAs' epilogues release an accumulator
//   on the even CTA's barrier.
template <int BN>
struct PairCfg {
  static constexpr int NT = 192;
  static constexpr int BH = BN / 2;                    // this CTA's token rows
  static constexpr int A_BYTES = BM * BK * 2;          // this CTA's 128 weight rows, one 64-k block
  static constexpr int B_BYTES = BH * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int CTRL = 512;
  static constexpr int OSTG_WARP = 4096;               // bulk-store staging per epilogue warp
  static constexpr int TMEM_COLS = 2 * BN;             // two accumulators of BN columns
  static constexpr int SMEM = 1024 + RING + CTRL + 4 * OSTG_WARP;
  static_assert((2 * STAGES + 6) * 8 + 12 <= CTRL, "pair GEMM control block overflows");
  static_assert(SMEM <= 227 * 1024 && TMEM_COLS <= 512, "pair GEMM resources");
};

template <int BN>
__global__ void __launch_bounds__(PairCfg<BN>::NT, 1)
    gemm_pair_kernel(const __grid_constant__ WMaps wm, const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ OMaps om, const Params p) {
  using C = PairCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *base = smem_raw + pad;
  uint8_t *sA = base;
  uint8_t *sB = base + C::STAGES * C::A_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + C::RING);
  uint64_t *empty = full + C::STAGES;
  uint64_t *tfull = empty + C::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint64_t *fbar = drain + 1;   // fixup: the other contributors' shares staged in the ring
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fbar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *bcast = reinterpret_cast<int *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());   // 0: the pair's MMA issuer
  const int pair = blockIdx.x >> 1, Gp = p.G >> 1;
  const int RTP = (p.rt_total + 1) >> 1;                  // row-tile pairs per token tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 8);   // four epilogue warps of each CTA
    mbar_init(&tempty[1], 8);
    mbar_init(drain, 1);
    mbar_init(fbar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.n_groups; ++g) tma_prefetch_desc(&wm.m[g]);
    tma_prefetch_desc(&tmX);
  }
  grid_dep_launch();
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // both CTAs' barriers and tensor memory exist
  const uint32_t tmem = *tmem_slot;
  const long long begin = range_begin(p.total, Gp, pair), end = range_begin(p.total, Gp, pair + 1);
  const int first_pt = static_cast<int>(begin / p.kbpt);

  // this CTA's weight rows of pair tile pt: (group, first row); phantom past the last row tile
  auto rows_of = [&](int pt, int &g, int &row0, bool &phantom) {
    const int rt = 2 * (pt % RTP) + rank;
    phantom = rt >= p.rt_total;
    const int rtc = phantom ? p.rt_total - 1 : rt;
    g = rtc / p.rtpg;
    row0 = (phantom ? p.rtpg : rtc % p.rtpg) * BM;   // phantom: past the group's rows (zero fill)
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const bool hint_w = p.tok_tiles == 1;
      const long long n_my = end - begin;
      auto full_addr = [&](int s) { return dsmem_addr(&full[s], 0u); };   // the even CTA's full barrier
      auto load_w = [&](int s, int g, int row0, int kb) {
        if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
        (void)hint_w;
        (void)pol_w;
        tma_load_2d_pair(sA + s * C::A_BYTES, &wm.m[g], full_addr(s), kb * BK, row0);
      };
      auto load_x = [&](int s, int tok, int kb) {
        tma_load_2d_pair(sB + s * C::B_BYTES, &tmX, full_addr(s), kb * BK, tok * BN + rank * C::BH);
      };
      const int n_pre = static_cast<int>(n_my < C::STAGES ? n_my : C::STAGES);
      // iteration -> (pair tile, k-block) and the tile's weight rows, advanced
      // incrementally: no 64-bit division in the issue loop (one thread
      // issues both loads of every ~650-cycle k-block)
      struct PIter {
        int pt, kb, g, row0, tok;
      };
      auto start = [&](long long it) {
        PIter q;
        q.pt = static_cast<int>(it / p.kbpt);
        q.kb = static_cast<int>(it - static_cast<long long>(q.pt) * p.kbpt);
        bool ph;
        rows_of(q.pt, q.g, q.row0, ph);
        q.tok = q.pt / RTP;
        return q;
      };
      auto advance = [&](PIter &q) {
        if (++q.kb == p.kbpt) {
          q.kb = 0;
          ++q.pt;
          bool ph;
          rows_of(q.pt, q.g, q.row0, ph);
          q.tok = q.pt / RTP;
        }
      };
      // weights of the first ring slots depend on nothing: stream them while
      // the previous kernel finishes, then wait for it before the activations
      PIter q = start(begin);
      for (int i = 0; i < n_pre; ++i, advance(q)) load_w(i, q.g, q.row0, q.kb);
      grid_dep_wait();
      q = start(begin);
      for (int i = 0; i < n_pre; ++i, advance(q)) load_x(i, q.tok, q.kb);
      uint32_t stage = n_pre % C::STAGES, phase = (n_pre == C::STAGES) ? 1u : 0u;
      long long issued = n_pre;
      bool ok = true;
      for (long long it = begin + n_pre; it < end; ++it, advance(q)) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        load_w(stage, q.g, q.row0, q.kb);
        load_x(stage, q.tok, q.kb);
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        // let the copies in flight land before shared memory goes away: the
        // even CTA waits for each issued phase of its full barriers (they
        // count both CTAs' bytes); the odd CTA's copies complete there too,
        // so it only holds on for a bounded moment
        if (rank == 0) {
          for (int s = 0; s < C::STAGES; ++s) {
            if (issued <= s) break;
            const long long last = s + C::STAGES * ((issued - 1 - s) / C::STAGES);
            mbar_wait(&full[s], static_cast<uint32_t>((last / C::STAGES) & 1), nullptr, p.timeout_ns);
          }
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 50000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
      uint32_t stage = 0, phase = 0;
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
          if (!mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k)
            umma_bf16_pair(d, sdesc_k_sw128(a0 + k * UK * 2), sdesc_k_sw128(b0 + k * UK * 2), idesc,
                           (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit_pair(&empty[stage]);   // frees this stage in both CTAs
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[buf]);       // accumulator ready in both CTAs
        it += kb1 - kb0;
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        umma_commit_pair(drain);   // all issued MMAs retire before tensor memory is freed
        mbar_wait(drain, 0, nullptr, p.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 64;
    const uint32_t tempty_leader0 = dsmem_addr(&tempty[0], 0u), tempty_leader1 = dsmem_addr(&tempty[1], 0u);
    // bulk-store epilogue staging (see the single-CTA kernel): two buffers
    // per warp, or the idle ring on the pair's last segment
    uint8_t *ostg = base + C::RING + C::CTRL + q * C::OSTG_WARP;
    uint32_t ocnt = 0;
    auto xbuf = [&]() -> uint8_t * {
      uint8_t *b = ostg + (ocnt & 1u) * 2048;
      if (ocnt >= 2) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
      }
      ++ocnt;
      return b;
    };
    grid_dep_wait();
    int seg = 0;
    for (long long it = begin; it < end; ++seg) {
      const int pt = static_cast<int>(it / p.kbpt);
      const int kb0 = static_cast<int>(it % p.kbpt);
      const int kb1 = static_cast<int>((kb0 + (end - it) < p.kbpt ? kb0 + (end - it) : p.kbpt));
      const int buf = seg & 1;
      const bool got = mbar_wait(&tfull[buf], static_cast<uint32_t>((seg >> 1) & 1), abort_flag, p.timeout_ns);
      if (bar_or(1, 128, !got || *abort_flag)) {
        if (et == 0) report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      int g, row0;
      bool phantom;
      rows_of(pt, g, row0, phantom);
      const int n = row0 + r;                                   // row within its group
      const size_t goff = static_cast<size_t>(g) * p.out_gstride;
      const int tok0 = (pt / RTP) * BN;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      float v[16];
      auto release = [&]() {   // this warp's accumulator rows are read
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&tempty[buf]);
          else
            mbar_arrive_remote(buf ? tempty_leader1 : tempty_leader0);
        }
      };
      if (phantom) {
        release();
      } else if (kb0 == 0 && kb1 == p.kbpt) {
        // the pair's last segment: every MMA of both CTAs has completed, the rings are idle
        const bool ring_out = it + (kb1 - kb0) == end;
        const float wsc = row_scale(p, p.wscale[g], n);
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
          if (p.tma_out)
            finalize_tma(p, om, v, n, tok0 + c * 16, wsc, ring_out ? base + (c * 4 + q) * 2048 : xbuf(), lane);
          else
            finalize(p, v, n, tok0 + c * 16, goff, wsc, nullptr);
        }
        release();
      } else {
        // partial tile: this CTA's fp32 share of its 128 rows to its slot
        // (tile_f4 layout); the CTA (of the same rank) completing the tile's
        // k-range sums all shares in pair order, its own straight from TMEM
        // (the accumulator is released after the fixup) and, on its last
        // segment, the others bulk-copied into its idle ring
        constexpr int SHARE = BM * BN;   // floats
        const int tile_h = pt * 2 + rank;
        const int slot = (pt == first_pt) ? 0 : 1;
        float4 *P4 = reinterpret_cast<float4 *>(p.partials + (static_cast<size_t>(blockIdx.x) * 2 + slot) * SHARE);
        for (int c = 0; c < BN / 16; ++c) {
          tmem_ld16(taddr + c * 16, v);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcg(P4 + tile_f4(c, i, r), make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
        }
        fence_proxy_async_global();   // the completing CTA may bulk-copy these shares
        epi_bar();
        if (et == 0) {
          __threadfence();
          const int nk = kb1 - kb0;
          const int old = atomicAdd(&p.counters[tile_h], nk);
          const int last = (old + nk == p.kbpt) ? 1 : 0;
          if (last) {
            p.counters[tile_h] = 0;
            __threadfence();
          }
          *bcast = last;
        }
        epi_bar();
        if (*bcast) {
          const long long t_beg = static_cast<long long>(pt) * p.kbpt;
          const int c_lo = cta_of(t_beg, p.total, Gp);
          const int c_hi = cta_of(t_beg + p.kbpt - 1, p.total, Gp);
          const int slot_lo = range_begin(p.total, Gp, c_lo) < t_beg ? 1 : 0;
          auto share_of = [&](int cc) -> const float4 * {
            return reinterpret_cast<const float4 *>(
                p.partials + (static_cast<size_t>(2 * cc + rank) * 2 + (cc == c_lo ? slot_lo : 0)) * SHARE);
          };
          const int others = c_hi - c_lo;
          const int staged = (it + (kb1 - kb0) == end) ? (others < C::RING / (SHARE * 4) ? others : C::RING / (SHARE * 4))
                                                       : 0;
          if (staged > 0) {
            if (et == 0) {
              fence_proxy_async_global();   // after the acquiring atomic: the copies read the published shares
              mbar_arrive_expect_tx(fbar, static_cast<uint32_t>(staged) * SHARE * 4);
              for (int cc = c_lo, k = 0; k < staged; ++cc) {
                if (cc == pair) continue;
                bulk_load(base + static_cast<size_t>(k) * SHARE * 4, share_of(cc), SHARE * 4, fbar);
                ++k;
              }
            }
            const bool got_sh = mbar_wait(fbar, 0, abort_flag, p.timeout_ns);
            if (bar_or(1, 128, !got_sh || *abort_flag)) {
              if (et == 0) report(p.status, DFLASH_ERR_TIMEOUT);
              *abort_flag = 1;
              if (et == 0) mbar_wait(fbar, 0, nullptr, p.timeout_ns);   // the copies land before the CTA exits
              break;
            }
          }
          const float4 *ring4 = reinterpret_cast<const float4 *>(base);
          const float wsc = row_scale(p, p.wscale[g], n);
          for (int c = 0; c < BN / 16; ++c) {
            float4 acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            int k = 0;   // staged shares met so far
            for (int cc = c_lo; cc <= c_hi; ++cc) {   // summed in pair order: deterministic
              float4 t[4];
              if (cc == pair) {
                tmem_ld16(taddr + c * 16, v);
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
              } else if (k < staged) {
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = ring4[static_cast<size_t>(k) * (SHARE / 4) + tile_f4(c, i, r)];
                ++k;
              } else {
                const float4 *Q4 = share_of(cc);
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = __ldcg(Q4 + tile_f4(c, i, r));
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                acc[i].x += t[i].x;
                acc[i].y += t[i].y;
                acc[i].z += t[i].z;
                acc[i].w += t[i].w;
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[4 * i] = acc[i].x;
              v[4 * i + 1] = acc[i].y;
              v[4 * i + 2] = acc[i].z;
              v[4 * i + 3] = acc[i].w;
            }
            if (p.tma_out) {
              uint8_t *b;
              if (staged > 0) {   // the first staged share's run for this group, read by this warp
                __syncwarp();
                b = base + (c * 4 + q) * 2048;
              } else {
                b = xbuf();
              }
              finalize_tma(p, om, v, n, tok0 + c * 16, wsc, b, lane);
            } else {
              finalize(p, v, n, tok0 + c * 16, goff, wsc, nullptr);
            }
          }
        }
        release();
        epi_bar();
      }
      it += kb1 - kb0;
    }
    if (p.tma_out && lane == 0) bulk_wait_read<0>();   // staging read before the CTA may exit
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the pair's MMAs read both CTAs' shared memory: nobody leaves early
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, C::TMEM_COLS);
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
  if (int e = cuda_check(cudaFuncSetAttribute(gemm_tc_kernel<BN, SPLIT, F8>,
                                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
                         "gemm cluster-size attribute"))   // cluster split-K up to 16 CTAs
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
int launch(const Launch &lc, const WMaps &tW, const CUtensorMap &tX, const CUtensorMap &tXl, const OMaps &tO,
           const Params &p) {
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
  return cuda_check(cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, SPLIT, F8>, tW, tX, tXl, tO, p), "gemm launch");
}

template <bool SPLIT, bool F8>
int launch_bn(int BN, const Launch &lc, const WMaps &tW, const CUtensorMap &tX, const CUtensorMap &tXl,
              const OMaps &tO, const Params &p) {
  switch (BN) {
    case 16: return launch<16, SPLIT, F8>(lc, tW, tX, tXl, tO, p);
    case 32: return launch<32, SPLIT, F8>(lc, tW, tX, tXl, tO, p);
    case 64: return launch<64, SPLIT, F8>(lc, tW, tX, tXl, tO, p);
    case 128: return launch<128, SPLIT, F8>(lc, tW, tX, tXl, tO, p);
    default: return launch<F8 ? 128 : 256, SPLIT, F8>(lc, tW, tX, tXl, tO, p);   // FP8 tiles stop at 128
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

// The pair kernel: attributes once per device; returns how many 2-CTA
// clusters can be resident at once (pairs need two SMs of one GPC), or < 0.
template <int BN>
int pair_setup() {
  using C = PairCfg<BN>;
  constexpr int MAX_DEV = 64;
  static std::atomic<int> per_dev[MAX_DEV];
  int dev = 0;
  if (int e = cuda_check(cudaGetDevice(&dev), "device")) return e;
  if (dev < 0 || dev >= MAX_DEV) return set_error(DFLASH_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, MAX_DEV);
  int v = per_dev[dev].load(std::memory_order_acquire);
  if (v == 0) {
    if (int e = cuda_check(cudaFuncSetAttribute(gemm_pair_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                C::SMEM),
                           "pair gemm smem attribute"))
      return e;
    cudaLaunchConfig_t cfg = {};
    int sms = 0;
    if (int e = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count")) return e;
    cfg.gridDim = dim3(2 * (sms / 2));
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (int e = cuda_check(cudaOccupancyMaxActiveClusters(&clusters, gemm_pair_kernel<BN>, &cfg),
                           "pair gemm cluster occupancy"))
      return e;
    v = clusters > 0 ? clusters : 1;
    per_dev[dev].store(v, std::memory_order_release);
  }
  return v;
}

template <int BN>
int launch_pair(const Launch &lc, const WMaps &tW, const CUtensorMap &tX, const OMaps &tO, const Params &p) {
  using C = PairCfg<BN>;
  if (int e = pair_setup<BN>(); e < 0) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(C::NT);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cuda_check(cudaLaunchKernelEx(&cfg, gemm_pair_kernel<BN>, tW, tX, tO, p), "pair gemm launch");
}

}  // namespace

int fp8_rows_to_bf16(const Launch &lc, const void *codes, long long n, void *out) {
  if (n <= 0 || n % 4 || !codes || !out || (reinterpret_cast<uintptr_t>(codes) & 3) ||
      (reinterpret_cast<uintptr_t>(out) & 7))
    return set_error(DFLASH_ERR_ARG, "fp8 weights to bf16: a positive multiple of 4 codes, buffers aligned");
  const long long n4 = n / 4;
  for (long long o = 0; o < n4; o += (1ll << 30)) {   // grid x stays within range
    const int cnt = static_cast<int>(n4 - o < (1ll << 30) ? n4 - o : (1ll << 30));
    e4m3_to_bf16_kernel<<<(cnt + 255) / 256, 256, 0, lc.stream>>>(static_cast<const uint32_t *>(codes) + o, cnt,
                                                                  static_cast<uint2 *>(out) + o);
  }
  return cuda_check(cudaGetLastError(), "fp8 weights to bf16 launch");
}

int gemm_pair_clusters() { return pair_setup<256>(); }

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

GemmPlan gemm_plan(int M, int N, int K, int n_groups, bool f8, bool split, bool swiglu, int per_sm, int num_sms,
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
    // all pipeline fill; at least 2-way where the k-range allows); a GEMM of
    // a handful of tiles (at most a sixteenth of the slots: the DFlash-2
    // conv coefficients, 4 tiles) takes clusters of up to 16 CTAs (the
    // non-portable size) at 4 or more k-blocks each, so that it still spreads
    // over some 64 SMs
    const bool wide = pl.tiles * 16 <= cap;
    long long s = std::min<long long>(std::min<long long>(wide ? 16 : 8, cap / pl.tiles),
                                      std::min<long long>(pl.kbpt, std::max<long long>(2, pl.kbpt / (wide ? 4 : 8))));
    // SwiGLU pairs rows 2i / 2i+1 in neighbouring lanes: row ranges must be
    // even-aligned, so a power-of-two cluster there
    if (swiglu)
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
  if ((!op.W && op.n_groups <= 1) || !op.X || (!op.out && op.epi != EPI_TOPK))
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
  const GemmPlan pl = gemm_plan(M, N, K, n_groups, f8, split, epi == EPI_SWIGLU, per_sm, lc.num_sms, lc.gemm_ctas);
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
  p.cand = op.cand;
  p.cand_ld = op.cand_ld;
  if (epi == EPI_TOPK && (!op.cand || op.cand_ld < (N + BM - 1) / BM || n_groups != 1))
    return set_error(DFLASH_ERR_ARG, "gemm %s: top-16 epilogue needs candidates for every tile", name);
  // row scales: always with FP8 codes; with bf16 weights when given (the
  // exact bf16 copies of FP8 codes keep their scales)
  for (int g = 0; g < p.n_groups; ++g) {
    p.wscale[g] = p.n_groups > 1 ? op.wscale_g[g] : op.wscale;
    if (f8 && !p.wscale[g]) return set_error(DFLASH_ERR_ARG, "gemm %s: FP8 weights without row scales", name);
  }
  p.partials = sc.partials;
  p.counters = sc.counters;
  p.status = lc.status;
  p.timeout_ns = lc.timeout_ns;
  if (tiles > sc.n_counters || static_cast<size_t>(p.G) * 2 * BM * BN > sc.partial_floats)
    return set_error(DFLASH_ERR_SHAPE, "gemm %s: workspace too small for %lld tiles", name, tiles);
  if (reinterpret_cast<uintptr_t>(sc.partials) & 15)
    return set_error(DFLASH_ERR_ALIGN, "gemm %s: partial scratch must be 16-byte aligned", name);
  // Tensor-bound 256-token tiles (bf16 weights and activations): CTA pairs
  // with the 2-SM MMA (a third less operand traffic per MMA) where that
  // pays, as measured:
  //  * at least one full 256-token tile (at 160 tokens pairs were slower:
  //    gate/up 344 -> 364 us per step);
  //  * a single-CTA cluster split-K plan only over a long k-range (128+
  //    k-blocks per tile: 512-token down 311 -> 275 us, while the O
  //    projection's 64 stay on two-CTA clusters, 190 against 202 us) and
  //    only if the pair plan keeps as many CTAs busy (its pair tiles are cut
  //    at most in two: with few of them it would leave SMs idle).
  // gemm_ctas < 0 (test hook) forces -gemm_ctas pairs.
  bool pairs = !f8 && !split && BN == 256 && epi != EPI_TOPK &&
               (lc.gemm_ctas < 0 || (lc.gemm_pairs && lc.gemm_ctas == 0 && M >= 256 &&
                                     (pl.csk == 1 || pl.kbpt >= 128))) &&
               (p.n_groups == 1 || p.rtpg % 2 == 0);
  long long ptiles = 0, gp = 0;
  if (pairs) {
    const int max_pairs = pair_setup<256>();
    if (max_pairs < 0) return max_pairs;
    const long long rtp = (pl.rtpg * static_cast<long long>(p.n_groups) + 1) / 2;
    ptiles = rtp * pl.tok_tiles;
    // as many pairs as fit at once, each at least 4 k-blocks and no pair
    // tile cut into more than 2 pieces (a fixup reads at most 256 KB)
    const long long min_kb = std::max<long long>(4, (pl.kbpt + 1) / 2);
    gp = std::min<long long>(max_pairs, (ptiles * pl.kbpt + min_kb - 1) / min_kb);
    if (lc.gemm_ctas < 0) gp = -lc.gemm_ctas;
    gp = std::max<long long>(1, std::min<long long>(gp, ptiles * pl.kbpt));
    if (lc.gemm_ctas == 0 && pl.csk > 1 && 2 * gp < pl.G) pairs = false;
  }
  if (pairs) {
    p.csk = 1;
    p.total = ptiles * pl.kbpt;
    p.G = static_cast<int>(2 * gp);
    if (2 * ptiles > sc.n_counters || static_cast<size_t>(p.G) * 2 * BM * BN > sc.partial_floats)
      return set_error(DFLASH_ERR_SHAPE, "gemm %s: workspace too small for %lld pair tiles", name, ptiles);
  }
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
                           BK, pairs ? BN / 2 : BN))   // a pair's CTA stages half of the token tile
    return e;
  if (split) {
    if (int e = make_tmap_2d(&tXl, op.X_lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, M,
                             static_cast<uint64_t>(op.ldx) * 2, BK, BN))
      return e;
  } else {
    tXl = tX;
  }
  // bulk-store epilogue: 256 / 128 / 64-token tiles of one group with a plain
  // epilogue, outputs (and low halves) 16-byte aligned with 16-byte rows;
  // box = 16 tokens x one warp's 32 rows (16 output columns for SwiGLU)
  OMaps tO;
  std::memset(&tO, 0, sizeof(tO));
  p.tma_out = 0;
  if (BN >= 64 && p.n_groups == 1 &&
      (epi == EPI_F32 || epi == EPI_ADD_F32 || epi == EPI_TANH_BIAS || epi == EPI_BF16 || epi == EPI_SWIGLU)) {
    const bool f32o = epi == EPI_F32 || epi == EPI_ADD_F32 || epi == EPI_TANH_BIAS;
    const int esz = f32o ? 4 : 2;
    const uint64_t cols = epi == EPI_SWIGLU ? static_cast<uint64_t>(N / 2) : static_cast<uint64_t>(N);
    const uintptr_t oal = reinterpret_cast<uintptr_t>(op.out) | reinterpret_cast<uintptr_t>(op.out_lo);
    if (!(oal & 15) && (static_cast<long long>(op.ldo) * esz) % 16 == 0 && (epi != EPI_SWIGLU || N % 2 == 0)) {
      const CUtensorMapDataType dt = f32o ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      const uint32_t bx = epi == EPI_SWIGLU ? 16 : 32;
      const uint64_t stride = static_cast<uint64_t>(op.ldo) * esz;
      if (int e = make_tmap_2d(&tO.o, op.out, dt, esz, cols, M, stride, bx, 16, CU_TENSOR_MAP_SWIZZLE_NONE)) return e;
      if (op.out_lo) {
        if (int e = make_tmap_2d(&tO.olo, op.out_lo, dt, esz, cols, M, stride, bx, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
          return e;
      } else {
        tO.olo = tO.o;
      }
      p.tma_out = 1;
    }
  }
  const double xb = (split ? 4.0 : 2.0) * M * K;
  // top-16 epilogue: 16 keys per token per 128-row tile (+ logits if asked)
  const double out_bytes = epi == EPI_TOPK ? 128.0 * M * ((N + BM - 1) / BM) + (op.out ? 4.0 * M * N : 0.0)
                           : (epi == EPI_F32 || epi == EPI_TANH_BIAS) ? 4.0 * M * N
                           : epi == EPI_ADD_F32                      ? 8.0 * M * N
                           : epi == EPI_F32_SPLIT                    ? 8.0 * M * N
                           : epi == EPI_SWIGLU                       ? (op.out_lo ? 2.0 : 1.0) * M * N
                                                                     : (op.out_lo ? 4.0 : 2.0) * M * N;
  const double ng = p.n_groups;
  ProfScope ps(lc, name, ng * (wbytes * static_cast<double>(N) * K + (f8 ? 4.0 * N : 0.0) + out_bytes) + xb,
               ng * (split ? 4.0 : 2.0) * M * N * K);
  if (pairs) return launch_pair<256>(lc, tW, tX, tO, p);
  if (f8)
    return split ? launch_bn<true, true>(BN, lc, tW, tX, tXl, tO, p) : launch_bn<false, true>(BN, lc, tW, tX, tXl, tO, p);
  return split ? launch_bn<true, false>(BN, lc, tW, tX, tXl, tO, p) : launch_bn<false, false>(BN, lc, tW, tX, tXl, tO, p);
}

}  // namespace dflash

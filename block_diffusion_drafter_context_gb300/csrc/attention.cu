// Block attention of the DFlash drafter: the 16 block queries of a request
// attend, without any mask inside the block, to every injected context token
// of that request's paged KV cache and to the 16 block keys themselves
// ("DFlash" §2.2 parallel block diffusion; mask semantics of "FlexDraft",
// Metodologia 1: bidirectional in the block, all of the clean prefix, no
// other block).
//
// bf16 path - split-KV, decode style, HBM-bound:
//   grid (split, kv head, request); one CTA handles the 16 queries x g query
//   heads that share one KV head, over one contiguous range of the context.
//   Warp 0 streams 64-token KV pages into a 3-deep shared-memory ring with TMA
//   (128-byte swizzle, so ldmatrix reads are conflict-free).  The consumers
//   are NG groups of g warps; group i takes chunks i, i+NG, ...; inside a
//   group each warp owns one query head (16 rows) and runs QK^T and PV on
//   mma.sync bf16 tensor cores with an online (exp2-domain) softmax, so NG
//   chunks are in flight per CTA; groups merge their softmax states in shared
//   memory at the end.  The last
//   split also covers the 16 block keys.  Splits write unnormalised partials
//   plus (max, sum); the CTA that finishes a (request, head) last merges them
//   in split order - deterministic, no spin-waits.
// fp32 path - plain CUDA-core loop for the tiny fp32 configuration.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace dflash {
namespace {

constexpr int CH = 64;            // tokens per stage (= one KV page)
constexpr int HD = 128;           // head dim of the bf16 path
constexpr int HALF = CH * 64 * 2; // one 64-dim half of a 64-token tile, bytes
constexpr int TILE = 2 * HALF;    // K or V tile of one stage
constexpr int ST = 3;             // pipeline depth (3 x 32 KB: fits beside a GEMM CTA on one SM)
constexpr int BLK = 16;           // block tokens
constexpr int SMEM = 1024 + ST * 2 * TILE + 128;

struct Params {
  int ng;                  // consumer groups
  const __nv_bfloat16 *q;
  int ldq;
  __nv_bfloat16 *out;
  __nv_bfloat16 *out_lo;   // low halves (split activations) or null
  int ldo;
  const int32_t *page_table;
  int max_pages, num_pages;
  const int32_t *ctx_len;
  float *part_o, *part_ml;
  int *counters;
  int nkv, g, split, max_splits;
  float scale_log2;
  int *status;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ uint32_t swz(uint32_t base, int tok, int dch) {
  return base + (dch >> 3) * HALF + tok * 128 + ((((dch & 7) ^ (tok & 7))) << 4);
}

// two consecutive bf16 outputs (high halves) and, if lo is given, their low halves
__device__ __forceinline__ void store2_hl(__nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t i, float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  *reinterpret_cast<__nv_bfloat162 *>(hi + i) = h;
  if (lo) *reinterpret_cast<uint32_t *>(lo + i) = pack_bf16(a - __low2float(h), b - __high2float(h));
}

__device__ __forceinline__ uint32_t mask_pair(uint32_t v, int tok, int valid) {
  return (tok < valid ? (v & 0xFFFFu) : 0u) | (tok + 1 < valid ? (v & 0xFFFF0000u) : 0u);
}

__global__ void __launch_bounds__(32 * 11, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmBK, const __grid_constant__ CUtensorMap tmBV,
                     const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *base = smem_raw + pad;
  uint8_t *sK = base;
  uint8_t *sV = base + ST * TILE;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + 2 * ST * TILE);
  uint64_t *empty = full + ST;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + ST);
  int *bcast = const_cast<int *>(abort_flag + 1);

  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.g;

  pdl_start();
  int n_ctx = p.ctx_len[b];
  const int cap = p.max_pages * CH;
  if (n_ctx < 0 || n_ctx > cap) {
    if (threadIdx.x == 0 && s == 0) report(p.status, DFLASH_ERR_DEVICE);
    n_ctx = n_ctx < 0 ? 0 : cap;
  }
  const int nsplit = n_ctx > 0 ? (n_ctx + p.split - 1) / p.split : 1;
  if (s >= nsplit) return;   // uniform for the CTA
  const int t0 = s * p.split;
  const int t1 = min(n_ctx, t0 + p.split);
  const int ctx_chunks = t1 > t0 ? (t1 - t0 + CH - 1) / CH : 0;
  const bool has_block = (s == nsplit - 1);
  const int nchunks = ctx_chunks + (has_block ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], g);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t stage = 0, phase = 0;
      int last_ci[ST];
      for (int i = 0; i < ST; ++i) last_ci[i] = -1;
      bool ok = true;
      for (int ci = 0; ci < nchunks; ++ci) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        uint8_t *dk = sK + stage * TILE, *dv = sV + stage * TILE;
        if (ci < ctx_chunks) {
          const int tok = t0 + ci * CH;
          const int page = p.page_table[static_cast<size_t>(b) * p.max_pages + tok / CH];
          if (page < 0 || page >= p.num_pages) {
            report(p.status, DFLASH_ERR_DEVICE);
            mbar_arrive(&full[stage]);   // completes the phase with no data
          } else {
            const int row = (page * p.nkv + h) * CH;
            mbar_arrive_expect_tx(&full[stage], 2 * TILE);
            tma_load_2d(dk, &tmK, &full[stage], 0, row);
            tma_load_2d(dk + HALF, &tmK, &full[stage], 64, row);
            tma_load_2d(dv, &tmV, &full[stage], 0, row);
            tma_load_2d(dv + HALF, &tmV, &full[stage], 64, row);
            last_ci[stage] = ci;
          }
        } else {
          const int row = (b * p.nkv + h) * BLK;
          mbar_arrive_expect_tx(&full[stage], 4 * BLK * 128);
          tma_load_2d(dk, &tmBK, &full[stage], 0, row);
          tma_load_2d(dk + HALF, &tmBK, &full[stage], 64, row);
          tma_load_2d(dv, &tmBV, &full[stage], 0, row);
          tma_load_2d(dv + HALF, &tmBV, &full[stage], 64, row);
          last_ci[stage] = ci;
        }
        if (++stage == ST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        // let every issued copy land before shared memory is released
        for (int i = 0; i < ST; ++i)
          if (last_ci[i] >= 0)
            mbar_wait(&full[i], static_cast<uint32_t>((last_ci[i] / ST) & 1), nullptr, p.timeout_ns);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;                // consumer warp
  const int grp = cw / g;                 // chunk group
  const int w = cw % g;                   // query head within the group
  const int hq = h * g + w;
  const int gr = lane >> 2, t2 = (lane & 3) * 2;
  const int mi = lane >> 3, rr = lane & 7;

  uint32_t qa[8][4];
  {
    const __nv_bfloat16 *q0 = p.q + static_cast<size_t>(b * BLK + gr) * p.ldq + hq * HD;
    const __nv_bfloat16 *q1 = q0 + 8 * static_cast<size_t>(p.ldq);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qa[kk][0] = *reinterpret_cast<const uint32_t *>(q0 + kk * 16 + t2);
      qa[kk][1] = *reinterpret_cast<const uint32_t *>(q1 + kk * 16 + t2);
      qa[kk][2] = *reinterpret_cast<const uint32_t *>(q0 + kk * 16 + 8 + t2);
      qa[kk][3] = *reinterpret_cast<const uint32_t *>(q1 + kk * 16 + 8 + t2);
    }
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool failed = false;

  for (int ci = grp; ci < nchunks; ci += p.ng) {
    const int stage = ci % ST;
    const uint32_t phase = static_cast<uint32_t>((ci / ST) & 1);
    if (!mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns)) {
      failed = true;
      break;
    }
    const int valid = ci < ctx_chunks ? min(CH, t1 - (t0 + ci * CH)) : BLK;
    const uint32_t kb = smem_u32(sK + stage * TILE), vb = smem_u32(sV + stage * TILE);

    float sc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(swz(kb, np * 16 + (mi >> 1) * 8 + rr, kk * 2 + (mi & 1)), b0, b1, b2, b3);
        mma_bf16_16816(sc[2 * np], qa[kk], b0, b1);
        mma_bf16_16816(sc[2 * np + 1], qa[kk], b2, b3);
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int tok = nt * 8 + t2;
      sc[nt][0] = tok < valid ? sc[nt][0] * p.scale_log2 : -INFINITY;
      sc[nt][1] = tok + 1 < valid ? sc[nt][1] * p.scale_log2 : -INFINITY;
      sc[nt][2] = tok < valid ? sc[nt][2] * p.scale_log2 : -INFINITY;
      sc[nt][3] = tok + 1 < valid ? sc[nt][3] * p.scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      sc[nt][0] = fast_exp2(sc[nt][0] - mn0);
      sc[nt][1] = fast_exp2(sc[nt][1] - mn0);
      sc[nt][2] = fast_exp2(sc[nt][2] - mn1);
      sc[nt][3] = fast_exp2(sc[nt][3] - mn1);
      rs0 += sc[nt][0] + sc[nt][1];
      rs1 += sc[nt][2] + sc[nt][3];
    }
    l0 = l0 * a0 + rs0;
    l1 = l1 * a1 + rs1;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      o[nd][0] *= a0;
      o[nd][1] *= a0;
      o[nd][2] *= a1;
      o[nd][3] *= a1;
    }
    const bool partial = valid < CH;
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
      uint32_t a[4];
      a[0] = pack_bf16(sc[2 * k2][0], sc[2 * k2][1]);
      a[1] = pack_bf16(sc[2 * k2][2], sc[2 * k2][3]);
      a[2] = pack_bf16(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1]);
      a[3] = pack_bf16(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3]);
      const int tlo = k2 * 16 + t2, thi = tlo + 8;
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(swz(vb, k2 * 16 + (mi & 1) * 8 + rr, dp * 2 + (mi >> 1)), b0, b1, b2, b3);
        if (partial) {   // rows past the valid tokens may hold stale data
          b0 = mask_pair(b0, tlo, valid);
          b1 = mask_pair(b1, thi, valid);
          b2 = mask_pair(b2, tlo, valid);
          b3 = mask_pair(b3, thi, valid);
        }
        mma_bf16_16816(o[2 * dp], a, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], a, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- merge the groups' softmax states (all chunks are consumed, so the
  // stage buffers are free for the exchange)
  if (bar_or(3, 32 * g * p.ng, failed || *abort_flag)) {
    if (threadIdx.x == 32) report(p.status, DFLASH_ERR_TIMEOUT);
    return;
  }
  if (p.ng > 1) {
    float *xs = reinterpret_cast<float *>(base);
    if (grp > 0) {
      float *dst = xs + (static_cast<size_t>((grp - 1) * g + w) * 32 + lane) * 68;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        dst[nd * 4 + 0] = o[nd][0];
        dst[nd * 4 + 1] = o[nd][1];
        dst[nd * 4 + 2] = o[nd][2];
        dst[nd * 4 + 3] = o[nd][3];
      }
      dst[64] = m0;
      dst[65] = m1;
      dst[66] = l0;
      dst[67] = l1;
    }
    asm volatile("bar.sync 3, %0;" ::"r"(32 * g * p.ng) : "memory");
    if (grp > 0) return;
    for (int og = 1; og < p.ng; ++og) {
      const float *src = xs + (static_cast<size_t>((og - 1) * g + w) * 32 + lane) * 68;
      const float mb0 = src[64], mb1 = src[65];
      const float M0 = fmaxf(m0, mb0), M1 = fmaxf(m1, mb1);
      const float a0 = fast_exp2(m0 - M0), b0 = fast_exp2(mb0 - M0);
      const float a1 = fast_exp2(m1 - M1), b1 = fast_exp2(mb1 - M1);
      l0 = l0 * a0 + src[66] * b0;
      l1 = l1 * a1 + src[67] * b1;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        o[nd][0] = o[nd][0] * a0 + src[nd * 4 + 0] * b0;
        o[nd][1] = o[nd][1] * a0 + src[nd * 4 + 1] * b0;
        o[nd][2] = o[nd][2] * a1 + src[nd * 4 + 2] * b1;
        o[nd][3] = o[nd][3] * a1 + src[nd * 4 + 3] * b1;
      }
      m0 = M0;
      m1 = M1;
    }
  }
  const int nthr = 32 * g;   // group 0 carries on

  if (nsplit == 1) {
    const size_t o0 = static_cast<size_t>(b * BLK + gr) * p.ldo + hq * HD;
    const size_t o1 = o0 + 8 * static_cast<size_t>(p.ldo);
    const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      store2_hl(p.out, p.out_lo, o0 + nd * 8 + t2, o[nd][0] * i0, o[nd][1] * i0);
      store2_hl(p.out, p.out_lo, o1 + nd * 8 + t2, o[nd][2] * i1, o[nd][3] * i1);
    }
    return;
  }

  // ---- split partials: rows of this CTA are (w*16 + j), j = block position
  const size_t rows = static_cast<size_t>(BLK) * g;
  const size_t slot0 = (static_cast<size_t>(b) * p.nkv + h) * p.max_splits;
  {
    float *po = p.part_o + ((slot0 + s) * rows + w * BLK) * HD;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      __stcg(reinterpret_cast<float2 *>(po + gr * HD + nd * 8 + t2), make_float2(o[nd][0], o[nd][1]));
      __stcg(reinterpret_cast<float2 *>(po + (gr + 8) * HD + nd * 8 + t2), make_float2(o[nd][2], o[nd][3]));
    }
    if ((lane & 3) == 0) {
      float *pm = p.part_ml + ((slot0 + s) * rows + w * BLK) * 2;
      __stcg(reinterpret_cast<float2 *>(pm + gr * 2), make_float2(m0, l0));
      __stcg(reinterpret_cast<float2 *>(pm + (gr + 8) * 2), make_float2(m1, l1));
    }
  }
  __threadfence();
  asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");
  if (threadIdx.x == 32) {
    int *ctr = &p.counters[b * p.nkv + h];
    const int old = atomicAdd(ctr, 1);
    const int last = (old == nsplit - 1) ? 1 : 0;
    if (last) *ctr = 0;
    *bcast = last;
    __threadfence();
  }
  asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");
  if (!*bcast) return;

  // ---- merge the nsplit partials of this (request, kv head); each warp
  // merges its own 16 rows.  Lanes own splits for the (max, sum) pass
  // (combined with warp shuffles), then own 4 of the 128 columns for the
  // weighted sum of the partial outputs (16 independent loads per split).
  const float *pml = p.part_ml + (slot0 * rows + w * BLK) * 2;
  const float *pot = p.part_o + (slot0 * rows + w * BLK) * HD;
  float M[BLK], L[BLK];
#pragma unroll
  for (int j = 0; j < BLK; ++j) {
    M[j] = -INFINITY;
    L[j] = 0.f;
  }
  for (int s0 = 0; s0 < nsplit; s0 += 32) {        // running max / sum over groups of 32 splits
    const int ss = s0 + lane;
    float2 ml[BLK];
#pragma unroll
    for (int j = 0; j < BLK; ++j)
      ml[j] = ss < nsplit ? __ldcg(reinterpret_cast<const float2 *>(pml + (static_cast<size_t>(ss) * rows + j) * 2))
                          : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int j = 0; j < BLK; ++j) {
      const float gm = warp_max(ml[j].x);
      const float mn = fmaxf(M[j], gm);
      const float contrib = ss < nsplit ? fast_exp2(ml[j].x - mn) * ml[j].y : 0.f;
      L[j] = L[j] * fast_exp2(M[j] - mn) + warp_sum(contrib);
      M[j] = mn;
    }
  }
  float4 acc[BLK];
#pragma unroll
  for (int j = 0; j < BLK; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int ss = 0; ss < nsplit; ++ss) {
    float4 v[BLK];
#pragma unroll
    for (int j = 0; j < BLK; ++j)
      v[j] = __ldcg(reinterpret_cast<const float4 *>(pot + (static_cast<size_t>(ss) * rows + j) * HD) + lane);
#pragma unroll
    for (int j = 0; j < BLK; ++j) {
      const float m = __ldcg(pml + (static_cast<size_t>(ss) * rows + j) * 2);   // L2 hit, uniform
      const float wgt = fast_exp2(m - M[j]);
      acc[j].x += wgt * v[j].x;
      acc[j].y += wgt * v[j].y;
      acc[j].z += wgt * v[j].z;
      acc[j].w += wgt * v[j].w;
    }
  }
#pragma unroll
  for (int j = 0; j < BLK; ++j) {
    const float inv = 1.f / L[j];
    const size_t dst = static_cast<size_t>(b * BLK + j) * p.ldo + hq * HD + lane * 4;
    store2_hl(p.out, p.out_lo, dst, acc[j].x * inv, acc[j].y * inv);
    store2_hl(p.out, p.out_lo, dst + 2, acc[j].z * inv, acc[j].w * inv);
  }
}

// ------------------------------------------------------------------ fp32
template <int DPL>
__global__ void __launch_bounds__(512) attn_f32_kernel(const float *q, int ldq, const float *kc, const float *vc,
                                                       const float *bk, const float *bv, const int32_t *pt,
                                                       int max_pages, int num_pages, int page, const int32_t *ctx_len,
                                                       float *out, int ldo, int nkv, int g, float scale, int *status) {
  pdl_start();
  constexpr int D = DPL * 32;
  const int hq = blockIdx.x, b = blockIdx.y, j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = hq / g;
  int n = ctx_len[b];
  if (n < 0 || n > max_pages * page) {
    if (threadIdx.x == 0 && hq == 0) report(status, DFLASH_ERR_DEVICE);
    n = n < 0 ? 0 : max_pages * page;
  }
  float qv[DPL], acc[DPL];
  const float *qr = q + static_cast<size_t>(b * BLK + j) * ldq + hq * D;
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    qv[i] = qr[lane + 32 * i];
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int t = 0; t < n + BLK; ++t) {
    const float *kp, *vp;
    if (t < n) {
      const int pg = pt[static_cast<size_t>(b) * max_pages + t / page];
      if (pg < 0 || pg >= num_pages) {
        if (lane == 0) report(status, DFLASH_ERR_DEVICE);
        continue;
      }
      const size_t off = ((static_cast<size_t>(pg) * nkv + h) * page + t % page) * D;
      kp = kc + off;
      vp = vc + off;
    } else {
      const size_t off = ((static_cast<size_t>(b) * nkv + h) * BLK + (t - n)) * D;
      kp = bk + off;
      vp = bv + off;
    }
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) d = fmaf(qv[i], kp[lane + 32 * i], d);
    const float sc = warp_sum(d) * scale;
    const float mn = fmaxf(m, sc);
    const float a = expf(m - mn), pw = expf(sc - mn);
    l = l * a + pw;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = acc[i] * a + pw * vp[lane + 32 * i];
    m = mn;
  }
  float *orow = out + static_cast<size_t>(b * BLK + j) * ldo + hq * D;
#pragma unroll
  for (int i = 0; i < DPL; ++i) orow[lane + 32 * i] = acc[i] / l;
}

}  // namespace

int attention_bf16(const Launch &lc, const AttnArgs &a) {
  if (a.B <= 0) return DFLASH_OK;
  if (a.d != HD || a.page_size != CH)
    return set_error(DFLASH_ERR_UNSUPPORTED, "bf16 attention needs head_dim 128 and 64-token pages");
  const int g = a.nq / a.nkv;
  if (g < 1 || g > 8) return set_error(DFLASH_ERR_UNSUPPORTED, "bf16 attention: q heads per kv head must be 1..8");
  static bool attr_done = false;
  if (!attr_done) {
    if (int e = cuda_check(cudaFuncSetAttribute(attn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM),
                           "attention smem attribute"))
      return e;
    attr_done = true;
  }
  CUtensorMap tK, tV, tBK, tBV;
  const uint64_t kv_rows = static_cast<uint64_t>(a.num_pages) * a.nkv * CH;
  const uint64_t blk_rows = static_cast<uint64_t>(a.B) * a.nkv * BLK;
  if (int e = make_tmap_2d(&tK, a.k_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, kv_rows, HD * 2, 64, CH)) return e;
  if (int e = make_tmap_2d(&tV, a.v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, kv_rows, HD * 2, 64, CH)) return e;
  if (int e = make_tmap_2d(&tBK, a.bk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, blk_rows, HD * 2, 64, BLK)) return e;
  if (int e = make_tmap_2d(&tBV, a.bv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, blk_rows, HD * 2, 64, BLK)) return e;
  Params p = {};
  p.ng = (1 + 2 * g) * 32 <= 352 ? 2 : 1;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.ldq = a.nq * HD;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.out_lo = static_cast<__nv_bfloat16 *>(a.out_lo);
  p.ldo = a.nq * HD;
  p.page_table = a.page_table;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.ctx_len = a.ctx_len;
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.counters = a.counters;
  p.nkv = a.nkv;
  p.g = g;
  p.split = a.split_tokens;
  p.max_splits = a.max_splits;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(HD)));
  p.status = lc.status;
  p.timeout_ns = lc.timeout_ns;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.max_splits, a.nkv, a.B);
  cfg.blockDim = dim3(32 * (1 + p.ng * g));
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope ps(lc, "attention", -1.0, -1.0);
  return cuda_check(cudaLaunchKernelEx(&cfg, attn_bf16_kernel, tK, tV, tBK, tBV, p), "attention launch");
}

int attention_f32(const Launch &lc, const AttnArgs &a) {
  if (a.B <= 0) return DFLASH_OK;
  const int g = a.nq / a.nkv;
  dim3 grid(a.nq, a.B), block(512);
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(a.d)));
  ProfScope ps(lc, "attention", -1.0, -1.0);
  const float *q = static_cast<const float *>(a.q);
  float *o = static_cast<float *>(a.out);
#define ARGS q, a.nq * a.d, static_cast<const float *>(a.k_cache), static_cast<const float *>(a.v_cache), \
             static_cast<const float *>(a.bk), static_cast<const float *>(a.bv), a.page_table, a.max_pages, \
             a.num_pages, a.page_size, a.ctx_len, o, a.nq * a.d, a.nkv, g, scale, lc.status
  if (a.d == 64)
    launch_pdl(attn_f32_kernel<2>, grid, block, 0, lc.stream, ARGS);
  else if (a.d == 128)
    launch_pdl(attn_f32_kernel<4>, grid, block, 0, lc.stream, ARGS);
  else
    return set_error(DFLASH_ERR_UNSUPPORTED, "fp32 attention: head_dim must be 64 or 128");
#undef ARGS
  return cuda_check(cudaGetLastError(), "attention_f32 launch");
}

}  // namespace dflash

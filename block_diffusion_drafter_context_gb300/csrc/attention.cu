// Block attention of the DFlash drafter: the 16 block queries of a request
// attend, without any mask inside the block, to every injected context token
// of that request's paged KV cache and to the 16 block keys themselves
// ("DFlash" §2.2 parallel block diffusion; mask semantics of "FlexDraft",
// Metodologia 1: bidirectional in the block, all of the clean prefix, no
// other block).
//
// bf16 path - split-KV, decode style, HBM-bound, on the 5th-generation tensor
// cores:
//   grid (split, kv head, request); the S splits of one (request, kv head)
//   form one thread-block cluster.  A CTA takes the 16 queries x g query
//   heads sharing one KV head (16g rows, padded to the UMMA M of 128) over
//   one contiguous range of the context, in 64-token chunks (one KV page):
//     warp 0     TMA: Q once, then K and V^T pages into a 3-deep smem ring
//                (128-byte swizzle; V pages are stored transposed so both
//                products take K-major operands);
//     warp 1     tcgen05.mma: S = Q K^T (M=128, N=64, K=128) into one of two
//                TMEM buffers, then PV = P V (M=128, N=128, K=64) into TMEM;
//     warps 2-5  one TMEM lane (= query row) per thread: online softmax in
//                the exp2 domain on its 64 scores (no shuffles), P written
//                back to smem in bf16 as the A operand of PV, O accumulated
//                in registers.
//   QK of chunk i+1 overlaps the softmax of chunk i.  The last split also
//   covers the 16 block keys.  At the end the cluster's CTAs exchange
//   (max, sum, O) through distributed shared memory and each finalises 16g/S
//   rows: the split partials never leave the chip.
// fp32 path - plain CUDA-core loop for the tiny fp32 configuration.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace dflash {
namespace {

constexpr int CH = 64;                       // tokens per chunk (= one KV page)
constexpr int HD = 128;                      // head dim of the bf16 path
constexpr int ST = 3;                        // KV ring depth
constexpr int BLK = 16;                      // block tokens
constexpr int MROWS = 128;                   // UMMA M (query rows, padded)
constexpr int Q_BYTES = MROWS * HD * 2;      // 32 KB: two 64-dim halves of [128][64]
constexpr int K_BYTES = CH * HD * 2;         // 16 KB: two halves of [64 tok][64]
constexpr int V_BYTES = HD * CH * 2;         // 16 KB: [128 d][64 tok]
constexpr int P_BYTES = MROWS * CH * 2;      // 16 KB: [128 rows][64 tok]
constexpr int SMEM = 1024 + Q_BYTES + ST * (K_BYTES + V_BYTES) + 2 * P_BYTES + 256;
constexpr int NTHR = 192;
constexpr int TMEM_COLS = 256;               // S x 2 (64 columns each) + PV (128 columns)

struct Params {
  __nv_bfloat16 *out;
  __nv_bfloat16 *out_lo;   // low halves (split activations) or null
  int ldo;
  const int32_t *page_table;
  int max_pages, num_pages;
  const int32_t *ctx_len;
  int nkv, g, split, S;
  float scale_log2;
  int *status;
  unsigned long long timeout_ns;
};

// two consecutive bf16 outputs (high halves) and, if lo is given, their low halves
__device__ __forceinline__ void store2_hl(__nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t i, float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  *reinterpret_cast<__nv_bfloat162 *>(hi + i) = h;
  if (lo) *reinterpret_cast<uint32_t *>(lo + i) = pack_bf16(a - __low2float(h), b - __high2float(h));
}

__global__ void __launch_bounds__(NTHR, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmBK,
                   const __grid_constant__ CUtensorMap tmBV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *base = smem_raw + pad;
  uint8_t *sQ = base;
  uint8_t *sK = sQ + Q_BYTES;
  uint8_t *sV = sK + ST * K_BYTES;
  uint8_t *sP = sV + ST * V_BYTES;
  uint64_t *bar = reinterpret_cast<uint64_t *>(sP + 2 * P_BYTES);
  uint64_t *qfull = bar, *full = bar + 1, *empty = full + ST, *sfull = empty + ST, *sempty = sfull + 2,
           *pfull = sempty + 2, *ofull = pfull + 2, *oempty = ofull + 1, *drain = oempty + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.g, R = BLK * g;

  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 4);
      mbar_init(&pfull[i], 4);
    }
    mbar_init(ofull, 1);
    mbar_init(oempty, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // query rows past 16g are padding: keep them zero so their scores stay finite
  {
    const int per_half = (MROWS - R) * 128 / 16;   // 16-byte chunks
    for (int i = threadIdx.x; i < 2 * per_half; i += NTHR) {
      const int half = i / per_half, k = i % per_half;
      *reinterpret_cast<uint4 *>(sQ + half * (MROWS * 128) + R * 128 + k * 16) = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_start();
  int n_ctx = p.ctx_len[b];
  const int cap = p.max_pages * CH;
  if (n_ctx < 0 || n_ctx > cap) {
    if (threadIdx.x == 0 && s == 0) report(p.status, DFLASH_ERR_DEVICE);
    n_ctx = n_ctx < 0 ? 0 : cap;
  }
  const int nsplit = n_ctx > 0 ? (n_ctx + p.split - 1) / p.split : 1;
  const bool active = s < nsplit;   // inactive CTAs still join the cluster merge
  const int t0 = s * p.split;
  const int t1 = min(n_ctx, t0 + p.split);
  const int ctx_chunks = (active && t1 > t0) ? (t1 - t0 + CH - 1) / CH : 0;
  const bool has_block = active && (s == nsplit - 1);
  const int nchunks = ctx_chunks + (has_block ? 1 : 0);

  float O[HD];
#pragma unroll
  for (int i = 0; i < HD; ++i) O[i] = 0.f;
  float m = -INFINITY, l = 0.f;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nchunks > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(qfull, g * 2 * BLK * 128);
      for (int w = 0; w < g; ++w)
        for (int half = 0; half < 2; ++half)
          tma_load_2d(sQ + half * (MROWS * 128) + w * BLK * 128, &tmQ, qfull, (h * g + w) * HD + half * 64, b * BLK);
      int last_ci[ST];
      for (int i = 0; i < ST; ++i) last_ci[i] = -1;
      bool ok = true;
      for (int ci = 0; ci < nchunks; ++ci) {
        const int st = ci % ST;
        if (!mbar_wait(&empty[st], static_cast<uint32_t>(((ci / ST) & 1) ^ 1), abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        uint8_t *dk = sK + st * K_BYTES, *dv = sV + st * V_BYTES;
        const CUtensorMap *mk = &tmBK, *mv = &tmBV;
        int rowk = (b * p.nkv + h) * CH, rowv = (b * p.nkv + h) * HD;
        if (ci < ctx_chunks) {
          const int tok = t0 + ci * CH;
          const int page = p.page_table[static_cast<size_t>(b) * p.max_pages + tok / CH];
          if (page < 0 || page >= p.num_pages) {
            report(p.status, DFLASH_ERR_DEVICE);
            mbar_arrive(&full[st]);   // completes the phase with no data
            continue;
          }
          mk = &tmK;
          mv = &tmV;
          rowk = (page * p.nkv + h) * CH;
          rowv = (page * p.nkv + h) * HD;
        }
        mbar_arrive_expect_tx(&full[st], K_BYTES + V_BYTES);
        tma_load_2d(dk, mk, &full[st], 0, rowk);
        tma_load_2d(dk + K_BYTES / 2, mk, &full[st], 64, rowk);
        tma_load_2d(dv, mv, &full[st], 0, rowv);
        last_ci[st] = ci;
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        for (int i = 0; i < ST; ++i)   // let every issued copy land before smem goes away
          if (last_ci[i] >= 0) mbar_wait(&full[i], static_cast<uint32_t>((last_ci[i] / ST) & 1), nullptr, p.timeout_ns);
        mbar_wait(qfull, 0, nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nchunks > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(MROWS, CH);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(MROWS, HD);
      const uint32_t pv_tmem = tmem + 128;
      bool ok = mbar_wait(qfull, 0, abort_flag, p.timeout_ns);
      auto issue_qk = [&](int ci) -> bool {
        const int st = ci % ST, sb = ci & 1;
        if (!mbar_wait(&full[st], static_cast<uint32_t>((ci / ST) & 1), abort_flag, p.timeout_ns)) return false;
        if (!mbar_wait(&sempty[sb], static_cast<uint32_t>(((ci >> 1) & 1) ^ 1), abort_flag, p.timeout_ns)) return false;
        tc_fence_after();
        const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK + st * K_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16(tmem + sb * CH, sdesc_k_sw128(q0 + (kk >> 2) * (MROWS * 128) + (kk & 3) * 32),
                    sdesc_k_sw128(k0 + (kk >> 2) * (K_BYTES / 2) + (kk & 3) * 32), idesc_qk, kk > 0 ? 1u : 0u);
        umma_commit(&sfull[sb]);
        return true;
      };
      auto issue_pv = [&](int ci) -> bool {
        const int st = ci % ST, pb = ci & 1;
        // only the 16-token k-steps holding valid tokens: V columns past them
        // (block slots 16..63, the unused tail of a last page) are never read,
        // so whatever they hold cannot reach O through 0 * Inf
        const int valid = ci < ctx_chunks ? min(CH, t1 - (t0 + ci * CH)) : BLK;
        const int ksteps = (valid + 15) / 16;
        if (!mbar_wait(&pfull[pb], static_cast<uint32_t>((ci >> 1) & 1), abort_flag, p.timeout_ns)) return false;
        if (!mbar_wait(oempty, static_cast<uint32_t>((ci & 1) ^ 1), abort_flag, p.timeout_ns)) return false;
        tc_fence_after();
        const uint32_t p0 = smem_u32(sP + pb * P_BYTES), v0 = smem_u32(sV + st * V_BYTES);
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk)
          if (kk < ksteps)
            umma_bf16(pv_tmem, sdesc_k_sw128(p0 + kk * 32), sdesc_k_sw128(v0 + kk * 32), idesc_pv, kk > 0 ? 1u : 0u);
        umma_commit(ofull);
        umma_commit(&empty[st]);   // PV is the last reader of this KV stage
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int ci = 0; ci < nchunks && ok; ++ci) {
        if (ci + 1 < nchunks) ok = issue_qk(ci + 1);
        if (ok) ok = issue_pv(ci);
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(drain);   // every issued MMA retires before TMEM is released
      mbar_wait(drain, 0, nullptr, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax / O
    const int q = warp & 3;
    const int r = q * 32 + lane;            // query row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    float alpha_pending = 1.f;
    bool failed = false;
    for (int ci = 0; ci < nchunks; ++ci) {
      const int sb = ci & 1, pb = ci & 1;
      if (!mbar_wait(&sfull[sb], static_cast<uint32_t>((ci >> 1) & 1), abort_flag, p.timeout_ns)) {
        failed = true;
        break;
      }
      tc_fence_after();
      float sc[CH];
#pragma unroll
      for (int c = 0; c < CH / 16; ++c) {
        float v[16];
        tmem_ld16(lane_base + sb * CH + c * 16, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) sc[c * 16 + i] = v[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sb]);
      const int valid = ci < ctx_chunks ? min(CH, t1 - (t0 + ci * CH)) : BLK;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        sc[c] = c < valid ? sc[c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sc[c]);
      }
      const float mn = fmaxf(m, mx);
      const float alpha = fast_exp2(m - mn);
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        sc[c] = fast_exp2(sc[c] - mn);
        rs += sc[c];
      }
      l = l * alpha + rs;
      m = mn;
      // P row -> smem (bf16, 128-byte swizzled K-major A operand of PV)
      uint8_t *prow = sP + pb * P_BYTES + r * 128;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint4 u;
        u.x = pack_bf16(sc[8 * k + 0], sc[8 * k + 1]);
        u.y = pack_bf16(sc[8 * k + 2], sc[8 * k + 3]);
        u.z = pack_bf16(sc[8 * k + 4], sc[8 * k + 5]);
        u.w = pack_bf16(sc[8 * k + 6], sc[8 * k + 7]);
        *reinterpret_cast<uint4 *>(prow + ((k ^ (r & 7)) << 4)) = u;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[pb]);
      if (ci > 0) {   // fold in the previous chunk's PV (relative to that chunk's max)
        if (!mbar_wait(ofull, static_cast<uint32_t>((ci - 1) & 1), abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD / 16; ++c) {
          float v[16];
          tmem_ld16(lane_base + 128 + c * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) O[c * 16 + i] = O[c * 16 + i] * alpha_pending + v[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(oempty);
      }
      alpha_pending = alpha;
    }
    if (!failed && nchunks > 0) {
      if (mbar_wait(ofull, static_cast<uint32_t>((nchunks - 1) & 1), abort_flag, p.timeout_ns)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD / 16; ++c) {
          float v[16];
          tmem_ld16(lane_base + 128 + c * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) O[c * 16 + i] = O[c * 16 + i] * alpha_pending + v[i];
        }
        tc_fence_before();
      } else {
        failed = true;
      }
    }
    if (failed) {
      report(p.status, DFLASH_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  // all roles done: TMEM and the KV ring are free
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);

  const int qq = warp & 3;
  const int rr = qq * 32 + lane;
  const bool row_thread = warp >= 2 && rr < R;
  if (p.S == 1) {
    if (row_thread && nchunks > 0) {
      const int hq = h * g + rr / BLK, j = rr % BLK;
      const float inv = 1.f / l;
      const size_t o0 = static_cast<size_t>(b * BLK + j) * p.ldo + hq * HD;
#pragma unroll
      for (int c = 0; c < HD; c += 2) store2_hl(p.out, p.out_lo, o0 + c, O[c] * inv, O[c + 1] * inv);
    }
    return;
  }

  // ---- cluster merge: every CTA publishes (m, l, O) of its rows in its own
  // smem; after a cluster barrier CTA k finalises rows [k*R/S, (k+1)*R/S)
  // reading all S partials through distributed shared memory
  float *xo = reinterpret_cast<float *>(sK);            // [128][HD] partial O
  float *xml = xo + MROWS * HD;                           // [128][2] (max, sum)
  if (row_thread) {
#pragma unroll
    for (int c = 0; c < HD; c += 4)
      *reinterpret_cast<float4 *>(xo + rr * HD + c) = make_float4(O[c], O[c + 1], O[c + 2], O[c + 3]);
    xml[2 * rr] = m;
    xml[2 * rr + 1] = l;
  }
  cluster_sync();
  const int per = R / p.S;
  const int rank = static_cast<int>(cluster_ctarank());
  for (int it = threadIdx.x; it < per * (HD / 4); it += NTHR) {
    const int row = rank * per + it / (HD / 4), c4 = it % (HD / 4);
    float M = -INFINITY;
    float2 ml[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ml[k] = k < p.S ? ld_dsmem_f2(dsmem_addr(xml + 2 * row, k)) : make_float2(-INFINITY, 0.f);
      M = fmaxf(M, ml[k].x);
    }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k < p.S) {
        const float w = ml[k].y > 0.f ? fast_exp2(ml[k].x - M) : 0.f;
        L += w * ml[k].y;
        const float4 v = ld_dsmem_f4(dsmem_addr(xo + row * HD + 4 * c4, k));
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
    }
    const float inv = 1.f / L;
    const int hq = h * g + row / BLK, j = row % BLK;
    const size_t dst = static_cast<size_t>(b * BLK + j) * p.ldo + hq * HD + 4 * c4;
    store2_hl(p.out, p.out_lo, dst, acc.x * inv, acc.y * inv);
    store2_hl(p.out, p.out_lo, dst + 2, acc.z * inv, acc.w * inv);
  }
  cluster_sync();   // nobody leaves while others still read its smem
}

// ------------------------------------------------------------------ fp32
// K pages [page][nkv][slot][d]; V pages transposed [page][nkv][d][slot];
// block K [B][nkv][64][d], block V^T [B][nkv][d][64].
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
    int vstride;
    if (t < n) {
      const int pg = pt[static_cast<size_t>(b) * max_pages + t / page];
      if (pg < 0 || pg >= num_pages) {
        if (lane == 0) report(status, DFLASH_ERR_DEVICE);
        continue;
      }
      kp = kc + ((static_cast<size_t>(pg) * nkv + h) * page + t % page) * D;
      vp = vc + (static_cast<size_t>(pg) * nkv + h) * D * page + t % page;
      vstride = page;
    } else {
      kp = bk + ((static_cast<size_t>(b) * nkv + h) * 64 + (t - n)) * D;
      vp = bv + (static_cast<size_t>(b) * nkv + h) * D * 64 + (t - n);
      vstride = 64;
    }
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) d = fmaf(qv[i], kp[lane + 32 * i], d);
    const float sc = warp_sum(d) * scale;
    const float mn = fmaxf(m, sc);
    const float a = expf(m - mn), pw = expf(sc - mn);
    l = l * a + pw;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = acc[i] * a + pw * vp[static_cast<size_t>(lane + 32 * i) * vstride];
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
  if (a.max_splits != 1 && a.max_splits != 2 && a.max_splits != 4 && a.max_splits != 8)
    return set_error(DFLASH_ERR_UNSUPPORTED, "bf16 attention: splits per request must be 1, 2, 4 or 8");
  static bool attr_done = false;
  if (!attr_done) {
    if (int e = cuda_check(cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM),
                           "attention smem attribute"))
      return e;
    attr_done = true;
  }
  CUtensorMap tQ, tK, tV, tBK, tBV;
  const uint64_t kv_pages = static_cast<uint64_t>(a.num_pages) * a.nkv;
  const uint64_t bkv = static_cast<uint64_t>(a.B) * a.nkv;
  if (int e = make_tmap_2d(&tQ, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.nq) * HD,
                           static_cast<uint64_t>(a.B) * BLK, static_cast<uint64_t>(a.nq) * HD * 2, 64, BLK))
    return e;
  if (int e = make_tmap_2d(&tK, a.k_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, kv_pages * CH, HD * 2, 64, CH))
    return e;
  if (int e = make_tmap_2d(&tV, a.v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CH, kv_pages * HD, CH * 2, 64, HD))
    return e;
  if (int e = make_tmap_2d(&tBK, a.bk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, bkv * CH, HD * 2, 64, CH)) return e;
  if (int e = make_tmap_2d(&tBV, a.bv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CH, bkv * HD, CH * 2, 64, HD)) return e;
  Params p = {};
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.out_lo = static_cast<__nv_bfloat16 *>(a.out_lo);
  p.ldo = a.nq * HD;
  p.page_table = a.page_table;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.ctx_len = a.ctx_len;
  p.nkv = a.nkv;
  p.g = g;
  p.split = a.split_tokens;
  p.S = a.max_splits;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(HD)));
  p.status = lc.status;
  p.timeout_ns = lc.timeout_ns;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.max_splits, a.nkv, a.B);
  cfg.blockDim = dim3(NTHR);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.max_splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  ProfScope ps(lc, "attention", -1.0, -1.0);
  return cuda_check(cudaLaunchKernelEx(&cfg, attn_tc_kernel, tQ, tK, tV, tBK, tBV, p), "attention launch");
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

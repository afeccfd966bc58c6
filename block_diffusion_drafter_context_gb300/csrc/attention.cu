// Block attention of the DFlash drafter: the 16 block queries of a request
// attend, without any mask inside the block, to every injected context token
// of that request's paged KV cache and to the 16 block keys themselves
// ("DFlash" §2.2 parallel block diffusion; mask semantics of "FlexDraft",
// Metodologia 1: bidirectional in the block, all of the clean prefix, no
// other block).
//
// bf16 path - persistent, balanced split-KV, HBM-bound, on the 5th-generation
// tensor cores.  The work is the flat list of 64-token chunks (one KV page
// each) over (request, kv head): ceil(n_b/64) context chunks plus one chunk of
// the 16 block keys per (request, kv head).  One CTA per SM takes an equal
// contiguous run of that list, so ragged batches stay balanced and a CTA's
// pipeline never drains between requests.  Per CTA:
//   warp 0     TMA: K and V^T pages into a 6-deep smem ring (128-byte swizzle;
//              V pages are stored transposed so both products take K-major
//              operands); for g <= 4 also the 16g query rows of each new
//              (request, kv head), into shared memory;
//   warp 1     tcgen05.mma S = Q K^T (M=128, N=64, K=128) into one of three
//              TMEM score buffers; for g = 5..8 Q, the A operand, is read
//              from one of two TMEM Q buffers that the softmax warps fill a
//              (request, kv head) ahead;
//   warps 2-5  one TMEM lane (= query row) per thread: online softmax in the
//              exp2 domain, P written back to TMEM in bf16 (no shared memory:
//              that room holds the ring's depth, which the chunk's
//              load-to-PV lifetime needs to keep HBM busy).  O stays in TMEM;
//              it is rescaled only when a row's running max grows by more
//              than 2^8 (the exp2 values stay below 256 in between, exact in
//              fp32 sums);
//   warp 6     tcgen05.mma O += P V (M=128, N=128, K = the chunk's valid
//              tokens rounded up to 16), P, the A operand, read from TMEM.
// A (request, kv head) whose chunks all fall in one CTA is normalised and
// written directly.  One cut by a CTA boundary leaves (max, sum, O) partials
// in a small L2-resident scratch, and the last contributing CTA to arrive (a
// self-resetting per-(request, kv head) counter) merges them.
// fp32 path - plain CUDA-core loop for the tiny fp32 configuration.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace dflash {
namespace {

constexpr int CH = 64;                       // tokens per chunk (= one KV page)
constexpr int HD = 128;                      // head dim of the bf16 path
constexpr int ST = 6;                        // KV ring depth
constexpr int BLK = 16;                      // query rows per head in the tile (block size S <= 16 of them real)
constexpr int MROWS = 128;                   // UMMA M (query rows, padded)
constexpr int Q_BYTES = MROWS * HD * 2;      // 32 KB: shared-memory Q (g <= 4), two 64-dim halves of [128][64]
constexpr int K_BYTES = CH * HD * 2;         // 16 KB: two halves of [64 tok][64]
constexpr int V_BYTES = HD * CH * 2;         // 16 KB: [128 d][64 tok]
constexpr int CTRL_BYTES = 512;              // mbarriers, TMEM address, schedule
constexpr int SMEM = 1024 + Q_BYTES + ST * (K_BYTES + V_BYTES) + CTRL_BYTES;
constexpr int NTHR = 224;                    // producer, QK issuer, 4 softmax warps, PV issuer
constexpr int NSB = 3;                       // S buffers in TMEM: QK runs two chunks ahead
constexpr int TMEM_COLS = 512;   // S x 3 (64 columns each), Q at 192, O (128 columns) at 256, P x 2 at 384, Q at 448
constexpr uint32_t O_COL = 256;
constexpr uint32_t P_COL = 384;              // P buffers: 32 columns each (64 bf16 tokens per row)
// Q buffers in TMEM (g = 5..8: the QK product's A operand, 128 dims = 64
// columns per row), one per (request, kv head) in flight: the next one is
// written while the current one is read
__device__ __forceinline__ uint32_t q_col(int buf) { return buf ? 448u : 192u; }
constexpr float RESCALE_LOG2 = 8.f;
constexpr int DEFAULT_MIN_CHUNKS = 4;        // fewer CTAs than SMs when the whole list is short
static_assert(SMEM <= 232448, "attention smem over the per-block limit");

struct Params {
  const __nv_bfloat16 *q;  // [B*S][nq*HD] block queries (normed, rotated)
  __nv_bfloat16 *out;
  __nv_bfloat16 *out_lo;   // low halves (split activations) or null
  int ldo;
  const int32_t *page_table;
  int max_pages, num_pages;
  const int32_t *ctx_len;
  int B, nkv, g;
  int S;                   // block size: queries per request and block keys (2..16)
  int min_chunks;          // at least this many chunks per CTA
  int cs;                  // >1: cluster mode, cs CTAs (one cluster) per (request, kv head)
  float scale_log2;
  int *counters;           // [B * nkv], zero between launches
  float *partials;         // [gridDim.x * 2][ATTN_PART_FLOATS]
  int *status;
  unsigned long long timeout_ns;
};

// This CTA's run of the chunk list (written by warp 0, read by every role).
struct Sched {
  int b, h, k;             // first chunk: request, kv head, index in that list
  int n_mine;              // chunks in the run (0: idle CTA)
  long long lo, total;     // global index of the first chunk; list length
  int G;                   // CTAs that received a run
  int merge_flag;
};

// control block: mbarriers, TMEM address, abort flag, schedule
constexpr int N_MBAR = 3 + 2 * ST + 2 * NSB + 8;
static_assert(N_MBAR * 8 + 8 + sizeof(Sched) <= CTRL_BYTES, "attention control block overflows");

__device__ __forceinline__ int ctx_of(const Params &p, int b) {
  const int n = p.ctx_len[b], cap = p.max_pages * CH;
  return n < 0 ? 0 : (n > cap ? cap : n);
}
__device__ __forceinline__ int chunks_of(int n) { return (n + CH - 1) / CH + 1; }
__device__ __forceinline__ long long run_lo(int c, long long total, int G) {
  return static_cast<long long>(c) * total / G;
}
// the CTA whose run holds global chunk x
__device__ __forceinline__ int run_owner(long long x, long long total, int G) {
  return static_cast<int>(((x + 1) * G + total - 1) / total) - 1;
}

// Cursor over the chunk list: (request, kv head, chunk) in list order.
struct Walk {
  int b, h, k, n, nch;
  long long x;
  __device__ void init(const Params &p, const Sched &s) {
    b = s.b;
    h = s.h;
    k = s.k;
    n = ctx_of(p, b);
    nch = chunks_of(n);
    x = s.lo;
  }
  __device__ void next(const Params &p) {
    ++x;
    if (++k < nch) return;
    k = 0;
    if (++h < p.nkv) return;
    h = 0;
    if (++b < p.B) {
      n = ctx_of(p, b);
      nch = chunks_of(n);
    }
  }
  __device__ bool block_chunk() const { return k == nch - 1; }
  __device__ int valid(int S) const { return k < nch - 1 ? min(CH, n - k * CH) : S; }
};

// 16 consecutive outputs of one row: high bf16 halves and, if lo, low halves
__device__ __forceinline__ void store16_hl(__nv_bfloat16 *hi, __nv_bfloat16 *lo, const float (&v)[16], float s) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = v[2 * i] * s, b = v[2 * i + 1] * s;
    const __nv_bfloat162 hb = __floats2bfloat162_rn(a, b);
    h[i] = *reinterpret_cast<const uint32_t *>(&hb);
    l[i] = pack_bf16(a - __low2float(hb), b - __high2float(hb));
  }
  uint4 *dh = reinterpret_cast<uint4 *>(hi);
  dh[0] = make_uint4(h[0], h[1], h[2], h[3]);
  dh[1] = make_uint4(h[4], h[5], h[6], h[7]);
  if (lo) {
    uint4 *dl = reinterpret_cast<uint4 *>(lo);
    dl[0] = make_uint4(l[0], l[1], l[2], l[3]);
    dl[1] = make_uint4(l[4], l[5], l[6], l[7]);
  }
}

// Last arriver of a (request, kv head): combine the (max, sum, O) partials of
// contributor CTAs cf..cl for tile row `trow`, columns [c0, c0 + 64 * nq).
// A partial is O rows [128][HD] (row-major, fp32), max [128], sum [128];
// contributor cc's slot is 0 when this (request, head) is its first segment,
// which holds for every contributor but possibly the first.  The (max, sum)
// of up to 16 contributors load together; O of two contributors per round
// trip, 16 float4 per row half.
constexpr int MERGE_MAX = 16;
__device__ __noinline__ void merge_row(const Params &p, int cf, int cl, bool first_slot0, int trow, int c0, int nq64,
                                       __nv_bfloat16 *out, __nv_bfloat16 *out_lo) {
  auto part = [&](int cc) -> const float * {
    const int slot = (cc > cf || first_slot0) ? 0 : 1;
    return p.partials + (static_cast<size_t>(cc) * 2 + slot) * ATTN_PART_FLOATS;
  };
  const int np = cl - cf + 1;
  float mw[MERGE_MAX], lw[MERGE_MAX];
  float M = -INFINITY;
#pragma unroll
  for (int u = 0; u < MERGE_MAX; ++u) {
    mw[u] = u < np ? __ldcg(part(cf + u) + HD * MROWS + trow) : -INFINITY;
    lw[u] = u < np ? __ldcg(part(cf + u) + HD * MROWS + MROWS + trow) : 0.f;
  }
  for (int cc = cf + MERGE_MAX; cc <= cl; ++cc) M = fmaxf(M, __ldcg(part(cc) + HD * MROWS + trow));
#pragma unroll
  for (int u = 0; u < MERGE_MAX; ++u) M = fmaxf(M, mw[u]);
  float L = 0.f;
#pragma unroll
  for (int u = 0; u < MERGE_MAX; ++u) {
    mw[u] = u < np ? fast_exp2(mw[u] - M) : 0.f;   // now the contributor's weight
    L += mw[u] * lw[u];
  }
  for (int cc = cf + MERGE_MAX; cc <= cl; ++cc) {
    const float *pp = part(cc);
    L += fast_exp2(__ldcg(pp + HD * MROWS + trow) - M) * __ldcg(pp + HD * MROWS + MROWS + trow);
  }
  const float inv = 1.f / L;
  for (int h = 0; h < nq64; ++h) {          // 64-column halves of this lane's range
    const int cb = c0 + 64 * h;
    float acc[64];
#pragma unroll
    for (int t = 0; t < 64; ++t) acc[t] = 0.f;
    for (int cc = cf; cc <= cl; cc += 2) {
      const bool two = cc + 1 <= cl;
      const float4 *a = reinterpret_cast<const float4 *>(part(cc) + static_cast<size_t>(trow) * HD + cb);
      const float4 *b = reinterpret_cast<const float4 *>(part(two ? cc + 1 : cc) + static_cast<size_t>(trow) * HD + cb);
      float4 va[16], vb[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        va[t] = __ldcg(a + t);
        vb[t] = two ? __ldcg(b + t) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const int ua = cc - cf, ub = ua + 1;
      float wa = 0.f, wb = 0.f;
#pragma unroll
      for (int u = 0; u < MERGE_MAX; ++u) {   // register-array lookup without indexing
        wa = u == ua ? mw[u] : wa;
        wb = u == ub ? mw[u] : wb;
      }
      if (ua >= MERGE_MAX) wa = fast_exp2(__ldcg(part(cc) + HD * MROWS + trow) - M);
      if (two && ub >= MERGE_MAX) wb = fast_exp2(__ldcg(part(cc + 1) + HD * MROWS + trow) - M);
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        acc[4 * t + 0] = fmaf(wb, vb[t].x, fmaf(wa, va[t].x, acc[4 * t + 0]));
        acc[4 * t + 1] = fmaf(wb, vb[t].y, fmaf(wa, va[t].y, acc[4 * t + 1]));
        acc[4 * t + 2] = fmaf(wb, vb[t].z, fmaf(wa, va[t].z, acc[4 * t + 2]));
        acc[4 * t + 3] = fmaf(wb, vb[t].w, fmaf(wa, va[t].w, acc[4 * t + 3]));
      }
    }
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float v[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) v[t] = acc[16 * q4 + t];
      store16_hl(out + cb + 16 * q4, out_lo ? out_lo + cb + 16 * q4 : nullptr, v, inv);
    }
  }
}

// DUP (g <= 4): head w of the group owns TMEM quadrant w, and its 16 query
// rows are loaded twice (quadrant lanes 0-15 and 16-31), so S reaches both
// halves of the warp and the two lanes of a row each take 32 of a chunk's 64
// scores: every softmax warp works and each lane does half a row.
// Otherwise (g = 5..8): row 16w + j per lane over all 64 scores.
// Q: for g <= 4 the producer loads it into shared memory by TMA once the
// previous (request, kv head)'s QKs are done; for g = 5..8 the softmax warps
// write it into one of two TMEM buffers a segment ahead (the QK reads A from
// TMEM), which hides that reload and halves the shared-memory reads of QK.
// Measured per case: the TMEM form gained 5 % on 16k-32k contexts at g = 5
// and lost 3 % at g = 4 with 1k-8k contexts, where (request, kv head)
// switches are frequent.
template <bool DUP>
__global__ void __launch_bounds__(NTHR, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmBK,
                   const __grid_constant__ CUtensorMap tmBV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *base = smem_raw + pad;
  constexpr bool QT = !DUP;   // Q in TMEM
  uint8_t *sQ = base;
  uint8_t *sK = sQ + Q_BYTES;
  uint8_t *sV = sK + ST * K_BYTES;
  uint64_t *bar = reinterpret_cast<uint64_t *>(sV + ST * V_BYTES);
  uint64_t *qfull = bar, *qempty = bar + 2, *full = bar + 3, *empty = full + ST, *sfull = empty + ST,
           *sempty = sfull + NSB, *pfull = sempty + NSB, *pdone = pfull + 2, *oempty = pdone + 2,
           *mready = oempty + 1, *mdone = mready + 1, *drain = mdone + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  Sched *sch = reinterpret_cast<Sched *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.g;
  const int R = DUP ? 32 * g : BLK * g;     // TMEM lanes (= A rows) that hold query rows
  const int nact = (R + 31) / 32;           // softmax warps serving them

  if (threadIdx.x == 0) {
    mbar_init(&qfull[0], QT ? nact : 1);   // TMEM: written by the softmax warps; smem: by TMA
    mbar_init(&qfull[1], nact);
    mbar_init(qempty, 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], nact);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], nact);
      mbar_init(&pdone[i], 1);
    }
    mbar_init(oempty, nact);
    mbar_init(mready, nact);
    mbar_init(mdone, 1);
    mbar_init(drain, 2);   // both MMA issuers
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (!QT) {
    // A rows past R (query padding) are never touched by TMA: zero them once
    // so everything stays finite
    const int per_half = (MROWS - R) * 128 / 16;   // 16-byte chunks
    for (int i = threadIdx.x; i < 2 * per_half; i += NTHR) {
      const int half = i / per_half, k = i % per_half;
      *reinterpret_cast<uint4 *>(sQ + half * (MROWS * 128) + R * 128 + k * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 2 && warp <= 5) {
    // P and Q rows no softmax lane writes (quadrants without query rows,
    // query padding) enter the products too: zero both P and both Q buffers
    // of this warp's quadrant once
    const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    const uint32_t lz = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
#pragma unroll
    for (int c = 0; c < 64; c += 16) {
      tmem_st16_nw(lz + P_COL + c, z);
      if (QT) {
        tmem_st16_nw(lz + q_col(0) + c, z);
        tmem_st16_nw(lz + q_col(1) + c, z);
      }
    }
    tmem_wait_st();
    tc_fence_before();
  }

  pdl_start();
  // ---------------------------------------------------------------- schedule
  if (p.cs > 1) {
    // cluster mode: cluster = one (request, kv head); its cs CTAs split the
    // chunk list evenly and merge on chip at the end
    if (threadIdx.x == 0) {
      const int list = blockIdx.x / p.cs, r = blockIdx.x % p.cs;
      const int b = list / p.nkv;
      const int raw = p.ctx_len[b], cap = p.max_pages * CH;
      if (r == 0 && (raw < 0 || raw > cap)) report(p.status, DFLASH_ERR_DEVICE);
      const int nch = chunks_of(ctx_of(p, b));
      const int k0 = r * nch / p.cs, k1 = (r + 1) * nch / p.cs;
      sch->b = b;
      sch->h = list % p.nkv;
      sch->k = k0;
      sch->n_mine = k1 - k0;
      sch->lo = 0;
      sch->total = 0;
      sch->G = 0;
      sch->merge_flag = 0;
    }
  } else if (warp == 0) {
    // Lane i sums the chunk counts of a contiguous slice of the requests; a
    // warp scan gives the list length and the slice holding this CTA's start.
    const int per = (p.B + 31) / 32;
    const int b0 = min(p.B, lane * per), b1 = min(p.B, b0 + per);
    const int cap = p.max_pages * CH;
    long long sum = 0;
    for (int b = b0; b < b1; ++b) {
      const int raw = p.ctx_len[b];
      if (blockIdx.x == 0 && (raw < 0 || raw > cap)) report(p.status, DFLASH_ERR_DEVICE);
      sum += chunks_of(raw < 0 ? 0 : (raw > cap ? cap : raw));
    }
    long long inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    const long long total = __shfl_sync(0xffffffffu, inc, 31) * p.nkv;
    const long long want = (total + p.min_chunks - 1) / p.min_chunks;
    const int G = static_cast<int>(want < static_cast<long long>(gridDim.x) ? (want < 1 ? 1 : want) : gridDim.x);
    const int c = blockIdx.x;
    const long long lo = c < G ? run_lo(c, total, G) : 0, hi = c < G ? run_lo(c + 1, total, G) : 0;
    const long long ex = (inc - sum) * p.nkv, in = inc * p.nkv;
    if (lane == 0) {
      sch->n_mine = static_cast<int>(hi - lo);
      sch->lo = lo;
      sch->total = total;
      sch->G = G;
      sch->merge_flag = 0;
    }
    if (c < G && lo >= ex && lo < in) {   // exactly one lane: the slices partition the list
      long long pre = ex;
      for (int b = b0; b < b1; ++b) {
        const int nch = chunks_of(ctx_of(p, b));
        const long long span = static_cast<long long>(nch) * p.nkv;
        if (lo < pre + span) {
          const long long off = lo - pre;
          sch->b = b;
          sch->h = static_cast<int>(off / nch);
          sch->k = static_cast<int>(off % nch);
          break;
        }
        pre += span;
      }
    }
  }
  __syncthreads();
  const Sched sc = *sch;
  const int n = sc.n_mine;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol_kv = policy_evict_first();
      Walk w;
      w.init(p, sc);
      int last_ci[ST];
      for (int i = 0; i < ST; ++i) last_ci[i] = -1;
      int seg = -1, q_issued = -1;
      bool ok = true;
      for (int i = 0; i < n; ++i) {
        const int st = i % ST;
        const bool first = i == 0 || w.k == 0;
        if (first) ++seg;
        if (!mbar_wait(&empty[st], static_cast<uint32_t>(((i / ST) & 1) ^ 1), abort_flag, p.timeout_ns)) {
          ok = false;
          break;
        }
        // the KV page first: it streams while the previous (request, head) drains
        const CUtensorMap *mk = &tmBK, *mv = &tmBV;
        int rowk = (w.b * p.nkv + w.h) * CH, rowv = (w.b * p.nkv + w.h) * HD;
        bool load = true;
        if (!w.block_chunk()) {
          const int page = p.page_table[static_cast<size_t>(w.b) * p.max_pages + w.k];
          if (page < 0 || page >= p.num_pages) {
            report(p.status, DFLASH_ERR_DEVICE);
            mbar_arrive(&full[st]);   // completes the phase with no data
            load = false;
          } else {
            mk = &tmK;
            mv = &tmV;
            rowk = (page * p.nkv + w.h) * CH;
            rowv = (page * p.nkv + w.h) * HD;
          }
        }
        if (load) {   // K/V pages are read once per step: evict first
          uint8_t *dk = sK + st * K_BYTES, *dv = sV + st * V_BYTES;
          mbar_arrive_expect_tx(&full[st], K_BYTES + V_BYTES);
          tma_load_2d_hint(dk, mk, &full[st], 0, rowk, pol_kv);
          tma_load_2d_hint(dk + K_BYTES / 2, mk, &full[st], 64, rowk, pol_kv);
          tma_load_2d_hint(dv, mv, &full[st], 0, rowv, pol_kv);
          last_ci[st] = i;
        }
        if (!QT && first) {   // the query rows of this (request, kv head), once its predecessor's QKs are done
          if (seg > 0 && !mbar_wait(qempty, static_cast<uint32_t>((seg - 1) & 1), abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(qfull, (DUP ? 2 : 1) * g * 2 * BLK * 128);
          for (int hw = 0; hw < g; ++hw)
            for (int half = 0; half < 2; ++half) {
              const int col = (w.h * g + hw) * HD + half * 64;
              uint8_t *dst = sQ + half * (MROWS * 128) + (DUP ? 32 : BLK) * hw * 128;
              tma_load_2d(dst, &tmQ, qfull, col, w.b * p.S);   // rows past S: the next request's, unused
              if (DUP) tma_load_2d(dst + BLK * 128, &tmQ, qfull, col, w.b * p.S);
            }
          q_issued = seg;
        }
        w.next(p);
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
        for (int i = 0; i < ST; ++i)   // let every issued copy land before smem goes away
          if (last_ci[i] >= 0)
            mbar_wait(&full[i], static_cast<uint32_t>((last_ci[i] / ST) & 1), nullptr, p.timeout_ns);
        if (q_issued >= 0) mbar_wait(qfull, static_cast<uint32_t>(q_issued & 1), nullptr, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    // (one thread issues a tcgen05.mma about every 100 cycles, so QK and PV
    // have an issuing warp each and overlap on the tensor core)
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(MROWS, CH);
      Walk wq;
      wq.init(p, sc);
      int seg_q = -1;
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const int st = i % ST, sb = i % NSB;
        const bool first = i == 0 || wq.k == 0;
        const bool last = i == n - 1 || wq.k == wq.nch - 1;
        if (first) ++seg_q;
        // this (request, kv head)'s query rows: TMEM Q buffer seg_q & 1,
        // filled by the softmax warps for the (seg_q >> 1)-th time, or the
        // shared-memory Q, filled by TMA for the seg_q-th time
        const int qb = QT ? (seg_q & 1) : 0;
        const uint32_t qpar = static_cast<uint32_t>((QT ? seg_q >> 1 : seg_q) & 1);
        ok = mbar_wait(&full[st], static_cast<uint32_t>((i / ST) & 1), abort_flag, p.timeout_ns) &&
             (!first || mbar_wait(&qfull[qb], qpar, abort_flag, p.timeout_ns)) &&
             mbar_wait(&sempty[sb], static_cast<uint32_t>(((i / NSB) & 1) ^ 1), abort_flag, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t k0 = smem_u32(sK + st * K_BYTES);
        if constexpr (QT) {
          const uint32_t qa = tmem + q_col(qb);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)   // A = Q from TMEM: 16 dims = 8 columns per k-step
            umma_bf16_ts(tmem + sb * CH, qa + static_cast<uint32_t>(kk * 8),
                         sdesc_k_sw128(k0 + (kk >> 2) * (K_BYTES / 2) + (kk & 3) * 32), idesc_qk, kk > 0 ? 1u : 0u);
        } else {
          const uint32_t q0 = smem_u32(sQ);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16(tmem + sb * CH, sdesc_k_sw128(q0 + (kk >> 2) * (MROWS * 128) + (kk & 3) * 32),
                      sdesc_k_sw128(k0 + (kk >> 2) * (K_BYTES / 2) + (kk & 3) * 32), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&sfull[sb]);
        if (!QT && last) umma_commit(qempty);   // the shared-memory Q may take the next (request, head)
        wq.next(p);
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(drain);   // every issued MMA retires before TMEM is released
      mbar_wait(drain, 0, nullptr, p.timeout_ns);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(MROWS, HD);
      Walk wp;
      wp.init(p, sc);
      int seg_p = -1;
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const int st = i % ST, pb = i & 1;
        const bool first = i == 0 || wp.k == 0;
        if (first) ++seg_p;
        // only the 16-token k-steps holding valid tokens: V columns past them
        // (block slots 16..63, the unused tail of a last page) are never read,
        // so whatever they hold cannot reach O through 0 * Inf
        const int ksteps = (wp.valid(p.S) + 15) / 16;
        ok = mbar_wait(&pfull[pb], static_cast<uint32_t>((i >> 1) & 1), abort_flag, p.timeout_ns) &&
             mbar_wait(&full[st], static_cast<uint32_t>((i / ST) & 1), abort_flag, p.timeout_ns) &&
             (!first || seg_p == 0 ||
              mbar_wait(oempty, static_cast<uint32_t>((seg_p - 1) & 1), abort_flag, p.timeout_ns));
        if (!ok) break;
        tc_fence_after();
        const uint32_t pt = tmem + P_COL + static_cast<uint32_t>(pb * 32), v0 = smem_u32(sV + st * V_BYTES);
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk)   // A = P from TMEM: 16 tokens = 8 columns per k-step
          if (kk < ksteps)
            umma_bf16_ts(tmem + O_COL, pt + static_cast<uint32_t>(kk * 8), sdesc_k_sw128(v0 + kk * 32), idesc_pv,
                         (kk > 0 || !first) ? 1u : 0u);
        umma_commit(&pdone[pb]);
        umma_commit(&empty[st]);   // PV is the last reader of this KV stage (its QK finished before P existed)
        wp.next(p);
      }
      if (!ok) {
        report(p.status, DFLASH_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr, p.timeout_ns);
    }
  } else if ((warp & 3) * 32 < R && n > 0) {
    // ------------------------------------------------------------ softmax
    constexpr int NC = DUP ? CH / 2 : CH;           // scores per lane
    const int q = warp & 3;
    const int hi = DUP ? lane >> 4 : 0;             // DUP: second half of the chunk's columns
    const int lrow = DUP ? q * 32 + (lane & 15) : q * 32 + lane;   // P / O row (TMEM lane) this lane serves
    const int trow = DUP ? q * BLK + (lane & 15) : lrow;          // tile row 16 * head + position
    const bool real = trow < BLK * g;
    const bool olane = DUP ? lane < 16 : real;      // lanes whose own TMEM lane holds a real O row
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    Walk w;
    w.init(p, sc);
    int seg = -1, nparts = 0;
    bool seg_whole = false, failed = false;
    float m = -INFINITY, l = 0.f;   // running max (scaled, log2 domain) and sum of this lane's row
    auto waitw = [&](uint64_t *b, uint32_t par) -> bool {   // warp-uniform bounded wait
      const bool ok = mbar_wait(b, par, abort_flag, p.timeout_ns);
      return !__any_sync(0xffffffffu, !ok);
    };
    // The query rows of (request bt, kv head ht) into Q buffer qb, this
    // lane's TMEM lane holding row qj of the group's query head qhw (both
    // lanes of a DUP pair hold it); rows past the block size stay zero.
    // Column c holds dims 2c (low half) and 2c + 1: the A layout of QK.
    const int qhw = DUP ? q : trow / BLK, qj = DUP ? (lane & 15) : trow % BLK;
    auto write_q = [&](int bt, int ht, int qb) {
      const bool live = qhw < g && qj < p.S;
      const uint4 *src = reinterpret_cast<const uint4 *>(
          p.q + (static_cast<size_t>(bt) * p.S + qj) * (static_cast<size_t>(p.nkv) * g * HD) +
          static_cast<size_t>(ht * g + qhw) * HD);
      uint4 u[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) u[t] = live ? __ldg(src + t) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {   // 16 columns per store
        uint32_t wv[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          wv[4 * t] = u[4 * c4 + t].x;
          wv[4 * t + 1] = u[4 * c4 + t].y;
          wv[4 * t + 2] = u[4 * c4 + t].z;
          wv[4 * t + 3] = u[4 * c4 + t].w;
        }
        tmem_st16_nw(lane_base + q_col(qb) + static_cast<uint32_t>(16 * c4), wv);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qfull[qb]);
    };
    for (int i = 0; i < n; ++i) {
      const int sb = i % NSB;
      const bool first = i == 0 || w.k == 0;
      const bool last = i == n - 1 || w.k == w.nch - 1;
      if (first) {
        ++seg;
        seg_whole = w.k == 0;
        // Q of this segment (the first one only: the others were written a
        // segment ahead); the next one's follows this chunk's P
        if (QT && i == 0) write_q(w.b, w.h, 0);
      }
      const int valid = w.valid(p.S);
      if (!waitw(&sfull[sb], static_cast<uint32_t>((i / NSB) & 1))) {
        failed = true;
        break;
      }
      tc_fence_after();
      float x[NC];
      {
        uint32_t r0[16], r1[16], r2[16], r3[16];   // the four loads in flight together
        tmem_ld16_nw(lane_base + sb * CH, r0);
        tmem_ld16_nw(lane_base + sb * CH + 16, r1);
        tmem_ld16_nw(lane_base + sb * CH + 32, r2);
        tmem_ld16_nw(lane_base + sb * CH + 48, r3);
        tmem_wait_ld();
        tmem_regs_ready(r0);
        tmem_regs_ready(r1);
        tmem_regs_ready(r2);
        tmem_regs_ready(r3);
#pragma unroll
        for (int c = 0; c < NC; ++c) {   // DUP: lanes 16-31 take columns 32..63 (a select, no indexing)
          const uint32_t a = c < 16 ? r0[c & 15] : c < 32 ? r1[c & 15] : c < 48 ? r2[c & 15] : r3[c & 15];
          const uint32_t b = c < 16 ? r2[c & 15] : r3[c & 15];
          x[c] = __uint_as_float((DUP && hi) ? b : a);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sb]);
      if (valid < CH) {   // last page or block keys: mask the columns past the valid tokens
        const int c0 = hi * NC;
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (c0 + c >= valid) x[c] = -INFINITY;
      }
      float mx;
      {
        float a0 = x[0], a1 = x[1], a2 = x[2], a3 = x[3];
#pragma unroll
        for (int c = 4; c < NC; c += 4) {
          a0 = fmaxf(a0, x[c]);
          a1 = fmaxf(a1, x[c + 1]);
          a2 = fmaxf(a2, x[c + 2]);
          a3 = fmaxf(a3, x[c + 3]);
        }
        mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
        if (DUP) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      }
      const float mxs = mx * p.scale_log2;
      if (first) {
        m = mxs;
        l = 0.f;
      } else {
        const bool need = mxs > m + RESCALE_LOG2;
        if (__any_sync(0xffffffffu, need)) {   // O holds chunks up to i-1: wait for that PV, rescale in TMEM
          if (!waitw(&pdone[(i - 1) & 1], static_cast<uint32_t>(((i - 1) >> 1) & 1))) {
            failed = true;
            break;
          }
          tc_fence_after();
          const float f = need ? fast_exp2(m - mxs) : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < HD / 16; c0 += 4) {   // four loads in flight, then four stores
            uint32_t ov[4][16];
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld16_nw(lane_base + O_COL + (c0 + u) * 16, ov[u]);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              tmem_regs_ready(ov[u]);
#pragma unroll
              for (int j = 0; j < 16; ++j) ov[u][j] = __float_as_uint(__uint_as_float(ov[u][j]) * f);
              tmem_st16_nw(lane_base + O_COL + (c0 + u) * 16, ov[u]);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          if (need) {
            l *= f;
            m = mxs;
          }
        }
      }
      const float nm = -m;
      float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
      for (int c = 0; c < NC; c += 4) {
        x[c] = fast_exp2(fmaf(x[c], p.scale_log2, nm));
        x[c + 1] = fast_exp2(fmaf(x[c + 1], p.scale_log2, nm));
        x[c + 2] = fast_exp2(fmaf(x[c + 2], p.scale_log2, nm));
        x[c + 3] = fast_exp2(fmaf(x[c + 3], p.scale_log2, nm));
        r0 += x[c];
        r1 += x[c + 1];
        r2 += x[c + 2];
        r3 += x[c + 3];
      }
      float rs = (r0 + r1) + (r2 + r3);
      if (DUP) rs += __shfl_xor_sync(0xffffffffu, rs, 16);
      l += rs;
      // P buffer i&1 was last read by the PV of chunk i-2
      if (i >= 2 && !waitw(&pdone[i & 1], static_cast<uint32_t>(((i - 2) >> 1) & 1))) {
        failed = true;
        break;
      }
      tc_fence_after();
      // P in bf16 into this lane's row of P buffer i & 1: column j holds
      // tokens 2j (low half) and 2j + 1, the A layout of the PV product
      {
        uint32_t pw[32];
        if constexpr (DUP) {
          // each lane of a pair holds half the row: trade halves with the
          // partner (lane ^ 16) so both write the whole row (lanes 16-31
          // into the duplicate rows, whose O nobody reads)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t mine = pack_bf16(x[2 * j], x[2 * j + 1]);
            const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 16);
            pw[j] = hi ? other : mine;
            pw[16 + j] = hi ? mine : other;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) pw[j] = pack_bf16(x[2 * j], x[2 * j + 1]);
        }
        const uint32_t pcol = lane_base + P_COL + static_cast<uint32_t>((i & 1) * 32);
        uint32_t w0[16], w1[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          w0[j] = pw[j];
          w1[j] = pw[16 + j];
        }
        tmem_st16_nw(pcol, w0);
        tmem_st16_nw(pcol + 16, w1);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[i & 1]);
      // the next (request, kv head)'s Q, if the run reaches it, into the
      // other buffer: it held the previous segment's Q, whose QKs all
      // completed before this warp consumed their scores.  Written after the
      // P of this segment's first chunk, so the loads overlap its PV.
      if (QT && first && (n - i) - (w.nch - w.k) > 0) {
        const bool nb = w.h + 1 < p.nkv;
        write_q(nb ? w.b : w.b + 1, nb ? w.h + 1 : 0, (seg + 1) & 1);
      }

      if (last) {
        // ---- end of this CTA's part of a (request, kv head)
        if (!waitw(&pdone[i & 1], static_cast<uint32_t>((i >> 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
        const bool whole = p.cs <= 1 && seg_whole && w.k == w.nch - 1;
        if (p.cs > 1) {
          // cluster mode: (max, sum, O) of this CTA's share into its own smem
          // (the K ring is idle: every QK has completed) for the on-chip merge
          float *xo = reinterpret_cast<float *>(sK);
#pragma unroll
          for (int c0 = 0; c0 < HD / 16; c0 += 4) {
            uint32_t ov[4][16];
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld16_nw(lane_base + O_COL + (c0 + u) * 16, ov[u]);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              tmem_regs_ready(ov[u]);
              if (olane) {
                float4 *d4 = reinterpret_cast<float4 *>(xo + trow * HD + (c0 + u) * 16);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                  d4[t] = make_float4(__uint_as_float(ov[u][4 * t]), __uint_as_float(ov[u][4 * t + 1]),
                                      __uint_as_float(ov[u][4 * t + 2]), __uint_as_float(ov[u][4 * t + 3]));
              }
            }
          }
          if (olane) reinterpret_cast<float2 *>(xo + MROWS * HD)[trow] = make_float2(m, l);
          tc_fence_before();
          w.next(p);
          continue;
        }
        const int hq = w.h * g + trow / BLK, j = trow % BLK;
        const bool out_row = j < p.S;   // tile rows past the block size are not queries
        const size_t orow = static_cast<size_t>(w.b * p.S + j) * p.ldo + static_cast<size_t>(hq) * HD;
        float *part = p.partials + (static_cast<size_t>(blockIdx.x) * 2 + (seg == 0 ? 0 : 1)) * ATTN_PART_FLOATS;
        const float inv = 1.f / l;
#pragma unroll
        for (int c0 = 0; c0 < HD / 16; c0 += 4) {   // four loads in flight
          uint32_t ov[4][16];
#pragma unroll
          for (int u = 0; u < 4; ++u) tmem_ld16_nw(lane_base + O_COL + (c0 + u) * 16, ov[u]);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            tmem_regs_ready(ov[u]);
            const int c = c0 + u;
            float v[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(ov[u][t]);
            if (olane) {
              if (whole) {
                if (out_row) store16_hl(p.out + orow + c * 16, p.out_lo ? p.out_lo + orow + c * 16 : nullptr, v, inv);
              } else {
                float4 *d4 = reinterpret_cast<float4 *>(part + static_cast<size_t>(trow) * HD + c * 16);
#pragma unroll
                for (int t = 0; t < 4; ++t) d4[t] = make_float4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(oempty);   // the next (request, head) may overwrite O
        if (!whole) {
          if (olane) {
            part[HD * MROWS + trow] = m;
            part[HD * MROWS + MROWS + trow] = l;
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) mbar_arrive(mready);
          const long long start = w.x - w.k, end = start + w.nch;
          const int cf = run_owner(start, sc.total, sc.G), cl = run_owner(end - 1, sc.total, sc.G);
          if (q == 0 && lane == 0) {
            int flag = 0;
            if (mbar_wait(mready, static_cast<uint32_t>(nparts & 1), abort_flag, p.timeout_ns)) {
              __threadfence();
              int *ctr = p.counters + w.b * p.nkv + w.h;
              const int old = atomicAdd(ctr, 1);
              if (old == cl - cf) {   // every contributor's partial is in: merge here
                atomicExch(ctr, 0);
                __threadfence();
                flag = 1;
              }
            }
            sch->merge_flag = flag;
            mbar_arrive(mdone);
          }
          if (!waitw(mdone, static_cast<uint32_t>(nparts & 1))) {
            failed = true;
            break;
          }
          ++nparts;
          if (sch->merge_flag && real && out_row)   // DUP: the two lanes of a row take 64 columns each
            merge_row(p, cf, cl, run_lo(cf, sc.total, sc.G) == start, trow, DUP ? hi * 64 : 0, DUP ? 1 : 2,
                      p.out + orow, p.out_lo ? p.out_lo + orow : nullptr);
        }
      }
      w.next(p);
    }
    if (failed) {
      report(p.status, DFLASH_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  }
  if (p.cs > 1 && n == 0 && warp >= 2 && warp <= 5) {   // an empty share: weight 0 in the merge
    const int t = threadIdx.x - 64;
    if (t < MROWS) reinterpret_cast<float2 *>(reinterpret_cast<float *>(sK) + MROWS * HD)[t] = make_float2(-INFINITY, 0.f);
  }

  // all roles done: TMEM and the KV ring are free
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);

  if (p.cs > 1) {
    // ---- cluster merge through distributed shared memory: CTA r finalises
    // tile rows [r*R/cs, (r+1)*R/cs) from the cs shares (16g real rows)
    cluster_sync();
    const float *xo = reinterpret_cast<const float *>(sK);
    const float2 *xml = reinterpret_cast<const float2 *>(xo + MROWS * HD);
    const int rows = BLK * g, rank = static_cast<int>(cluster_ctarank());
    const int r0 = rank * rows / p.cs, r1 = (rank + 1) * rows / p.cs;
    const int b = sch->b, h = sch->h;
    for (int it = threadIdx.x; it < (r1 - r0) * (HD / 4); it += NTHR) {
      const int row = r0 + it / (HD / 4), c4 = it % (HD / 4);
      float2 ml[8];
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ml[k] = k < p.cs ? ld_dsmem_f2(dsmem_addr(xml + row, k)) : make_float2(-INFINITY, 0.f);
        M = fmaxf(M, ml[k].x);
      }
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < p.cs && ml[k].y > 0.f) {
          const float wk = fast_exp2(ml[k].x - M);
          L += wk * ml[k].y;
          const float4 v = ld_dsmem_f4(dsmem_addr(xo + row * HD + 4 * c4, k));
          acc.x += wk * v.x;
          acc.y += wk * v.y;
          acc.z += wk * v.z;
          acc.w += wk * v.w;
        }
      }
      const float inv = 1.f / L;
      const int hq = h * g + row / BLK, j = row % BLK;
      if (j >= p.S) continue;   // not a query of this block size
      const size_t dst = static_cast<size_t>(b * p.S + j) * p.ldo + static_cast<size_t>(hq) * HD + 4 * c4;
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      const __nv_bfloat162 h1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2 *>(p.out + dst) =
          make_uint2(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1));
      if (p.out_lo)
        *reinterpret_cast<uint2 *>(p.out_lo + dst) =
            make_uint2(pack_bf16(acc.x * inv - __low2float(h0), acc.y * inv - __high2float(h0)),
                       pack_bf16(acc.z * inv - __low2float(h1), acc.w * inv - __high2float(h1)));
    }
    cluster_sync();   // no CTA leaves while others still read its shares
  }
}

// ------------------------------------------------------------------ fp32
// K pages [page][nkv][slot][d]; V pages transposed [page][nkv][d][slot];
// block K [B][nkv][64][d], block V^T [B][nkv][d][64].
template <int DPL>
__global__ void __launch_bounds__(512) attn_f32_kernel(const float *q, int ldq, const float *kc, const float *vc,
                                                       const float *bk, const float *bv, const int32_t *pt,
                                                       int max_pages, int num_pages, int page, const int32_t *ctx_len,
                                                       float *out, int ldo, int nkv, int g, int S, float scale,
                                                       int *status) {
  pdl_start();
  constexpr int D = DPL * 32;
  const int hq = blockIdx.x, b = blockIdx.y, j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (j >= S) return;   // one warp per query of the block
  const int h = hq / g;
  int n = ctx_len[b];
  if (n < 0 || n > max_pages * page) {
    if (threadIdx.x == 0 && hq == 0) report(status, DFLASH_ERR_DEVICE);
    n = n < 0 ? 0 : max_pages * page;
  }
  float qv[DPL], acc[DPL];
  const float *qr = q + static_cast<size_t>(b * S + j) * ldq + hq * D;
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    qv[i] = qr[lane + 32 * i];
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int t = 0; t < n + S; ++t) {
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
  float *orow = out + static_cast<size_t>(b * S + j) * ldo + hq * D;
#pragma unroll
  for (int i = 0; i < DPL; ++i) orow[lane + 32 * i] = acc[i] / l;
}

}  // namespace


int attention_bf16(const Launch &lc, const AttnArgs &a) {
  if (a.B <= 0) return DFLASH_OK;
  if (a.S < 2 || a.S > BLK) return set_error(DFLASH_ERR_UNSUPPORTED, "attention: block size must be 2..16");
  if (a.d != HD || a.page_size != CH)
    return set_error(DFLASH_ERR_UNSUPPORTED, "bf16 attention needs head_dim 128 and 64-token pages");
  const int g = a.nq / a.nkv;
  if (g < 1 || g > 8 || g * a.nkv != a.nq)
    return set_error(DFLASH_ERR_UNSUPPORTED, "bf16 attention: q heads per kv head must be 1..8");
  if (!a.counters || !a.partials) return set_error(DFLASH_ERR_ARG, "bf16 attention: scratch missing");
  const int grid = lc.num_sms;
  if (a.partial_slots < 2ull * grid) return set_error(DFLASH_ERR_SHAPE, "bf16 attention: partial scratch too small");
  if (static_cast<size_t>(a.B) * a.nkv > a.counter_cap)
    return set_error(DFLASH_ERR_SHAPE, "bf16 attention: batch x kv heads over the counter capacity");
  // set on every call: per device, idempotent, a host call (no stream work)
  if (int e = cuda_check(cudaFuncSetAttribute(g <= 4 ? attn_tc_kernel<true> : attn_tc_kernel<false>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM),
                         "attention smem attribute"))
    return e;
  CUtensorMap tQ, tK, tV, tBK, tBV;
  const uint64_t kv_pages = static_cast<uint64_t>(a.num_pages) * a.nkv;
  const uint64_t bkv = static_cast<uint64_t>(a.B) * a.nkv;
  if (int e = make_tmap_2d(&tQ, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.nq) * HD,
                           static_cast<uint64_t>(a.B) * a.S, static_cast<uint64_t>(a.nq) * HD * 2, 64, BLK))
    return e;
  if (int e = make_tmap_2d(&tK, a.k_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, kv_pages * CH, HD * 2, 64, CH))
    return e;
  if (int e = make_tmap_2d(&tV, a.v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CH, kv_pages * HD, CH * 2, 64, HD))
    return e;
  if (int e = make_tmap_2d(&tBK, a.bk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, HD, bkv * CH, HD * 2, 64, CH)) return e;
  if (int e = make_tmap_2d(&tBV, a.bv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CH, bkv * HD, CH * 2, 64, HD)) return e;
  Params p = {};
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.out_lo = static_cast<__nv_bfloat16 *>(a.out_lo);
  p.ldo = a.nq * HD;
  p.page_table = a.page_table;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.ctx_len = a.ctx_len;
  p.B = a.B;
  p.nkv = a.nkv;
  p.g = g;
  p.S = a.S;
  p.min_chunks = a.min_chunks > 0 ? a.min_chunks : DEFAULT_MIN_CHUNKS;
  // few (request, kv head) lists: one cluster of cs CTAs per list, merged on
  // chip (global round trips cost ~2 us here); otherwise the balanced
  // persistent split.  A forced split length (test hook) means persistent.
  const long long lists = static_cast<long long>(a.B) * a.nkv;
  int cs = 1;
  if (a.min_chunks <= 0)
    while (cs < 8 && lists * cs * 2 <= grid) cs *= 2;
  p.cs = cs;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(HD)));
  p.counters = a.counters;
  p.partials = a.partials;
  p.status = lc.status;
  p.timeout_ns = lc.timeout_ns;
  ProfScope ps(lc, "attention", -1.0, -1.0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs > 1 ? static_cast<unsigned>(lists * cs) : static_cast<unsigned>(grid));
  cfg.blockDim = dim3(NTHR);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cuda_check(cudaLaunchKernelEx(&cfg, g <= 4 ? attn_tc_kernel<true> : attn_tc_kernel<false>, tQ, tK, tV, tBK,
                                       tBV, p),
                    "attention launch");
}

int attention_f32(const Launch &lc, const AttnArgs &a) {
  if (a.B <= 0) return DFLASH_OK;
  if (a.S < 2 || a.S > BLK) return set_error(DFLASH_ERR_UNSUPPORTED, "attention: block size must be 2..16");
  const int g = a.nq / a.nkv;
  dim3 grid(a.nq, a.B), block(512);
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(a.d)));
  ProfScope ps(lc, "attention", -1.0, -1.0);
  const float *q = static_cast<const float *>(a.q);
  float *o = static_cast<float *>(a.out);
#define ARGS q, a.nq * a.d, static_cast<const float *>(a.k_cache), static_cast<const float *>(a.v_cache), \
             static_cast<const float *>(a.bk), static_cast<const float *>(a.bv), a.page_table, a.max_pages, \
             a.num_pages, a.page_size, a.ctx_len, o, a.nq * a.d, a.nkv, g, a.S, scale, lc.status
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

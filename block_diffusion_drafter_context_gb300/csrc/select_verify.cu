// DFlash-2 Path Selector and greedy verification.
//
// Path Selector ("DFlash 2", Arquitectura del Sistema item 1): every pair of
// adjacent candidates is scored, all pairs in parallel, by the drafter logit
// of the current candidate plus a low-rank bilinear compatibility of the two
// tokens' 256-d embeddings under a context gate:
//   s[j][p][c] = z_j[c] + sigmoid(w_g . h_j + b_g) * (A e256[p]) . (B e256[c])
// (p over position j-1's candidates, the anchor for the first mask position;
// c over position j's).  The greedy traversal then walks the 15 positions,
// each time taking the best continuation of the previous choice (ties to the
// lower token id).
//
// Greedy verification ("DFlash 2", Flujo de Inferencia steps 4-5; "DFlash en
// NVIDIA Blackwell", Contexto tecnico): the accepted length is the longest
// prefix on which draft and target agree; the target token at the first
// mismatch is the bonus; committed = accepted drafts + bonus, then -1.
#include "common.cuh"
#include "internal.h"

namespace dflash {
namespace {

constexpr int K = 16;   // candidates per position
// J = block size - 1 mask positions per request (1..15) is a runtime argument.

// grid (15 positions, B); 256 threads.  The 32 tokens' embeddings and the
// two rank-r projections are staged in chunks of ECH embedding columns
// (A^T, B^T with a padded pitch: conflict-free), each warp owns 4 of the 32
// rows and each lane one rank index, so u(p) = A e[p] and w(c) = B e[c] are
// shared-memory dot products with no dependent global loads.
constexpr int ECH = 128;
template <typename T>
__global__ void __launch_bounds__(256) pair_scores_kernel(const int32_t *anchor, const int32_t *topk_ids,
                                                          const float *topk_logits, const T *hfinal, int H,
                                                          const T *e256, const T *A, const T *Bm, int r, int E,
                                                          const float *w_g, float b_g, int J, float *scores) {
  pdl_start();
  extern __shared__ float sh[];
  const int rp = r + 1;
  float *se = sh;                     // [32][ECH]: rows 0..15 previous, 16..31 current
  float *smt = se + 32 * ECH;         // [2][ECH][rp]: A^T, B^T chunk
  float *su = smt + 2 * ECH * rp;     // [16][r]
  float *sw = su + 16 * r;            // [16][r]
  float *red = sw + 16 * r;           // [8]
  __shared__ int tok[32];
  const int j = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 32) {
    int t;
    if (tid < 16)
      t = (j == 0) ? anchor[b] : topk_ids[(b * J + j - 1) * K + tid];
    else
      t = topk_ids[(b * J + j) * K + tid - 16];
    tok[tid] = t;
  }
  // context gate on the final-normed hidden state of mask position j+1
  const T *h = hfinal + (static_cast<size_t>(b) * (J + 1) + j + 1) * H;
  float dot = 0.f;
  for (int c = tid; c < H; c += blockDim.x) dot += Elt<T>::ld(h + c) * w_g[c];
  dot = warp_sum(dot);
  if (lane == 0) red[warp] = dot;
  __syncthreads();
  float gsum = 0.f;
  for (int i = 0; i < 8; ++i) gsum += red[i];
  const float gate = 1.f / (1.f + expf(-(gsum + b_g)));
  float acc[4][2];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = 0.f;
  for (int e0 = 0; e0 < E; e0 += ECH) {
    const int ne = min(ECH, E - e0);
    __syncthreads();   // the previous chunk is consumed
    for (int i = tid; i < 32 * ne; i += blockDim.x) {
      const int row = i / ne, c = i % ne;
      se[row * ECH + c] = Elt<T>::ld(e256 + static_cast<size_t>(tok[row]) * E + e0 + c);
    }
    for (int i = tid; i < 2 * r * ne; i += blockDim.x) {
      const int m = i / (r * ne), rem = i % (r * ne), k = rem / ne, c = rem % ne;
      smt[(m * ECH + c) * rp + k] = Elt<T>::ld((m ? Bm : A) + static_cast<size_t>(k) * E + e0 + c);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {   // rows warp, warp+8, ...: A for the previous tokens, B for the current
      const int row = warp + 8 * q;
      const float *ev = se + row * ECH;
      const float *mt = smt + (row < 16 ? 0 : ECH * rp);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int k = lane + 32 * kk;
        if (k < r) {
          float a = acc[q][kk];
          for (int c = 0; c < ne; ++c) a = fmaf(mt[c * rp + k], ev[c], a);
          acc[q][kk] = a;
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int row = warp + 8 * q;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int k = lane + 32 * kk;
      if (k < r) (row < 16 ? su : sw)[(row & 15) * r + k] = acc[q][kk];
    }
  }
  __syncthreads();
  {
    const int p = tid >> 4, c = tid & 15;
    float bil = 0.f;
    for (int k = 0; k < r; ++k) bil = fmaf(su[p * r + k], sw[c * r + k], bil);
    scores[((static_cast<size_t>(b) * J + j) * K + p) * K + c] = topk_logits[(b * J + j) * K + c] + gate * bil;
  }
}

// one warp per request; lanes 0..15 are the candidates of the current position
__global__ void greedy_kernel(const float *scores, const int32_t *topk_ids, int B, int J, int use_scores,
                              int32_t *draft) {
  pdl_start();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= B) return;
  int prev = 0;
  for (int j = 0; j < J; ++j) {
    const int id = lane < K ? topk_ids[(b * J + j) * K + lane] : 0x7fffffff;
    if (!use_scores) {
      if (lane == 0) draft[b * J + j] = id;
      continue;
    }
    float v = lane < K ? scores[((static_cast<size_t>(b) * J + j) * K + prev) * K + lane] : -INFINITY;
    int bi = lane, bid = id;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      const int id2 = __shfl_xor_sync(0xffffffffu, bid, o);
      if (v2 > v || (v2 == v && id2 < bid)) {
        v = v2;
        bi = i2;
        bid = id2;
      }
    }
    if (lane == 0) draft[b * J + j] = bid;
    prev = bi;
  }
}

__global__ void verify_kernel(const int32_t *draft, const int32_t *target, int B, int J, int32_t *accept, int32_t *bonus,
                              int32_t *committed) {
  pdl_start();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int k = 0;
  const int S = J + 1;
  while (k < J && draft[b * J + k] == target[b * S + k]) ++k;
  accept[b] = k;
  bonus[b] = target[b * S + k];
  for (int i = 0; i < S; ++i) committed[b * S + i] = i <= k ? target[b * S + i] : -1;
}

// ---------------------------------------------------------------------------
// The other selection / verification modes ("DFlash 2", Arquitectura del
// Sistema item 1: sampling over the precomputed scores, or rejection
// sampling that restores the target's exact distribution).  Random numbers
// are inputs.

// Path sampling: one warp per request, lanes 0..15 the candidates; q_j =
// softmax(s_j(prev, .) / T) and the first candidate (in candidate order)
// whose running probability exceeds u_j * total.
__global__ void sample_kernel(const float *scores, const float *topk_logits, const int32_t *topk_ids, int B, int J,
                              float inv_t, const float *uniforms, int32_t *draft, float *qprob) {
  pdl_start();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (b >= B) return;
  int prev = 0;
  for (int j = 0; j < J; ++j) {
    const size_t row = static_cast<size_t>(b) * J + j;
    float s = -INFINITY;
    if (lane < K) s = (scores ? scores[(row * K + prev) * K + lane] : topk_logits[row * K + lane]) * inv_t;
    const float mx = warp_max(s);
    const float e = lane < K ? expf(s - mx) : 0.f;
    const float q = e / warp_sum(e);
    float cum = q;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, cum, o);
      if (lane >= o) cum += t;
    }
    const float total = __shfl_sync(0xffffffffu, cum, K - 1);
    const float u = uniforms[row];
    const unsigned hit = __ballot_sync(0xffffffffu, lane < K && cum > u * total);
    const unsigned pos = __ballot_sync(0xffffffffu, lane < K && q > 0.f);
    const int c = hit ? __ffs(hit) - 1 : 31 - __clz(pos);
    const int id = __shfl_sync(0xffffffffu, lane < K ? topk_ids[row * K + lane] : 0, c);
    if (lane < K) qprob[row * K + lane] = q;
    if (lane == 0) draft[row] = id;
    prev = c;
  }
}

// Target rows are cut into LSE_CH chunks for the log-sum-exp and RES_CH
// chunks for the residual draw, so that a single request still spreads
// over many CTAs.
constexpr int LSE_CH = 8;
constexpr int RES_CH = 32;
constexpr float LOG2E = 1.4426950408889634f;

// Chunk [x0, x1) of a row (x0 a multiple of 4 when the row is 16-byte
// aligned): max, or sum of exp2(x * LOG2E + off), with 16-byte loads, four
// in flight per thread.
template <bool SUM>
__device__ __forceinline__ float chunk_reduce(const float *row, int x0, int x1, bool vec, float off) {
  float acc = SUM ? 0.f : -INFINITY;
  auto f = [&](float x) { acc = SUM ? acc + exp2f(fmaf(x, LOG2E, off)) : fmaxf(acc, x); };
  int x = x0;
  if (vec) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const int i0 = x0 >> 2, i1 = x1 >> 2;
    int i = i0 + threadIdx.x;
    for (; i + 3 * static_cast<int>(blockDim.x) < i1; i += 4 * blockDim.x) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = r4[i + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        f(v[u].x);
        f(v[u].y);
        f(v[u].z);
        f(v[u].w);
      }
    }
    for (; i < i1; i += blockDim.x) {
      const float4 v = r4[i];
      f(v.x);
      f(v.y);
      f(v.z);
      f(v.w);
    }
    x = i1 << 2;
  }
  for (int t = x + static_cast<int>(threadIdx.x); t < x1; t += blockDim.x) f(row[t]);
  return acc;
}

__device__ __forceinline__ int chunk_len(int V, int nch, bool vec) {
  int per = (V + nch - 1) / nch;
  return vec ? (per + 3) & ~3 : per;
}

// (max, sum exp(x - max)) of one chunk of one target row: grid (LSE_CH,
// S positions, B), 256 threads; a max pass, then a branch-free sum pass.
__global__ void __launch_bounds__(256) row_lse_kernel(const float *logits, int V, float2 *part) {
  pdl_start();
  const float *row = logits + (static_cast<size_t>(blockIdx.z) * gridDim.y + blockIdx.y) * V;
  const bool vec = (V & 3) == 0;
  const int per = chunk_len(V, LSE_CH, vec);
  const int x0 = min(V, blockIdx.x * per), x1 = min(V, x0 + per);
  float m = chunk_reduce<false>(row, x0, x1, vec, 0.f);
  __shared__ float sm[8], ss[8];
  __shared__ float bm;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float wm = warp_max(m);
  if (lane == 0) sm[warp] = wm;
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int w = 0; w < 8; ++w) M = fmaxf(M, sm[w]);
    bm = M;
  }
  __syncthreads();
  const float M = bm, off = -M * LOG2E;
  float s = M == -INFINITY ? 0.f : chunk_reduce<true>(row, x0, x1, vec, off);
  s = warp_sum(s);
  __syncthreads();
  if (lane == 0) ss[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float S = 0.f;
    for (int w = 0; w < 8; ++w) S += ss[w];
    part[(static_cast<size_t>(blockIdx.z) * gridDim.y + blockIdx.y) * LSE_CH + blockIdx.x] = make_float2(M, S);
  }
}

__device__ __forceinline__ float row_lse(const float2 *part, int S, int b, int i) {
  const float2 *p = part + (static_cast<size_t>(b) * S + i) * LSE_CH;
  float M = -INFINITY;
#pragma unroll
  for (int c = 0; c < LSE_CH; ++c) M = fmaxf(M, p[c].x);
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < LSE_CH; ++c) sum += p[c].y == 0.f ? 0.f : p[c].y * exp2f((p[c].x - M) * LOG2E);
  return M + logf(sum);
}

// The accept decisions of request b (lanes 0..14 of one warp): k = first rejection.
__device__ __forceinline__ int first_reject(const float *logits, int V, int J, const float2 *part,
                                            const int32_t *draft, const int32_t *topk_ids, const float *qprob,
                                            const float *u_accept, int b, int lane) {
  bool ok = true;
  if (lane < J) {
    const size_t row = static_cast<size_t>(b) * J + lane;
    const int d = draft[row];
    int c = 0;   // the draft token's place among the candidates
    for (int i = 0; i < K; ++i)
      if (topk_ids[row * K + i] == d) {
        c = i;
        break;
      }
    const float p = expf(logits[(static_cast<size_t>(b) * (J + 1) + lane) * V + d] - row_lse(part, J + 1, b, lane));
    ok = u_accept[row] * qprob[row * K + c] < p;
  }
  const unsigned fail = __ballot_sync(0xffffffffu, lane < J && !ok);
  return fail ? __ffs(fail) - 1 : J;
}

// r(x) of the decisive row: max(0, p(x) - q(x)) after a rejection, p(x) after 15 acceptances.
struct Resid {
  const float *z;
  float lse;
  bool resid;
  int cid[K];
  float cq[K];
  __device__ float w(int x) const {
    float v = expf(z[x] - lse);
    if (resid)
#pragma unroll
      for (int c = 0; c < K; ++c)
        if (cid[c] == x) v = fmaxf(v - cq[c], 0.f);
    return v;
  }
};

__device__ __forceinline__ void make_resid(Resid &r, const float *logits, int V, int J, const float2 *part,
                                           const int32_t *topk_ids, const float *qprob, int b, int k) {
  r.z = logits + (static_cast<size_t>(b) * (J + 1) + k) * V;
  r.lse = row_lse(part, J + 1, b, k);
  r.resid = k < J;
#pragma unroll
  for (int c = 0; c < K; ++c) {
    r.cid[c] = r.resid ? topk_ids[(static_cast<size_t>(b) * J + k) * K + c] : -1;
    r.cq[c] = r.resid ? qprob[(static_cast<size_t>(b) * J + k) * K + c] : 0.f;
  }
}

// Sums of r over RES_CH chunks of the decisive row: grid (RES_CH, B), 256 threads.
__global__ void __launch_bounds__(256) resid_sum_kernel(const float *logits, int V, int J, const float2 *part,
                                                        const int32_t *draft, const int32_t *topk_ids,
                                                        const float *qprob, const float *u_accept, float *csum) {
  pdl_start();
  const int b = blockIdx.y;
  __shared__ int k_sh;
  if (threadIdx.x < 32) {
    const int k = first_reject(logits, V, J, part, draft, topk_ids, qprob, u_accept, b, threadIdx.x);
    if (threadIdx.x == 0) k_sh = k;
  }
  __syncthreads();
  Resid r;
  make_resid(r, logits, V, J, part, topk_ids, qprob, b, k_sh);
  const bool vec = (V & 3) == 0;
  const int per = chunk_len(V, RES_CH, vec);
  const int x0 = min(V, blockIdx.x * per), x1 = min(V, x0 + per);
  float s = chunk_reduce<true>(r.z, x0, x1, vec, -r.lse * LOG2E);
  // candidates inside the chunk: r = p - min(p, q)
  if (threadIdx.x == 0 && r.resid)
    for (int c = 0; c < K; ++c)
      if (r.cid[c] >= x0 && r.cid[c] < x1) s -= fminf(expf(r.z[r.cid[c]] - r.lse), r.cq[c]);
  s = warp_sum(s);
  __shared__ float ws[8];
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += ws[w];
    csum[b * RES_CH + blockIdx.x] = fmaxf(t, 0.f);
  }
}

// One CTA (256 threads) per request: the accept decisions, the chunk holding
// u * Z (chunk sums in vocabulary order), then that chunk's inverse CDF:
// per-thread contiguous ranges, a block scan, the owner walks its range.
__global__ void __launch_bounds__(256) reject_kernel(const float *logits, int V, int J, const float2 *part,
                                                     const float *csum, const int32_t *draft,
                                                     const int32_t *topk_ids, const float *qprob,
                                                     const float *u_accept, const float *u_bonus, int32_t *accept,
                                                     int32_t *bonus, int32_t *committed) {
  pdl_start();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ int k_sh, chunk_sh, pick_sh;
  __shared__ float base_sh, total_sh;
  __shared__ float wsum[8];
  if (warp == 0) {
    const int k = first_reject(logits, V, J, part, draft, topk_ids, qprob, u_accept, b, lane);
    // chunk sums: running total in chunk order (lanes = chunks)
    const float c = lane < RES_CH ? csum[b * RES_CH + lane] : 0.f;
    float inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    const float Z = __shfl_sync(0xffffffffu, inc, 31);
    const float thr = u_bonus[b] * Z;
    const unsigned hit = __ballot_sync(0xffffffffu, lane < RES_CH && c > 0.f && thr < inc);
    const unsigned pos = __ballot_sync(0xffffffffu, lane < RES_CH && c > 0.f);
    const int ch = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lane == 0) {
      k_sh = k;
      chunk_sh = ch;
      total_sh = Z;
      pick_sh = -1;
    }
    if (ch >= 0 && lane == ch) base_sh = inc - c;
  }
  __syncthreads();
  const int k = k_sh, ch = chunk_sh;
  Resid r;
  make_resid(r, logits, V, J, part, topk_ids, qprob, b, k);
  if (ch >= 0) {
    const int per_c = chunk_len(V, RES_CH, (V & 3) == 0);
    const int c0 = min(V, ch * per_c), c1 = min(V, c0 + per_c);
    const int per = (c1 - c0 + blockDim.x - 1) / blockDim.x;
    const int x0 = min(c1, c0 + tid * per), x1 = min(c1, x0 + per);
    float mine = 0.f;
    for (int x = x0; x < x1; ++x) mine += r.w(x);
    float inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    float ex = base_sh + inc - mine;
    for (int w = 0; w < warp; ++w) ex += wsum[w];
    const float thr = u_bonus[b] * total_sh;
    if (mine > 0.f && thr >= ex && thr < ex + mine) {   // this thread's range holds the draw
      float c = ex;
      int pick = x1 - 1;
      for (int x = x0; x < x1; ++x) {
        c += r.w(x);
        if (c > thr) {
          pick = x;
          break;
        }
      }
      atomicMax(&pick_sh, pick);
    }
  }
  __syncthreads();
  if (tid == 0 && pick_sh < 0) {
    // rounding put the draw past every range: the last token of positive weight
    int last = V - 1;
    for (int x = V - 1; x >= 0; --x)
      if (r.w(x) > 0.f) {
        last = x;
        break;
      }
    pick_sh = last;
  }
  __syncthreads();
  if (tid == 0) {
    accept[b] = k;
    bonus[b] = pick_sh;
  }
  if (tid <= J) {
    int v = -1;
    if (tid < k) v = draft[static_cast<size_t>(b) * J + tid];
    else if (tid == k) v = pick_sh;
    committed[b * (J + 1) + tid] = v;
  }
}

// Bounded spin on a device flag (self test of the timeout path).
__global__ void wait_flag_kernel(const int32_t *flag, int *status, unsigned long long timeout_ns) {
  const volatile int32_t *f = flag;
  const uint64_t t0 = globaltimer_ns();
  while (*f == 0) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      report(status, DFLASH_ERR_TIMEOUT);
      return;
    }
  }
}

}  // namespace

int pair_scores(const Launch &lc, bool f32, const int32_t *anchor, const int32_t *topk_ids, const float *topk_logits,
                const void *final_hidden, int B, int J, int H, const void *e256, const void *sel_a, const void *sel_b,
                int r, int E, const float *w_g, float b_g, float *scores) {
  if (B <= 0) return DFLASH_OK;
  if (r < 1 || r > 64 || E < 1 || E > 1024)
    return set_error(DFLASH_ERR_UNSUPPORTED, "selector rank must be 1..64 and embedding width 1..1024");
  const size_t smem = (32 * static_cast<size_t>(ECH) + 2 * static_cast<size_t>(ECH) * (r + 1) + 32 * r + 8) * sizeof(float);
  dim3 grid(J, B);
  ProfScope ps(lc, "pair_scores", -1.0, -1.0);
  if (f32) {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(pair_scores_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    launch_pdl(pair_scores_kernel<float>, dim3(grid), dim3(256), smem, lc.stream,
        anchor, topk_ids, topk_logits, static_cast<const float *>(final_hidden), H, static_cast<const float *>(e256),
        static_cast<const float *>(sel_a), static_cast<const float *>(sel_b), r, E, w_g, b_g, J, scores);
  } else {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(pair_scores_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
    launch_pdl(pair_scores_kernel<__nv_bfloat16>, dim3(grid), dim3(256), smem, lc.stream,
        anchor, topk_ids, topk_logits, static_cast<const __nv_bfloat16 *>(final_hidden), H,
        static_cast<const __nv_bfloat16 *>(e256), static_cast<const __nv_bfloat16 *>(sel_a),
        static_cast<const __nv_bfloat16 *>(sel_b), r, E, w_g, b_g, J, scores);
  }
  return cuda_check(cudaGetLastError(), "pair_scores launch");
}

int sample_path(const Launch &lc, const float *scores, const float *topk_logits, const int32_t *topk_ids, int B,
                int J, float temperature, const float *uniforms, int32_t *draft, float *qprob) {
  if (B <= 0) return DFLASH_OK;
  ProfScope ps(lc, "sample_path", -1.0, -1.0);
  launch_pdl(sample_kernel, dim3((B + 3) / 4), dim3(128), 0, lc.stream, scores, topk_logits, topk_ids, B,
             J, 1.f / temperature, uniforms, draft, qprob);
  return cuda_check(cudaGetLastError(), "sample_path launch");
}

int verify_rejection(const Launch &lc, const float *target_logits, int V, float *scratch, const int32_t *draft,
                     const int32_t *topk_ids, const float *qprob, const float *u_accept, const float *u_bonus, int B,
                     int J, int32_t *accept, int32_t *bonus, int32_t *committed) {
  if (B <= 0) return DFLASH_OK;
  const int S = J + 1;
  float2 *part = reinterpret_cast<float2 *>(scratch);                  // [B][S][LSE_CH]
  float *csum = scratch + static_cast<size_t>(B) * S * LSE_CH * 2;     // [B][RES_CH]
  {
    ProfScope ps(lc, "target_lse", 4.0 * B * S * V, -1.0);
    launch_pdl(row_lse_kernel, dim3(LSE_CH, S, B), dim3(256), 0, lc.stream, target_logits, V, part);
    if (int e = cuda_check(cudaGetLastError(), "target lse launch")) return e;
  }
  ProfScope ps(lc, "verify_rejection", 4.0 * B * V, -1.0);
  launch_pdl(resid_sum_kernel, dim3(RES_CH, B), dim3(256), 0, lc.stream, target_logits, V, J,
             static_cast<const float2 *>(part), draft, topk_ids, qprob, u_accept, csum);
  if (int e = cuda_check(cudaGetLastError(), "residual sums launch")) return e;
  launch_pdl(reject_kernel, dim3(B), dim3(256), 0, lc.stream, target_logits, V, J, static_cast<const float2 *>(part),
             static_cast<const float *>(csum), draft, topk_ids, qprob, u_accept, u_bonus, accept, bonus, committed);
  return cuda_check(cudaGetLastError(), "verify_rejection launch");
}

int verify_rejection_scratch_floats(int B, int S) { return B * (S * LSE_CH * 2 + RES_CH); }

int greedy_path(const Launch &lc, const float *scores, const int32_t *topk_ids, int B, int J, bool use_scores,
                int32_t *draft) {
  if (B <= 0) return DFLASH_OK;
  ProfScope ps(lc, "greedy_path", -1.0, -1.0);
  launch_pdl(greedy_kernel, dim3((B + 3) / 4), dim3(128), 0, lc.stream, scores, topk_ids, B, J, use_scores ? 1 : 0,
             draft);
  return cuda_check(cudaGetLastError(), "greedy launch");
}

int verify(const Launch &lc, const int32_t *draft, const int32_t *target, int B, int J, int32_t *accept,
           int32_t *bonus, int32_t *committed) {
  if (B <= 0) return DFLASH_OK;
  ProfScope ps(lc, "verify", -1.0, -1.0);
  launch_pdl(verify_kernel, dim3((B + 127) / 128), dim3(128), 0, lc.stream, draft, target, B, J, accept, bonus,
             committed);
  return cuda_check(cudaGetLastError(), "verify launch");
}

int wait_flag(const Launch &lc, const int32_t *flag) {
  wait_flag_kernel<<<1, 1, 0, lc.stream>>>(flag, lc.status, lc.timeout_ns);   // ordinary launch: sees every earlier write
  return cuda_check(cudaGetLastError(), "wait_flag launch");
}

}  // namespace dflash

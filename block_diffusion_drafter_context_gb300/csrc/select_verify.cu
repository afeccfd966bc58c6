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

constexpr int K = 16;
constexpr int J = 15;

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
                                                          const float *w_g, float b_g, float *scores) {
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
  const T *h = hfinal + (static_cast<size_t>(b) * 16 + j + 1) * H;
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
__global__ void greedy_kernel(const float *scores, const int32_t *topk_ids, int B, int use_scores, int32_t *draft) {
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

__global__ void verify_kernel(const int32_t *draft, const int32_t *target, int B, int32_t *accept, int32_t *bonus,
                              int32_t *committed) {
  pdl_start();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int k = 0;
  while (k < J && draft[b * J + k] == target[b * 16 + k]) ++k;
  accept[b] = k;
  bonus[b] = target[b * 16 + k];
  for (int i = 0; i < 16; ++i) committed[b * 16 + i] = i <= k ? target[b * 16 + i] : -1;
}

// ---------------------------------------------------------------------------
// The other selection / verification modes ("DFlash 2", Arquitectura del
// Sistema item 1: sampling over the precomputed scores, or rejection
// sampling that restores the target's exact distribution).  Random numbers
// are inputs.

// Path sampling: one warp per request, lanes 0..15 the candidates; q_j =
// softmax(s_j(prev, .) / T) and the first candidate (in candidate order)
// whose running probability exceeds u_j * total.
__global__ void sample_kernel(const float *scores, const float *topk_logits, const int32_t *topk_ids, int B,
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

// log-sum-exp of one row of target logits: grid (16 positions, B), 256 threads.
__global__ void __launch_bounds__(256) row_lse_kernel(const float *logits, int V, float *lse) {
  pdl_start();
  const float *row = logits + (static_cast<size_t>(blockIdx.y) * 16 + blockIdx.x) * V;
  float m = -INFINITY, s = 0.f;
  auto add = [&](float x) {
    if (x > m) {
      s = s * expf(m - x) + 1.f;
      m = x;
    } else {
      s += expf(x - m);
    }
  };
  if ((V & 3) == 0) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    for (int i = threadIdx.x; i < V / 4; i += blockDim.x) {
      const float4 v = r4[i];
      add(v.x);
      add(v.y);
      add(v.z);
      add(v.w);
    }
  } else {
    for (int i = threadIdx.x; i < V; i += blockDim.x) add(row[i]);
  }
  __shared__ float sm[8], ss[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float wm = warp_max(m);
  s = warp_sum(m == -INFINITY ? 0.f : s * expf(m - wm));
  if (lane == 0) {
    sm[warp] = wm;
    ss[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY, S = 0.f;
    for (int w = 0; w < 8; ++w) M = fmaxf(M, sm[w]);
    for (int w = 0; w < 8; ++w) S += ss[w] == 0.f ? 0.f : ss[w] * expf(sm[w] - M);
    lse[blockIdx.y * 16 + blockIdx.x] = M + logf(S);
  }
}

// Rejection-sampling verification, one CTA (256 threads) per request: accept
// while u_i * q_i(d_i) < p_i(d_i); then the bonus by inverse CDF in
// vocabulary order from max(0, p_k - q_k) (p_15 after 15 acceptances).  Each
// thread owns a contiguous vocabulary range; a block scan of the range sums
// finds the range holding u * Z, whose owner walks it.
__global__ void __launch_bounds__(256) reject_kernel(const float *logits, int V, const float *lse,
                                                     const int32_t *draft, const int32_t *topk_ids,
                                                     const float *qprob, const float *u_accept,
                                                     const float *u_bonus, int32_t *accept, int32_t *bonus,
                                                     int32_t *committed) {
  pdl_start();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ int k_sh, pick_sh;
  __shared__ int cid[K];
  __shared__ float cq[K];
  __shared__ float wsum[8];
  if (warp == 0) {   // accept loop: lanes 0..14 test their position, the first failure wins
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
      const float p = expf(logits[(static_cast<size_t>(b) * 16 + lane) * V + d] - lse[b * 16 + lane]);
      ok = u_accept[row] * qprob[row * K + c] < p;
    }
    const unsigned fail = __ballot_sync(0xffffffffu, lane < J && !ok);
    if (lane == 0) k_sh = fail ? __ffs(fail) - 1 : J;
  }
  __syncthreads();
  const int k = k_sh;
  const bool resid = k < J;
  if (tid < K) {
    cid[tid] = resid ? topk_ids[(static_cast<size_t>(b) * J + k) * K + tid] : -1;
    cq[tid] = resid ? qprob[(static_cast<size_t>(b) * J + k) * K + tid] : 0.f;
  }
  __syncthreads();
  const float *zr = logits + (static_cast<size_t>(b) * 16 + k) * V;
  const float l = lse[b * 16 + k];
  const int per = (V + blockDim.x - 1) / blockDim.x;
  const int x0 = min(V, tid * per), x1 = min(V, x0 + per);
  auto weight = [&](int x, bool use_resid) -> float {   // r(x) = max(0, p(x) - q(x)), or p(x)
    float w = expf(zr[x] - l);
    if (use_resid)
#pragma unroll
      for (int c = 0; c < K; ++c)
        if (cid[c] == x) w = fmaxf(w - cq[c], 0.f);
    return w;
  };
  // range sums: p over the range minus min(p, q) for candidates inside it
  float mine = 0.f;
  for (int x = x0; x < x1; ++x) mine += expf(zr[x] - l);
  if (resid)
#pragma unroll
    for (int c = 0; c < K; ++c)
      if (cid[c] >= x0 && cid[c] < x1) mine -= fminf(expf(zr[cid[c]] - l), cq[c]);
  mine = fmaxf(mine, 0.f);
  // block exclusive scan of the range sums (thread order = vocabulary order)
  float inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  float base = 0.f, Z = 0.f;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) base += wsum[w];
    Z += wsum[w];
  }
  const float ex = base + inc - mine;
  // a residual that rounds to nothing (p = q on the candidates: no rejection
  // in exact arithmetic) takes the fallback below
  if (threadIdx.x == 0) pick_sh = -1;
  __syncthreads();
  if (!resid || Z > 0.f) {
    const float thr = u_bonus[b] * Z;
    if (thr >= ex && thr < ex + mine) {   // this thread's range holds the draw
      float c = ex;
      int pick = -1;
      for (int x = x0; x < x1; ++x) {
        const float w = weight(x, resid);
        c += w;
        if (c > thr) {
          pick = x;
          break;
        }
      }
      if (pick < 0) pick = x1 - 1;
      atomicMax(&pick_sh, pick);
    }
  }
  __syncthreads();
  if (pick_sh < 0 && tid == 0) {
    // rounding left no range holding the draw (or the residual vanished):
    // the last token of positive weight under p
    int last = V - 1;
    for (int x = V - 1; x >= 0; --x)
      if (expf(zr[x] - l) > 0.f) {
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
  if (tid < 16) {
    int v = -1;
    if (tid < k) v = draft[static_cast<size_t>(b) * J + tid];
    else if (tid == k) v = pick_sh;
    committed[b * 16 + tid] = v;
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
                const void *final_hidden, int B, int H, const void *e256, const void *sel_a, const void *sel_b, int r,
                int E, const float *w_g, float b_g, float *scores) {
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
        static_cast<const float *>(sel_a), static_cast<const float *>(sel_b), r, E, w_g, b_g, scores);
  } else {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(pair_scores_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
    launch_pdl(pair_scores_kernel<__nv_bfloat16>, dim3(grid), dim3(256), smem, lc.stream,
        anchor, topk_ids, topk_logits, static_cast<const __nv_bfloat16 *>(final_hidden), H,
        static_cast<const __nv_bfloat16 *>(e256), static_cast<const __nv_bfloat16 *>(sel_a),
        static_cast<const __nv_bfloat16 *>(sel_b), r, E, w_g, b_g, scores);
  }
  return cuda_check(cudaGetLastError(), "pair_scores launch");
}

int sample_path(const Launch &lc, const float *scores, const float *topk_logits, const int32_t *topk_ids, int B,
                float temperature, const float *uniforms, int32_t *draft, float *qprob) {
  if (B <= 0) return DFLASH_OK;
  ProfScope ps(lc, "sample_path", -1.0, -1.0);
  launch_pdl(sample_kernel, dim3((B + 3) / 4), dim3(128), 0, lc.stream, scores, topk_logits, topk_ids, B,
             1.f / temperature, uniforms, draft, qprob);
  return cuda_check(cudaGetLastError(), "sample_path launch");
}

int verify_rejection(const Launch &lc, const float *target_logits, int V, float *lse, const int32_t *draft,
                     const int32_t *topk_ids, const float *qprob, const float *u_accept,
                     const float *u_bonus, int B, int32_t *accept, int32_t *bonus, int32_t *committed) {
  if (B <= 0) return DFLASH_OK;
  {
    ProfScope ps(lc, "target_lse", 4.0 * B * 16 * V, -1.0);
    launch_pdl(row_lse_kernel, dim3(16, B), dim3(256), 0, lc.stream, target_logits, V, lse);
    if (int e = cuda_check(cudaGetLastError(), "target lse launch")) return e;
  }
  ProfScope ps(lc, "verify_rejection", -1.0, -1.0);
  launch_pdl(reject_kernel, dim3(B), dim3(256), 0, lc.stream, target_logits, V, static_cast<const float *>(lse),
             draft, topk_ids, qprob, u_accept, u_bonus, accept, bonus, committed);
  return cuda_check(cudaGetLastError(), "verify_rejection launch");
}

int greedy_path(const Launch &lc, const float *scores, const int32_t *topk_ids, int B, bool use_scores,
                int32_t *draft) {
  if (B <= 0) return DFLASH_OK;
  ProfScope ps(lc, "greedy_path", -1.0, -1.0);
  launch_pdl(greedy_kernel, dim3((B + 3) / 4), dim3(128), 0, lc.stream, scores, topk_ids, B, use_scores ? 1 : 0, draft);
  return cuda_check(cudaGetLastError(), "greedy launch");
}

int verify(const Launch &lc, const int32_t *draft, const int32_t *target, int B, int32_t *accept, int32_t *bonus,
           int32_t *committed) {
  if (B <= 0) return DFLASH_OK;
  ProfScope ps(lc, "verify", -1.0, -1.0);
  launch_pdl(verify_kernel, dim3((B + 127) / 128), dim3(128), 0, lc.stream, draft, target, B, accept, bonus, committed);
  return cuda_check(cudaGetLastError(), "verify launch");
}

int wait_flag(const Launch &lc, const int32_t *flag) {
  wait_flag_kernel<<<1, 1, 0, lc.stream>>>(flag, lc.status, lc.timeout_ns);   // ordinary launch: sees every earlier write
  return cuda_check(cudaGetLastError(), "wait_flag launch");
}

}  // namespace dflash

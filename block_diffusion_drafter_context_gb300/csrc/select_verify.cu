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

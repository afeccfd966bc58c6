// fp32 GEMM on CUDA cores for the fp32 drafter configuration (tiny shapes,
// where tf32 tensor-core rounding would exceed the fp32 tolerance).
//   out[m][n] = epi( sum_k X[m][k] * W[n][k] )
#include "common.cuh"
#include "internal.h"

namespace dflash {
namespace {

constexpr int TN = 32, TM = 16, TK = 32;

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float *__restrict__ W, int ldw,
                                                       const float *__restrict__ X, int ldx, int M, int N,
                                                       int K, int epi, void *out, int ldo,
                                                       const float *__restrict__ bias) {
  pdl_start();
  __shared__ float Ws[TN][TK + 1];
  __shared__ float Xs[TM][TK + 1];
  const int tx = threadIdx.x;   // 0..31: n within tile (one warp row)
  const int ty = threadIdx.y;   // 0..7: two tokens each
  const int n = blockIdx.x * TN + tx;
  const int m0 = blockIdx.y * TM + ty * 2;
  float acc0 = 0.f, acc1 = 0.f;
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = ty; i < TN; i += 8) {
      const int nn = blockIdx.x * TN + i, kk = k0 + tx;
      Ws[i][tx] = (nn < N && kk < K) ? W[static_cast<size_t>(nn) * ldw + kk] : 0.f;
    }
    for (int i = ty; i < TM; i += 8) {
      const int mm = blockIdx.y * TM + i, kk = k0 + tx;
      Xs[i][tx] = (mm < M && kk < K) ? X[static_cast<size_t>(mm) * ldx + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < TK; ++k) {
      const float w = Ws[tx][k];
      acc0 = fmaf(Xs[ty * 2][k], w, acc0);
      acc1 = fmaf(Xs[ty * 2 + 1][k], w, acc1);
    }
    __syncthreads();
  }
  const float acc[2] = {acc0, acc1};
  const bool nok = n < N;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int m = m0 + i;
    const float v = acc[i];
    if (epi == EPI_SWIGLU) {
      const float up = __shfl_xor_sync(0xffffffffu, v, 1);
      if (nok && !(n & 1) && m < M) static_cast<float *>(out)[static_cast<size_t>(m) * ldo + (n >> 1)] = v / (1.f + expf(-v)) * up;
      continue;
    }
    if (!nok || m >= M) continue;
    float *o = static_cast<float *>(out) + static_cast<size_t>(m) * ldo + n;
    if (epi == EPI_ADD_F32)
      *o += v;
    else if (epi == EPI_TANH_BIAS)
      *o = tanhf(v + bias[n]);
    else
      *o = v;
  }
}

}  // namespace

int gemm_f32(const Launch &lc, const GemmOp &op) {
  const int M = op.M, N = op.N, K = op.K;
  if (M <= 0 || N <= 0 || K <= 0) return DFLASH_OK;
  int epi = op.epi;
  if (epi == EPI_STORE_T || epi == EPI_F32_SPLIT) epi = EPI_F32;
  if (epi == EPI_BF16) return set_error(DFLASH_ERR_UNSUPPORTED, "gemm %s: bf16 output on the fp32 path", op.name);
  dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM), block(32, 8);
  ProfScope ps(lc, op.name, 4.0 * N * K + 4.0 * M * K + 4.0 * M * N, 2.0 * M * N * K);
  launch_pdl(gemm_f32_kernel, dim3(grid), dim3(block), 0, lc.stream, static_cast<const float *>(op.W), op.ldw,
                                                  static_cast<const float *>(op.X), op.ldx, M, N, K, epi, op.out,
                                                  op.ldo, op.bias);
  return cuda_check(cudaGetLastError(), "gemm_f32 launch");
}

}  // namespace dflash

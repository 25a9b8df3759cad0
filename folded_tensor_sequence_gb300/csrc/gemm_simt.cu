// fp32 GEMM on the CUDA cores (exact fp32 FFMA; tf32 tensor cores would
// miss a 1e-4 relative bound).  Same contract as the tensor-core GEMM:
// C[M][N] = sum_k A[m][k] * B[n][k], with the STORE, RESID and QKV epilogues.
// 64 x 64 tiles, 16-deep K slices through shared memory, 4 x 4 outputs per
// thread.  Used for fp32 layer plans, which are small.
#include "common.cuh"
#include "internal.h"

namespace tsp {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, int64_t lda,
                                                        const float* __restrict__ B, int64_t ldb, int M, int N,
                                                        int K, int epi, EpiParams ep) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = (int64_t)blockIdx.y * TM, n0 = (int64_t)blockIdx.x * TN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      const int r = i / TK, c = i % TK;
      const int64_t m = m0 + r;
      const int k = k0 + c;
      As[c][r] = (m < M && k < K) ? A[m * lda + k] : 0.0f;
      const int64_t n = n0 + r;
      Bs[c][r] = (n < N && k < K) ? B[n * ldb + k] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc[i][j];
      if (epi == EPI_STORE) {
        if (ep.split_col > 0 && n >= ep.split_col)
          static_cast<float*>(ep.aux)[m * ep.ldx + (n - ep.split_col)] = v;
        else
          static_cast<float*>(ep.out)[m * ep.ldo + n] = v;
      } else if (epi == EPI_RESID) {
        v += static_cast<const float*>(ep.resid)[m * ep.ldr + n];
        static_cast<float*>(ep.out)[m * ep.ldo + n] = v;
      } else {  // EPI_QKV: a shard's packed columns are Q (h/D) | K (Hk*dh/D) | V (Hk*dh/D)
        const int hs = ep.h / ep.D, ks = ep.Hk * ep.dh / ep.D;
        const int s = (int)(n / (hs + 2 * ks));
        const int within = (int)(n - (int64_t)s * (hs + 2 * ks));
        const int which = within < hs ? 0 : (within < hs + ks ? 1 : 2);
        const int cin = within - (which == 0 ? 0 : hs + (which - 1) * ks);
        const int head = s * ((which == 0 ? ep.H : ep.Hk) / ep.D) + cin / ep.dh, d = cin % ep.dh;
        if (which == 0) {
          static_cast<float*>(ep.q)[m * ep.h + head * ep.dh + d] = v;
        } else {
          const int64_t twoC = 2 * (int64_t)ep.C, per_rank = (int64_t)ep.B * twoC;
          const int64_t r = m / per_rank, rem = m % per_rank, b = rem / twoC, k = rem % twoC;
          const int64_t p = k < ep.C ? r * ep.C + k : (2 * ep.D - 1 - r) * ep.C + (k - ep.C);
          float* dst = static_cast<float*>(which == 1 ? ep.k : ep.v);
          dst[((b * ep.Hk + head) * ep.S + p) * ep.dh + d] = v;
        }
      }
    }
  }
}

}  // namespace

tsp_status gemm_f32_simt(const float* A, int64_t lda, const float* B, int64_t ldb, int M, int N, int K,
                         EpiKind epi, const EpiParams& ep, cudaStream_t stream) {
  if (M <= 0 || N <= 0) return TSP_OK;
  if (epi != EPI_STORE && epi != EPI_RESID && epi != EPI_QKV) return TSP_ERR_UNSUPPORTED;
  dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM);
  if (grid.y > 65535) return TSP_ERR_UNSUPPORTED;
  gemm_f32_kernel<<<grid, 256, 0, stream>>>(A, lda, B, ldb, M, N, K, (int)epi, ep);
  return cudaGetLastError() == cudaSuccess ? TSP_OK : TSP_ERR_CUDA;
}

}  // namespace tsp

// gemm_simt.cu -- fp32 CUDA-core GEMM for the fp32 variant of the step
// (small shapes; the bf16 path runs on the tcgen05 kernel in gemm_tc.cu).
//
// C[M,N] = A[M,K] * op(B) (+ C), A row-major, B either [N,K] (C = A B^T, the
// pages' x @ W.T) or [K,N] (C = A B), fp32 accumulation.
#include "common.cuh"
#include "kernels.h"

namespace canvas {

namespace {
constexpr int TM = 64, TN = 64, TK = 16;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ A, const T* __restrict__ B,
                                                         int b_mn_major, float* __restrict__ C, int M, int N,
                                                         int K, int accumulate) {
  __shared__ float sA[TK][TM + 4];
  __shared__ float sB[TK][TN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int e = threadIdx.x; e < TM * TK; e += 256) {
      const int mm = e / TK, kk = e % TK;
      const int gm = m0 + mm, gk = k0 + kk;
      sA[kk][mm] = (gm < M && gk < K) ? to_f32(A[(long long)gm * K + gk]) : 0.f;
    }
    for (int e = threadIdx.x; e < TN * TK; e += 256) {
      int nn, kk;
      if (b_mn_major) {
        kk = e / TN;
        nn = e % TN;
      } else {
        nn = e / TK;
        kk = e % TK;
      }
      const int gn = n0 + nn, gk = k0 + kk;
      float v = 0.f;
      if (gn < N && gk < K) v = to_f32(b_mn_major ? B[(long long)gk * N + gn] : B[(long long)gn * K + gk]);
      sB[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sA[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = sB[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float* c = C + (long long)gm * N + gn;
      *c = accumulate ? *c + acc[i][j] : acc[i][j];
    }
  }
}
}  // namespace

cudaError_t launch_gemm_simt(const void* A, const void* B, int b_mn_major, bool bf16, float* C, int M, int N,
                             int K, int accumulate, cudaStream_t stream) {
  dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM);
  if (bf16)
    gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(A),
                                                               static_cast<const __nv_bfloat16*>(B), b_mn_major,
                                                               C, M, N, K, accumulate);
  else
    gemm_simt_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(A), static_cast<const float*>(B),
                                                       b_mn_major, C, M, N, K, accumulate);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace canvas

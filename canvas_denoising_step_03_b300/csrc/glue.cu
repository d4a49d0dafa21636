// glue.cu -- the two element-wise kernels a caller needs to chain canvas
// steps into a multi-layer denoising loop: the canvas input (embedding of the
// current tokens plus the self-conditioning soft embedding of the previous
// step) and a round-to-bf16 cast of fp32 activations; and a diagnostic kernel
// that exercises the bounded-wait timeout path of every pipelined kernel.
//
// Self-conditioning: the expected embedding P.E of the previous step's
// softmax is added to the canvas input (AI Trends summary of a DiffusionGemma
// 26B notebook, aitrends.kr/articles/94089, glossary entry "자기 조건화"; the
// small MLP applied to it there needs trained weights and is left to the
// caller).
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace canvas {

namespace {

// v = E[tokens[r], :] + soft[r, :] (fp32); x = bf16(v), x32 = v (if non-null);
// 8 columns per thread
__global__ void __launch_bounds__(256) embed_input_kernel(const int32_t* __restrict__ tokens,
                                                          const __nv_bfloat16* __restrict__ E,
                                                          const float* __restrict__ soft, int rows, int D, int V,
                                                          __nv_bfloat16* __restrict__ x, float* __restrict__ x32) {
  const int per_row = D / 8;
  const long long total = (long long)rows * per_row;
  for (long long e = blockIdx.x * 256LL + threadIdx.x; e < total; e += (long long)gridDim.x * 256) {
    const int r = int(e / per_row), c = int(e % per_row) * 8;
    const int tok = tokens[r];
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (tok < 0 || tok >= V) {
      record_error(CANVAS_ERR_BOUNDS);
    } else {
      const uint4 u = *reinterpret_cast<const uint4*>(E + (long long)tok * D + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      }
      if (soft != nullptr) {
        const float4 s0 = *reinterpret_cast<const float4*>(soft + (long long)r * D + c);
        const float4 s1 = *reinterpret_cast<const float4*>(soft + (long long)r * D + c + 4);
        v[0] += s0.x; v[1] += s0.y; v[2] += s0.z; v[3] += s0.w;
        v[4] += s1.x; v[5] += s1.y; v[6] += s1.z; v[7] += s1.w;
      }
    }
    *reinterpret_cast<uint4*>(x + (long long)r * D + c) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
    if (x32 != nullptr) {
      float4* o = reinterpret_cast<float4*>(x32 + (long long)r * D + c);
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

// out[i] = bf16(in[i]), 8 per thread (n % 8 == 0)
__global__ void __launch_bounds__(256) cast_bf16_kernel(const float4* __restrict__ in, uint4* __restrict__ out,
                                                        long long n8) {
  for (long long e = blockIdx.x * 256LL + threadIdx.x; e < n8; e += (long long)gridDim.x * 256) {
    const float4 a = in[2 * e], b = in[2 * e + 1];
    out[e] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

// out = bf16(gelu(in)), GELU in its tanh form 0.5 x (1 + tanh(u)), u =
// sqrt(2/pi) (x + 0.044715 x^3), rounded once: the activation of the
// self-conditioning MLP.  Evaluated as x / (1 + exp(-2u)) (the identity
// 1 + tanh(u) = 2 / (1 + exp(-2u))), which keeps its relative accuracy for
// negative x, where 1 + tanh(u) would cancel.
__global__ void __launch_bounds__(256) gelu_bf16_kernel(const float4* __restrict__ in, uint4* __restrict__ out,
                                                        long long n8) {
  const float k0 = 0.7978845608028654f, k1 = 0.044715f;
  for (long long e = blockIdx.x * 256LL + threadIdx.x; e < n8; e += (long long)gridDim.x * 256) {
    const float4 a = in[2 * e], b = in[2 * e + 1];
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = v[j];
      v[j] = x / (1.0f + expf(-2.0f * k0 * (x + k1 * x * x * x)));
    }
    out[e] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                        pack_bf16x2(v[6], v[7]));
  }
}

// Committed positions per canvas (adaptive stopping): one block per canvas,
// a plain count of the commit mask's ones (integers: exact).
__global__ void __launch_bounds__(256) count_committed_kernel(const uint8_t* __restrict__ mask, int canvas_len,
                                                              int32_t* __restrict__ counts) {
  __shared__ int total;
  if (threadIdx.x == 0) total = 0;
  __syncthreads();
  const uint8_t* m = mask + (size_t)blockIdx.x * canvas_len;
  int c = 0;
  for (int i = threadIdx.x; i < canvas_len; i += blockDim.x) c += m[i] != 0 ? 1 : 0;
  atomicAdd(&total, c);
  __syncthreads();
  if (threadIdx.x == 0) counts[blockIdx.x] = total;
}

// One thread waits, through the same bounded wait as every pipelined kernel,
// on an mbarrier phase that nothing completes: after the wait limit it
// records CANVAS_ERR_TIMEOUT in the status word and the kernel returns.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag);
}

}  // namespace

cudaError_t launch_embed_input(const int32_t* tokens, const void* E, const float* soft, int rows, int D, int V,
                               void* x, float* x32, cudaStream_t stream) {
  const long long total = (long long)rows * (D / 8);
  const int blocks = int(std::min<long long>((total + 255) / 256, 148LL * 16));
  embed_input_kernel<<<blocks, 256, 0, stream>>>(tokens, static_cast<const __nv_bfloat16*>(E), soft, rows, D, V,
                                                 static_cast<__nv_bfloat16*>(x), x32);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_cast_bf16(const float* in, void* out, long long n, cudaStream_t stream) {
  const long long n8 = n / 8;
  const int blocks = int(std::min<long long>((n8 + 255) / 256, 148LL * 16));
  cast_bf16_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(in), static_cast<uint4*>(out), n8);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_gelu_bf16(const float* in, void* out, long long n, cudaStream_t stream) {
  const long long n8 = n / 8;
  const int blocks = int(std::min<long long>((n8 + 255) / 256, 148LL * 8));
  gelu_bf16_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(in), static_cast<uint4*>(out), n8);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_count_committed(const uint8_t* mask, int n_canvas, int canvas_len, int32_t* counts,
                                   cudaStream_t stream) {
  count_committed_kernel<<<n_canvas, 256, 0, stream>>>(mask, canvas_len, counts);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>();
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace canvas

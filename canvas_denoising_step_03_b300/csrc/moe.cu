// moe.cu -- the routing and data movement of a mixture-of-experts MLP block.
//
// Method: AI Trends summary of a DiffusionGemma 26B notebook
// (aitrends.kr/articles/94089), glossary entry "혼합 전문가(MoE)": every token
// is routed to its top-k experts, which run in parallel and are summed with
// weights, plus a shared expert that every token passes through; the routing
// score is the exponential of the router key's dot product with the input,
// renormalised (over the chosen experts) and scaled.  ThakiCloud,
// "DiffusionGemma 26B-A4B", "아키텍처": 128 experts, 8 active + 1 shared.
//
// The expert MLPs themselves are GEMMs on the tensor cores (gemm_tc.cu, its
// grouped mode); this file holds the steps between them:
//   moe_route_kernel    top-k of each token's router scores, their weights,
//                       per-expert token counts;
//   moe_offsets_kernel  each expert's row range in the grouped layout, padded
//                       to whole 128-row tiles, and the tile -> expert table;
//   moe_scatter_kernel  each (token, choice) copies the token's row into its
//                       expert's range and records where;
//   moe_act_kernel      the gated activation bf16(gelu(gate) * up);
//   moe_combine_kernel  out = sum over the token's choices (in choice order)
//                       of weight * expert output, + the shared expert.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace canvas {

namespace {

constexpr int kMaxExperts = 256;

// One warp per token: the top-k scores (largest first; equal scores: lower
// expert index first), w_j = exp(s_j - s_max) / sum over the chosen, times
// the expert's scale; counts[e] += 1 for every choice.
__global__ void __launch_bounds__(256) moe_route_kernel(MoeArgs a) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_global >= a.R) return;
  const int t = warp_global;
  constexpr int kPer = kMaxExperts / 32;
  float s[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = lane + 32 * j;
    s[j] = e < a.E ? a.scores[(size_t)t * a.E + e] : -INFINITY;
  }
  float chosen_s[16];
  int chosen_e[16];
  for (int r = 0; r < a.k; ++r) {
    // this lane's best (value, then lowest index), then across the warp
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = lane + 32 * j;
      if (e < a.E && (s[j] > bv || (s[j] == bv && e < be))) {
        bv = s[j];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be >= a.E) {  // no finite score left (a NaN input): keep the indices in range
      if (lane == 0) record_error(CANVAS_ERR_BOUNDS);
      be = 0;
    }
    chosen_s[r] = bv;
    chosen_e[r] = be;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (lane + 32 * j == be) s[j] = -INFINITY;  // taken
  }
  if (lane == 0) {
    const float m = chosen_s[0];
    float z = 0.f;
    float p[16];
    for (int r = 0; r < a.k; ++r) {
      p[r] = expf(chosen_s[r] - m);
      z += p[r];
    }
    for (int r = 0; r < a.k; ++r) {
      const int e = chosen_e[r];
      const float sc = a.expert_scale ? a.expert_scale[e] : 1.0f;
      a.topk_idx[(size_t)t * a.k + r] = e;
      a.topk_w[(size_t)t * a.k + r] = p[r] / z * sc;
      atomicAdd(&a.counts[e], 1);
    }
  }
}

// One block: expert e's rows start at offsets[e] (its count rounded up to
// whole 128-row tiles), tile t of the grouped layout belongs to the expert
// whose range holds it (-1 past the last), and the fill cursors are reset.
__global__ void __launch_bounds__(256) moe_offsets_kernel(MoeArgs a) {
  __shared__ int off[kMaxExperts + 1];
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < a.E; ++e) {
      off[e] = acc;
      acc += (a.counts[e] + 127) / 128 * 128;
    }
    off[a.E] = acc;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= a.E; e += blockDim.x) a.offsets[e] = off[e];
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.cursor[e] = 0;
  for (int tile = threadIdx.x; tile < a.max_tiles; tile += blockDim.x) {
    const int row = tile * 128;
    int g = -1;
    if (row < off[a.E]) {
      // the expert whose [off[e], off[e+1]) holds row (ranges are whole tiles)
      int lo = 0, hi = a.E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (off[mid] <= row) lo = mid; else hi = mid - 1;
      }
      g = lo;
    }
    a.group_of_mtile[tile] = g;
  }
}

// One warp per (token, choice): the token's row into its expert's next free
// row of the grouped layout; slot[t, j] records the row.  (The order of rows
// inside an expert's range depends on timing; every output row depends only
// on its own input row, and the combine reads them back by slot, so results
// do not.)
__global__ void __launch_bounds__(256) moe_scatter_kernel(MoeArgs a) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_global >= a.R * a.k) return;
  const int t = warp_global / a.k;
  const int e = a.topk_idx[warp_global];
  int pos = 0;
  if (lane == 0) {
    pos = a.offsets[e] + atomicAdd(&a.cursor[e], 1);
    a.slot[warp_global] = pos;
  }
  pos = __shfl_sync(0xffffffffu, pos, 0);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + (size_t)t * a.D);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.xg) + (size_t)pos * a.D);
  for (int c = lane; c < a.D / 8; c += 32) dst[c] = src[c];
}

// act[r, f] = bf16(gelu(gate[r, f]) * up[r, f]) (GELU in its tanh form,
// evaluated in fp32 as x / (1 + exp(-2u)): 1 + tanh(u) = 2 / (1 + exp(-2u))
// keeps its relative accuracy for negative x)
__global__ void __launch_bounds__(256) moe_act_kernel(const float4* __restrict__ gate, const float4* __restrict__ up,
                                                      uint2* __restrict__ act, long long n4) {
  const float k0 = 0.7978845608028654f, k1 = 0.044715f;
  for (long long e = blockIdx.x * 256LL + threadIdx.x; e < n4; e += (long long)gridDim.x * 256) {
    const float4 g4 = gate[e], u4 = up[e];
    float g[4] = {g4.x, g4.y, g4.z, g4.w};
    const float u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x = g[j];
      g[j] = x / (1.0f + expf(-2.0f * k0 * (x + k1 * x * x * x))) * u[j];
    }
    act[e] = make_uint2(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]));
  }
}

// out = sum_j w[t, j] * yg[slot[t, j]] (j in choice order) + shared[t]
// (fp32).  One block per (token, 512 columns): the token's weights and slots
// are read once into shared memory, and each thread issues the loads of all
// the token's choices for its four columns before it adds them.
constexpr int kCombineCols = 512;
constexpr int kMaxChoices = 16;
__global__ void __launch_bounds__(kCombineCols / 4) moe_combine_kernel(MoeArgs a) {
  __shared__ float w_s[kMaxChoices];
  __shared__ int slot_s[kMaxChoices];
  const int t = blockIdx.y;
  if (threadIdx.x < a.k) {
    w_s[threadIdx.x] = a.topk_w[(size_t)t * a.k + threadIdx.x];
    slot_s[threadIdx.x] = a.slot[(size_t)t * a.k + threadIdx.x];
  }
  __syncthreads();
  const int c = blockIdx.x * kCombineCols + threadIdx.x * 4;
  if (c >= a.D) return;
  float4 y[kMaxChoices];
#pragma unroll
  for (int j = 0; j < kMaxChoices; ++j)
    if (j < a.k) y[j] = __ldcs(reinterpret_cast<const float4*>(a.yg + (size_t)slot_s[j] * a.D + c));
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kMaxChoices; ++j) {
    if (j < a.k) {
      const float w = w_s[j];
      o.x = fmaf(w, y[j].x, o.x);
      o.y = fmaf(w, y[j].y, o.y);
      o.z = fmaf(w, y[j].z, o.z);
      o.w = fmaf(w, y[j].w, o.w);
    }
  }
  if (a.ys) {
    const float4 sh = *reinterpret_cast<const float4*>(a.ys + (size_t)t * a.D + c);
    o.x += sh.x;
    o.y += sh.y;
    o.z += sh.z;
    o.w += sh.w;
  }
  *reinterpret_cast<float4*>(a.out + (size_t)t * a.D + c) = o;
}

}  // namespace

cudaError_t launch_moe_route(const MoeArgs& a, cudaStream_t stream) {
  if (a.E > kMaxExperts || a.k > 16 || a.k > a.E) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.E, stream);
  if (e != cudaSuccess) return e;
  moe_route_kernel<<<(a.R * 32 + 255) / 256, 256, 0, stream>>>(a);
  moe_offsets_kernel<<<1, 256, 0, stream>>>(a);
  moe_scatter_kernel<<<(int)(((long long)a.R * a.k * 32 + 255) / 256), 256, 0, stream>>>(a);
  count_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_moe_act(const float* gate, const float* up, void* act, long long n, cudaStream_t stream) {
  const long long n4 = n / 4;
  const int blocks = int(std::min<long long>((n4 + 255) / 256, 148LL * 8));
  moe_act_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(gate), reinterpret_cast<const float4*>(up),
                                             static_cast<uint2*>(act), n4);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_moe_combine(const MoeArgs& a, cudaStream_t stream) {
  if (a.k > kMaxChoices || a.D % 4 != 0) return cudaErrorInvalidValue;
  const dim3 grid((a.D + kCombineCols - 1) / kCombineCols, a.R, 1);
  moe_combine_kernel<<<grid, kCombineCols / 4, 0, stream>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace canvas

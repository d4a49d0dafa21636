// prologue.cu -- QK RMSNorm + split-half RoPE of the canvas rows, the key
// preparation of global layers, and the gathering of the key-sequence tail.
//
// Method: AI Trends summary of a DiffusionGemma 26B notebook
// (aitrends.kr/articles/94089), "섹션별 상세": the rms() snippet
// (w * x * sqrt(d) / (||x||_2 + eps), norm in fp32, result cast back to the
// input dtype), the rotate() snippet (pairs t and t + d/2; angle
// (l + start) * freq[t mod d/2]; zero frequencies leave a channel unchanged --
// partial RoPE, result cast back to the input dtype), and the attention-block
// snippet (q and k are normed and rotated, v is not; on full-attention layers
// W_v = W_k, so the value is the raw shared projection r and the key is
// rotate(rms(r)) at the key's own position).
//
// Every row is normed in fp32, rotated in fp32 and stored once in the path's
// dtype (bf16: round to nearest even).  A global-layer canvas row first
// stores its raw projection r (it becomes a cache row like any other) and
// computes its key from the stored r.
//
// Layout of the key sequence (prefix read in place up to P64, then the dense
// tail buffers Kx / Vx): see kernels.h.
#include "common.cuh"
#include "kernels.h"

namespace canvas {

namespace {

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// value after a store in T (bf16: rounded; fp32: unchanged)
template <typename T>
__device__ __forceinline__ float stored(float v) {
  return to_f32(from_f32<T>(v));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kMaxPairsPerLane = 8;  // d <= 512: d/2 / 32 pairs per lane

// One row held by a warp as pairs (lo[k], hi[k]) = (x[t], x[t + d/2]),
// t = lane + 32 k, k < np = d / 64.
struct Row {
  float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
};

template <typename T>
__device__ __forceinline__ void load_row(const T* src, int d, Row& r) {
  const int lane = threadIdx.x & 31, half = d / 2, np = half / 32;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    if (k < np) {
      r.lo[k] = to_f32(src[lane + 32 * k]);
      r.hi[k] = to_f32(src[half + lane + 32 * k]);
    }
  }
}

__device__ __forceinline__ float row_norm(const Row& r, int d) {
  const int np = d / 64;
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k)
    if (k < np) ss += r.lo[k] * r.lo[k] + r.hi[k] * r.hi[k];
  return sqrtf(warp_sum(ss));
}

template <typename T>
__device__ __forceinline__ void store_row(T* dst, int d, const Row& r) {
  const int lane = threadIdx.x & 31, half = d / 2, np = half / 32;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    if (k < np) {
      dst[lane + 32 * k] = from_f32<T>(r.lo[k]);
      dst[half + lane + 32 * k] = from_f32<T>(r.hi[k]);
    }
  }
}

template <typename T>
__device__ __forceinline__ void zero_row(T* dst, int d) {
  for (int t = threadIdx.x & 31; t < d; t += 32) dst[t] = from_f32<T>(0.f);
}

// rotate(rms(x, gamma)) at position pos, in place (fp32)
__device__ __forceinline__ void norm_rope(Row& r, int d, const float* gamma, float eps, const float* freq,
                                          int pos) {
  const int lane = threadIdx.x & 31, half = d / 2, np = half / 32;
  const float scale = sqrtf(float(d)) / (row_norm(r, d) + eps);
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    if (k >= np) break;
    const int t = lane + 32 * k;
    const float a = gamma[t] * r.lo[k] * scale;
    const float b = gamma[t + half] * r.hi[k] * scale;
    const float f = freq[t];
    if (f != 0.f) {
      float c, s;
      rope_cos_sin(pos, rope_turns(f), &c, &s);
      r.lo[k] = c * a - s * b;
      r.hi[k] = c * b + s * a;
    } else {
      r.lo[k] = a;
      r.hi[k] = b;
    }
  }
}

template <typename T>
__device__ __forceinline__ void round_row(Row& r, int d) {
  const int np = d / 64;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    if (k < np) {
      r.lo[k] = stored<T>(r.lo[k]);
      r.hi[k] = stored<T>(r.hi[k]);
    }
  }
}

// Global layers: from a stored raw row r at position pos, write the key
// rotate(rms(r)) to kdst, r itself to vdst (if non-null) and the value row
// scalar sqrt(d) / (|r| + eps) to *vs (lane 0).
template <typename T>
__device__ __forceinline__ void global_row(Row& r, int d, const float* gamma_k, float eps, const float* freq,
                                           int pos, T* kdst, T* vdst, float* vs) {
  if (vdst) store_row(vdst, d, r);
  const float nrm = row_norm(r, d);
  if (vs && (threadIdx.x & 31) == 0) *vs = sqrtf(float(d)) / (nrm + eps);
  norm_rope(r, d, gamma_k, eps, freq, pos);
  store_row(kdst, d, r);
}

// One warp per (canvas token, head).  Heads: Hq query heads, then Hkv key
// heads, then (sliding) Hkv value heads.
template <typename T>
__global__ void __launch_bounds__(256) prologue_kernel(PrologueArgs p) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int G = p.Hq / p.Hkv;
  const int heads = p.Hq + p.Hkv + (p.global ? 0 : p.Hkv);
  const int total = p.B * p.C * heads;
  if (warp_global >= total) return;
  const int row = warp_global / heads;  // token b*C + i
  const int hh = warp_global % heads;
  const int b = row / p.C, i = row % p.C;
  const int d = p.d;
  const int P = p.prefix_len[b];
  if (P < 0) return;                     // reported by the key-prep kernel
  const int pos = P + i;
  const int t = P - (P & ~63) + i;       // tail row of this canvas token

  Row r;
  if (hh < p.Hq) {
    const int h = hh, hk = h / G, g = h % G;
    load_row(p.proj_q + (size_t)row * p.Hq * d + (size_t)h * d, d, r);
    norm_rope(r, d, p.gamma_q, p.eps, p.freq, pos);
    store_row(static_cast<T*>(p.Qp) + ((((size_t)b * p.Hkv + hk) * G + g) * p.C + i) * d, d, r);
  } else if (hh < p.Hq + p.Hkv) {
    const int hk = hh - p.Hq;
    load_row(p.proj_k + (size_t)row * p.Hkv * d + (size_t)hk * d, d, r);
    const size_t trow = ((size_t)b * p.Hkv + hk) * p.Tpad + t;
    T* kdst = static_cast<T*>(p.Kx) + trow * d;
    if (p.global) {
      round_row<T>(r, d);  // the stored raw row r: value, and source of the key
      global_row<T>(r, d, p.gamma_k, p.eps, p.freq, pos, kdst, static_cast<T*>(p.Vx) + trow * d,
                    p.vs_tail + trow);
    } else {
      norm_rope(r, d, p.gamma_k, p.eps, p.freq, pos);
      store_row(kdst, d, r);
    }
  } else {
    const int hk = hh - p.Hq - p.Hkv;
    load_row(p.proj_v + (size_t)row * p.Hkv * d + (size_t)hk * d, d, r);
    store_row(static_cast<T*>(p.Vx) + (((size_t)b * p.Hkv + hk) * p.Tpad + t) * d, d, r);
  }
}

// One warp per (b, KV head, row).  Rows [0, max_prefix) (global layers only):
// prefix keys Kt and value scalars for positions below P64.  Rows
// [max_prefix, max_prefix + Tpad): tail row t = row - max_prefix -- prefix
// rows P64 + t < P are gathered from the cache, rows past the canvas are
// zeroed, canvas rows are left to the prologue kernel.
template <typename T>
__global__ void __launch_bounds__(256) key_prep_kernel(KeyPrepArgs k) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int row0 = k.global ? 0 : k.max_prefix;
  const int L = k.max_prefix + k.Tpad - row0;
  const int total = k.B * k.Hkv * L;
  if (warp_global >= total) return;
  const int row = row0 + warp_global % L;
  const int hk = (warp_global / L) % k.Hkv;
  const int b = warp_global / (L * k.Hkv);
  const int P = k.prefix_len[b];
  if (P < 0 || P > k.max_prefix) {
    if (lane == 0 && row == row0 && hk == 0) record_error(CANVAS_ERR_BOUNDS);
    return;
  }
  const int P64 = P & ~63;
  const int d = k.d;
  int pos, t = -1;
  if (row < k.max_prefix) {
    pos = row;
    if (pos >= P64) return;
  } else {
    t = row - k.max_prefix;
    pos = P64 + t;
    const size_t trow = ((size_t)b * k.Hkv + hk) * k.Tpad + t;
    if (pos >= P + k.C) {  // past the canvas: zero rows (finite operands for padded blocks)
      zero_row(static_cast<T*>(k.Kx) + trow * d, d);
      zero_row(static_cast<T*>(k.Vx) + trow * d, d);
      if (k.global && lane == 0) k.vs_tail[trow] = 0.f;
      return;
    }
    if (pos >= P) return;  // canvas row
  }
  // a committed prefix row at position pos: locate it in the paged cache
  const int lp = pos / k.page_tokens, off = pos % k.page_tokens;
  const int page = (lp < k.max_pages) ? k.block_table[(size_t)b * k.max_pages + lp] : -1;
  if (page < 0 || page >= k.num_pages) {
    if (lane == 0) record_error(CANVAS_ERR_BOUNDS);
    return;
  }
  const size_t src = (((size_t)page * k.Hkv + hk) * k.page_tokens + off) * d;
  Row r;
  load_row(static_cast<const T*>(k.k_pool) + src, d, r);
  if (t < 0) {
    const size_t orow = ((size_t)b * k.Hkv + hk) * k.max_prefix + pos;
    global_row<T>(r, d, k.gamma_k, k.eps, k.freq, pos, static_cast<T*>(k.Kt) + orow * d, nullptr,
                  k.vs_pre + orow);
    return;
  }
  const size_t trow = ((size_t)b * k.Hkv + hk) * k.Tpad + t;
  if (k.global) {
    global_row<T>(r, d, k.gamma_k, k.eps, k.freq, pos, static_cast<T*>(k.Kx) + trow * d,
                  static_cast<T*>(k.Vx) + trow * d, k.vs_tail + trow);
  } else {
    store_row(static_cast<T*>(k.Kx) + trow * d, d, r);
    Row v;
    load_row(static_cast<const T*>(k.v_pool) + src, d, v);
    store_row(static_cast<T*>(k.Vx) + trow * d, d, v);
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueArgs& p, bool bf16, cudaStream_t stream) {
  const int heads = p.Hq + p.Hkv + (p.global ? 0 : p.Hkv);
  const long long warps = (long long)p.B * p.C * heads;
  const int blocks = int((warps * 32 + 255) / 256);
  if (bf16)
    prologue_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(p);
  else
    prologue_kernel<float><<<blocks, 256, 0, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_key_prep(const KeyPrepArgs& k, bool bf16, cudaStream_t stream) {
  const int rows = (k.global ? k.max_prefix : 0) + k.Tpad;
  const long long warps = (long long)k.B * k.Hkv * rows;
  const int blocks = int((warps * 32 + 255) / 256);
  if (bf16)
    key_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(k);
  else
    key_prep_kernel<float><<<blocks, 256, 0, stream>>>(k);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace canvas

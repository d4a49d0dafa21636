// prologue.cu -- QK RMSNorm + split-half RoPE of the canvas rows, and the
// key preparation of global layers.
//
// Method: AI Trends summary of a DiffusionGemma 26B notebook
// (aitrends.kr/articles/94089), "섹션별 상세": the rms() snippet
// (w * x * sqrt(d) / (||x||_2 + eps), norm in fp32), the rotate() snippet
// (pairs t and t + d/2; angle (l + start) * freq[t mod d/2]; zero frequencies
// leave a channel unchanged -- partial RoPE), and the attention-block snippet
// (q and k are normed and rotated, v is not; on full-attention layers
// W_v = W_k, so the value is the raw shared projection).
//
// Canvas rows (one warp per (token, head)): the fp32 projection is normed in
// fp32, rotated in fp32 at position prefix_len[b] + i, and stored once in the
// path's dtype (bf16: round to nearest even).
//
// Global layers keep the raw shared projection r in the cache.  With the
// constant QK-norm vector the pages report, rms(r) = gamma_k * s * r with the
// row scalar s = sqrt(d) / (||r|| + eps), and rotation is linear, so
// rotate(rms(r)) = gamma_k * s * rotate(r).  key_prep stores rotate(r) in the
// path's dtype and the scalars gamma_k * s (key scale) and s (value scale, for
// the unit-RMS value variant); the attention kernels apply them to scores.
#include "common.cuh"
#include "kernels.h"

namespace canvas {

namespace {

template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v);
template <>
__device__ __forceinline__ void store_elem<float>(float* p, float v) {
  *p = v;
}
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kMaxPairsPerLane = 8;  // d <= 512: d/2 / 32 pairs per lane

// rms-normalise and rotate one fp32 row held as pairs (lo[t], hi[t]) =
// (x[t], x[t + d/2]) for t = lane + 32 k; write it to dst in T.
template <typename T>
__device__ __forceinline__ void norm_rope_store(float (&lo)[kMaxPairsPerLane], float (&hi)[kMaxPairsPerLane],
                                                int d, const float* gamma, float eps, const float* freq, int pos,
                                                bool do_norm, T* dst) {
  const int lane = threadIdx.x & 31, half = d / 2, np = half / 32;
  float scale = 1.f;
  if (do_norm) {
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxPairsPerLane; ++k)
      if (k < np) ss += lo[k] * lo[k] + hi[k] * hi[k];
    ss = warp_sum(ss);
    scale = sqrtf(float(d)) / (sqrtf(ss) + eps);
  }
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    if (k >= np) break;
    const int t = lane + 32 * k;
    float a = lo[k], b = hi[k];
    if (do_norm) {
      a = gamma[t] * a * scale;
      b = gamma[t + half] * b * scale;
    }
    const float f = freq[t];
    float ra = a, rb = b;
    if (f != 0.f) {
      float c, s;
      rope_cos_sin(pos, rope_turns(f), &c, &s);
      ra = c * a - s * b;
      rb = c * b + s * a;
    }
    store_elem(dst + t, ra);
    store_elem(dst + t + half, rb);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) prologue_kernel(PrologueArgs p) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;
  const int heads = p.Hq + p.Hkv + (p.global ? 0 : p.Hkv);
  const int total = p.B * p.C * heads;
  if (warp_global >= total) return;
  const int row = warp_global / heads;  // token b*C + i
  const int hh = warp_global % heads;
  const int b = row / p.C, i = row % p.C;
  const int d = p.d, half = d / 2, np = half / 32;
  const int pos = p.prefix_len[b] + i;

  const float* src;
  int kind, h;  // 0 = q, 1 = k, 2 = v
  if (hh < p.Hq) {
    kind = 0; h = hh;
    src = p.proj_q + (size_t)row * p.Hq * d + (size_t)h * d;
  } else if (hh < p.Hq + p.Hkv) {
    kind = 1; h = hh - p.Hq;
    src = p.proj_k + (size_t)row * p.Hkv * d + (size_t)h * d;
  } else {
    kind = 2; h = hh - p.Hq - p.Hkv;
    src = p.proj_v + (size_t)row * p.Hkv * d + (size_t)h * d;
  }
  float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    if (k < np) {
      lo[k] = src[lane + 32 * k];
      hi[k] = src[half + lane + 32 * k];
    }
  }
  if (kind == 0) {
    const int hk = h / G, g = h % G;
    T* dst = static_cast<T*>(p.Qp) + ((((size_t)b * p.Hkv + hk) * G + g) * p.C + i) * d;
    norm_rope_store<T>(lo, hi, d, p.gamma_q, p.eps, p.freq, pos, true, dst);
  } else if (kind == 1) {
    T* dst = static_cast<T*>(p.Kc) + (((size_t)b * p.Hkv + h) * p.C + i) * d;
    if (p.global) {
      // raw shared projection r: stored as is (it is the value and the key source)
#pragma unroll
      for (int k = 0; k < kMaxPairsPerLane; ++k) {
        if (k >= np) break;
        store_elem(dst + lane + 32 * k, lo[k]);
        store_elem(dst + half + lane + 32 * k, hi[k]);
      }
    } else {
      norm_rope_store<T>(lo, hi, d, p.gamma_k, p.eps, p.freq, pos, true, dst);
    }
  } else {
    T* dst = static_cast<T*>(p.Vc) + (((size_t)b * p.Hkv + h) * p.C + i) * d;
#pragma unroll
    for (int k = 0; k < kMaxPairsPerLane; ++k) {
      if (k >= np) break;
      store_elem(dst + lane + 32 * k, lo[k]);
      store_elem(dst + half + lane + 32 * k, hi[k]);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) key_prep_kernel(KeyPrepArgs k) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int L = k.max_prefix + k.C;
  const int total = k.B * k.Hkv * L;
  // the factorisation rotate(rms(r)) = gamma * s * rotate(r) needs a constant gamma_k
  if (blockIdx.x == 0 && threadIdx.x < 32) {
    bool same = true;
    for (int t = lane; t < k.d; t += 32) same = same && (k.gamma_k[t] == k.gamma_k[0]);
    if (!__all_sync(0xffffffffu, same) && lane == 0) record_error(CANVAS_ERR_UNSUPPORTED);
  }
  if (warp_global >= total) return;
  const int j = warp_global % L;
  const int hk = (warp_global / L) % k.Hkv;
  const int b = warp_global / (L * k.Hkv);
  const int P = k.prefix_len[b];
  if (P < 0 || P > k.max_prefix) {
    if (lane == 0 && j == 0 && hk == 0) record_error(CANVAS_ERR_BOUNDS);
    return;
  }
  if (j >= P + k.C) return;
  const int d = k.d, half = d / 2, np = half / 32;
  const T* src;
  int pos;
  if (j < P) {
    const int lp = j / k.page_tokens, off = j % k.page_tokens;
    const int page = (lp < k.max_pages) ? k.block_table[(size_t)b * k.max_pages + lp] : -1;
    if (page < 0 || page >= k.num_pages) {
      if (lane == 0) record_error(CANVAS_ERR_BOUNDS);
      return;
    }
    src = static_cast<const T*>(k.pool) + (((size_t)page * k.Hkv + hk) * k.page_tokens + off) * d;
    pos = j;
  } else {
    src = static_cast<const T*>(k.Rc) + (((size_t)b * k.Hkv + hk) * k.C + (j - P)) * d;
    pos = j;  // canvas row i sits at P + i
  }
  float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxPairsPerLane; ++q) {
    if (q < np) {
      lo[q] = to_f32(src[lane + 32 * q]);
      hi[q] = to_f32(src[half + lane + 32 * q]);
      ss += lo[q] * lo[q] + hi[q] * hi[q];
    }
  }
  ss = warp_sum(ss);
  const float s = sqrtf(float(d)) / (sqrtf(ss) + k.eps);
  const size_t orow = ((size_t)b * k.Hkv + hk) * L + j;
  if (lane == 0) {
    k.ks[orow] = k.gamma_k[0] * s;
    k.vs[orow] = s;
  }
  T* dst = static_cast<T*>(k.Kt) + orow * d;
  norm_rope_store<T>(lo, hi, d, nullptr, 0.f, k.freq, pos, false, dst);
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
  const long long warps = (long long)k.B * k.Hkv * (k.max_prefix + k.C);
  const int blocks = int((warps * 32 + 255) / 256);
  if (bf16)
    key_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(k);
  else
    key_prep_kernel<float><<<blocks, 256, 0, stream>>>(k);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace canvas

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

#include <algorithm>

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

// One row held by a warp as pairs (lo[k], hi[k]) = (x[t], x[t + d/2]).  Lane
// `lane` owns chunks c < kChunks of kVec consecutive elements,
// t = (lane + 32 c) * kVec + e: each warp access covers 32 * kVec contiguous
// elements (coalesced), and the rotated pairs of a partial RoPE (the leading
// frequencies) are spread over all lanes rather than packed into a few.
struct Row {
  float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
};

template <int D>
struct RowShape {
  static constexpr int half = D / 2;
  static constexpr int np = half / 32;                 // elements per lane per half
  static constexpr int kVec = (np % 2 == 0) ? 2 : 1;   // consecutive elements per access
  static constexpr int kChunks = np / kVec;
  __device__ __forceinline__ static int elem(int lane, int k) { return (lane + 32 * (k / kVec)) * kVec + k % kVec; }
};

template <typename T, int N>
struct VecIO;
template <int N>
struct VecIO<__nv_bfloat16, N> {
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* x) {
    if constexpr (N == 2) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
      x[0] = __uint_as_float(u << 16);
      x[1] = __uint_as_float(u & 0xffff0000u);
    } else {
      x[0] = __bfloat162float(p[0]);
    }
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* x) {
    if constexpr (N == 2)
      *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(x[0], x[1]);
    else
      p[0] = __float2bfloat16_rn(x[0]);
  }
};
template <int N>
struct VecIO<float, N> {
  __device__ __forceinline__ static void load(const float* p, float* x) {
    if constexpr (N == 2) {
      const float2 v = *reinterpret_cast<const float2*>(p);
      x[0] = v.x;
      x[1] = v.y;
    } else {
      x[0] = p[0];
    }
  }
  __device__ __forceinline__ static void store(float* p, const float* x) {
    if constexpr (N == 2)
      *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    else
      p[0] = x[0];
  }
};

template <typename T, int D>
__device__ __forceinline__ void load_row(const T* src, Row& r) {
  using S = RowShape<D>;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < S::kChunks; ++c) {
    const int t = (lane + 32 * c) * S::kVec;
    VecIO<T, S::kVec>::load(src + t, r.lo + c * S::kVec);
    VecIO<T, S::kVec>::load(src + S::half + t, r.hi + c * S::kVec);
  }
}

// A projection row summed over its split-K partials (slices `stride` floats
// apart), in split order from 0: the same fp32 additions as the GEMM's own
// split reduce, so the row is bit-identical to a reduced projection.
template <int D>
__device__ __forceinline__ void load_split_row(const float* src, size_t stride, int splits, Row& r) {
  if (splits <= 1) {
    load_row<float, D>(src, r);
    return;
  }
  Row t;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) r.lo[k] = r.hi[k] = 0.f;
  for (int sp = 0; sp < splits; ++sp) {
    load_row<float, D>(src + sp * stride, t);
#pragma unroll
    for (int k = 0; k < D / 64; ++k) {
      r.lo[k] += t.lo[k];
      r.hi[k] += t.hi[k];
    }
  }
}

template <typename T, int D>
__device__ __forceinline__ void store_row(T* dst, const Row& r) {
  using S = RowShape<D>;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < S::kChunks; ++c) {
    const int t = (lane + 32 * c) * S::kVec;
    VecIO<T, S::kVec>::store(dst + t, r.lo + c * S::kVec);
    VecIO<T, S::kVec>::store(dst + S::half + t, r.hi + c * S::kVec);
  }
}

template <typename T, int D>
__device__ __forceinline__ void zero_row(T* dst) {
  Row z;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) z.lo[k] = z.hi[k] = 0.f;
  store_row<T, D>(dst, z);
}

template <int D>
__device__ __forceinline__ float row_norm(const Row& r) {
  constexpr int np = D / 64;
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < np; ++k) ss += r.lo[k] * r.lo[k] + r.hi[k] * r.hi[k];
  return sqrtf(warp_sum(ss));
}

// rotate(rms(x, gamma)) at position pos, in place (fp32)
template <int D>
__device__ __forceinline__ void norm_rope(Row& r, const float* gamma, float eps, const float* freq, int pos) {
  using S = RowShape<D>;
  constexpr int np = S::np, half = S::half;
  const int lane = threadIdx.x & 31;
  const float scale = sqrtf(float(D)) / (row_norm<D>(r) + eps);
#pragma unroll
  for (int k = 0; k < np; ++k) {
    const int t = S::elem(lane, k);
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

template <typename T, int D>
__device__ __forceinline__ void round_row(Row& r) {
#pragma unroll
  for (int k = 0; k < D / 64; ++k) {
    r.lo[k] = stored<T>(r.lo[k]);
    r.hi[k] = stored<T>(r.hi[k]);
  }
}

// Global layers: from a stored raw row r at position pos, write the key
// rotate(rms(r)) to kdst, r itself to vdst (if non-null) and the value row
// scalar sqrt(d) / (|r| + eps) to *vs (lane 0).
template <typename T, int D>
__device__ __forceinline__ void global_row(Row& r, const float* gamma_k, float eps, const float* freq, int pos,
                                           T* kdst, T* vdst, float* vs) {
  if (vdst) store_row<T, D>(vdst, r);
  const float nrm = row_norm<D>(r);
  if (vs && (threadIdx.x & 31) == 0) *vs = sqrtf(float(D)) / (nrm + eps);
  norm_rope<D>(r, gamma_k, eps, freq, pos);
  store_row<T, D>(kdst, r);
}

// Four stored raw rows r[j] at positions pos0 + j (global layers): their keys
// rotate(rms(r[j])) to kdst + j D and value scalars to vs[j].  The same
// arithmetic as global_row, element by element, with each QK-norm weight,
// frequency and turn split loaded or formed once for the four rows and one
// norm per row.
template <typename T, int D>
__device__ __forceinline__ void global_rows4(Row (&r)[4], const float* gamma, float eps, const float* freq, int pos0,
                                             T* kdst, float* vs) {
  using S = RowShape<D>;
  constexpr int np = S::np, half = S::half;
  const int lane = threadIdx.x & 31;
  float scale[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    scale[j] = sqrtf(float(D)) / (row_norm<D>(r[j]) + eps);
    if (lane == 0) vs[j] = scale[j];
  }
#pragma unroll
  for (int k = 0; k < np; ++k) {
    const int t = S::elem(lane, k);
    const float g_lo = gamma[t], g_hi = gamma[t + half];
    const float f = freq[t];
    if (f != 0.f) {
      const RopeTurns tw = rope_turns(f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = g_lo * r[j].lo[k] * scale[j];
        const float b = g_hi * r[j].hi[k] * scale[j];
        float c, sn;
        rope_cos_sin(pos0 + j, tw, &c, &sn);
        r[j].lo[k] = c * a - sn * b;
        r[j].hi[k] = c * b + sn * a;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        r[j].lo[k] = g_lo * r[j].lo[k] * scale[j];
        r[j].hi[k] = g_hi * r[j].hi[k] * scale[j];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) store_row<T, D>(kdst + j * D, r[j]);
}

// One warp per (canvas token, head).  Heads: Hq query heads, then Hkv key
// heads, then (sliding) Hkv value heads.
template <typename T, int D>
__global__ void __launch_bounds__(256) prologue_kernel(PrologueArgs p) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int G = p.Hq / p.Hkv;
  const int heads = p.Hq + p.Hkv + (p.global ? 0 : p.Hkv);
  const int total = p.B * p.C * heads;
  if (warp_global >= total) return;
  const int row = warp_global / heads;  // token b*C + i
  const int hh = warp_global % heads;
  const int b = row / p.C, i = row % p.C;
  constexpr int d = D;
  const int P = p.prefix_len[b];
  if (P < 0) return;                     // reported by the key-prep kernel
  const int pos = P + i;
  const int t = P - (P & ~63) + i;       // tail row of this canvas token

  Row r;
  const size_t M = (size_t)p.B * p.C;
  if (hh < p.Hq) {
    const int h = hh, hk = h / G, g = h % G;
    load_split_row<D>(p.proj_q + (size_t)row * p.Hq * d + (size_t)h * d, M * p.Hq * d, p.splits, r);
    norm_rope<D>(r, p.gamma_q, p.eps, p.freq, pos);
    store_row<T, D>(static_cast<T*>(p.Qp) + ((((size_t)b * p.Hkv + hk) * G + g) * p.C + i) * d, r);
  } else if (hh < p.Hq + p.Hkv) {
    const int hk = hh - p.Hq;
    load_split_row<D>(p.proj_k + (size_t)row * p.Hkv * d + (size_t)hk * d, M * p.Hkv * d, p.splits, r);
    const size_t trow = ((size_t)b * p.Hkv + hk) * p.Tpad + t;
    T* kdst = static_cast<T*>(p.Kx) + trow * d;
    if (p.global) {
      round_row<T, D>(r);  // the stored raw row r: value, and source of the key
      global_row<T, D>(r, p.gamma_k, p.eps, p.freq, pos, kdst, static_cast<T*>(p.Vx) + trow * d,
                       p.vs_tail + trow);
    } else {
      norm_rope<D>(r, p.gamma_k, p.eps, p.freq, pos);
      store_row<T, D>(kdst, r);
    }
  } else {
    const int hk = hh - p.Hq - p.Hkv;
    load_split_row<D>(p.proj_v + (size_t)row * p.Hkv * d + (size_t)hk * d, M * p.Hkv * d, p.splits, r);
    store_row<T, D>(static_cast<T*>(p.Vx) + (((size_t)b * p.Hkv + hk) * p.Tpad + t) * d, r);
  }
}

template <typename T, int D>
__device__ __forceinline__ void key_prep_row(const KeyPrepArgs& k, int w, int row0, int L) {
  const int lane = threadIdx.x & 31;
  const int row = row0 + w % L;
  const int hk = (w / L) % k.Hkv;
  const int b = w / (L * k.Hkv);
  const int P = k.prefix_len[b];
  if (P < 0 || P > k.max_prefix) {
    if (lane == 0 && row == row0 && hk == 0) record_error(CANVAS_ERR_BOUNDS);
    return;
  }
  const int P64 = P & ~63;
  constexpr int d = D;
  int pos, t = -1;
  if (row < k.max_prefix) {
    pos = row;
    if (pos >= P64) return;
  } else {
    t = row - k.max_prefix;
    pos = P64 + t;
    const size_t trow = ((size_t)b * k.Hkv + hk) * k.Tpad + t;
    if (pos >= P + k.C) {  // past the canvas: zero rows (finite operands for padded blocks)
      zero_row<T, D>(static_cast<T*>(k.Kx) + trow * d);
      zero_row<T, D>(static_cast<T*>(k.Vx) + trow * d);
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
  load_row<T, D>(static_cast<const T*>(k.k_pool) + src, r);
  if (t < 0) {
    const size_t orow = ((size_t)b * k.Hkv + hk) * k.max_prefix + pos;
    global_row<T, D>(r, k.gamma_k, k.eps, k.freq, pos, static_cast<T*>(k.Kt) + orow * d, nullptr,
                     k.vs_pre + orow);
    return;
  }
  const size_t trow = ((size_t)b * k.Hkv + hk) * k.Tpad + t;
  if (k.global) {
    global_row<T, D>(r, k.gamma_k, k.eps, k.freq, pos, static_cast<T*>(k.Kx) + trow * d,
                     static_cast<T*>(k.Vx) + trow * d, k.vs_tail + trow);
  } else {
    store_row<T, D>(static_cast<T*>(k.Kx) + trow * d, r);
    Row v;
    load_row<T, D>(static_cast<const T*>(k.v_pool) + src, v);
    store_row<T, D>(static_cast<T*>(k.Vx) + trow * d, v);
  }
}

// Global layers, prefix rows below P64: four consecutive positions per warp
// (one block-table lookup, the four rows' loads in flight together), each
// written as its prepared key to Kt with its value scalar.
template <typename T, int D>
__device__ __forceinline__ void key_prep_prefix4(const KeyPrepArgs& k, int w, int G4) {
  const int lane = threadIdx.x & 31;
  const int g4 = w % G4;
  const int hk = (w / G4) % k.Hkv;
  const int b = w / (G4 * k.Hkv);
  const int P = k.prefix_len[b];
  if (P < 0 || P > k.max_prefix) return;  // reported by the tail pass
  const int pos0 = 4 * g4;
  if (pos0 >= (P & ~63)) return;  // P64 is a multiple of 4: a group is all prefix or all past it
  const int lp = pos0 / k.page_tokens, off = pos0 % k.page_tokens;  // the four rows share the page
  const int page = (lp < k.max_pages) ? k.block_table[(size_t)b * k.max_pages + lp] : -1;
  if (page < 0 || page >= k.num_pages) {
    if (lane == 0) record_error(CANVAS_ERR_BOUNDS);
    return;
  }
  const T* src = static_cast<const T*>(k.k_pool) + (((size_t)page * k.Hkv + hk) * k.page_tokens + off) * D;
  Row r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) load_row<T, D>(src + j * D, r[j]);
  const size_t orow = ((size_t)b * k.Hkv + hk) * k.max_prefix + pos0;
  global_rows4<T, D>(r, k.gamma_k, k.eps, k.freq, pos0, static_cast<T*>(k.Kt) + orow * D, k.vs_pre + orow);
}

// Grid-stride over warps.  Global layers first prepare the prefix keys Kt
// (four rows per warp, above).  Then one warp per tail row t = 0 .. Tpad-1
// of every (b, KV head): prefix rows P64 + t < P are gathered from the cache
// (global: prepared, raw values kept), rows past the canvas are zeroed,
// canvas rows are left to the prologue kernel.
template <typename T, int D>
__global__ void __launch_bounds__(256, 2) key_prep_kernel(KeyPrepArgs k) {
  const int nwarps = int((gridDim.x * blockDim.x) >> 5);
  const int w0 = int((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (k.global && k.page_tokens % 4 == 0) {
    const int G4 = (k.max_prefix + 3) / 4;
    const int total4 = k.B * k.Hkv * G4;
    for (int w = w0; w < total4; w += nwarps) key_prep_prefix4<T, D>(k, w, G4);
  } else if (k.global) {
    const int totalp = k.B * k.Hkv * k.max_prefix;  // pages of other sizes: one row per warp
    for (int w = w0; w < totalp; w += nwarps) key_prep_row<T, D>(k, w, 0, k.max_prefix);
  }
  const int total = k.B * k.Hkv * k.Tpad;
  for (int w = w0; w < total; w += nwarps) key_prep_row<T, D>(k, w, k.max_prefix, k.Tpad);
}

// Block commit: one warp per (block row b*C + i, KV head), the row at
// position prefix_len[b] + i written into its page.  Sliding layers: the final
// key rotate(rms(k)) and the value; global layers: the raw shared projection
// r.  Each row is computed in fp32 and stored once in T, exactly as the
// prologue stores the same rows of a canvas.
template <typename T, int D>
__global__ void __launch_bounds__(256) kv_append_kernel(KvAppendArgs p) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int total = p.B * p.C * p.Hkv;
  if (warp_global >= total) return;
  const int lane = threadIdx.x & 31;
  const int row = warp_global / p.Hkv;  // block row b*C + i
  const int hk = warp_global % p.Hkv;
  const int b = row / p.C, i = row % p.C;
  const int P = p.prefix_len[b];
  const int pos = P + i;
  if (P < 0 || pos >= p.max_prefix) {
    if (lane == 0) record_error(CANVAS_ERR_BOUNDS);
    return;
  }
  const int lp = pos / p.page_tokens;
  const int page = lp < p.max_pages ? p.block_table[(size_t)b * p.max_pages + lp] : -1;
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0) record_error(CANVAS_ERR_BOUNDS);
    return;
  }
  const size_t prow = ((size_t)page * p.Hkv + hk) * p.page_tokens + pos % p.page_tokens;
  Row r;
  load_row<float, D>(p.proj_k + (size_t)row * p.Hkv * D + (size_t)hk * D, r);
  if (p.global) {
    store_row<T, D>(static_cast<T*>(p.k_pool) + prow * D, r);
    return;
  }
  norm_rope<D>(r, p.gamma_k, p.eps, p.freq, pos);
  store_row<T, D>(static_cast<T*>(p.k_pool) + prow * D, r);
  load_row<float, D>(p.proj_v + (size_t)row * p.Hkv * D + (size_t)hk * D, r);
  store_row<T, D>(static_cast<T*>(p.v_pool) + prow * D, r);
}

// prefix_len[b] += C, after every row of the block has been written (a
// separate launch: the append kernel reads prefix_len in every warp)
__global__ void advance_prefix_kernel(int32_t* prefix_len, int B, int C) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) prefix_len[b] += C;
}

template <typename T>
cudaError_t launch_kv_append_t(const KvAppendArgs& p, int blocks, cudaStream_t stream) {
  switch (p.d) {
    case 64: kv_append_kernel<T, 64><<<blocks, 256, 0, stream>>>(p); break;
    case 128: kv_append_kernel<T, 128><<<blocks, 256, 0, stream>>>(p); break;
    case 256: kv_append_kernel<T, 256><<<blocks, 256, 0, stream>>>(p); break;
    case 512: kv_append_kernel<T, 512><<<blocks, 256, 0, stream>>>(p); break;
    case 192: kv_append_kernel<T, 192><<<blocks, 256, 0, stream>>>(p); break;
    case 320: kv_append_kernel<T, 320><<<blocks, 256, 0, stream>>>(p); break;
    case 384: kv_append_kernel<T, 384><<<blocks, 256, 0, stream>>>(p); break;
    case 448: kv_append_kernel<T, 448><<<blocks, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prologue_t(const PrologueArgs& p, int blocks, cudaStream_t stream) {
  if (sizeof(T) == 2 && (p.d & (p.d - 1)) != 0) return cudaErrorInvalidValue;
  switch (p.d) {
    case 64: prologue_kernel<T, 64><<<blocks, 256, 0, stream>>>(p); break;
    case 128: prologue_kernel<T, 128><<<blocks, 256, 0, stream>>>(p); break;
    case 256: prologue_kernel<T, 256><<<blocks, 256, 0, stream>>>(p); break;
    case 512: prologue_kernel<T, 512><<<blocks, 256, 0, stream>>>(p); break;
    case 192: prologue_kernel<T, 192><<<blocks, 256, 0, stream>>>(p); break;
    case 320: prologue_kernel<T, 320><<<blocks, 256, 0, stream>>>(p); break;
    case 384: prologue_kernel<T, 384><<<blocks, 256, 0, stream>>>(p); break;
    case 448: prologue_kernel<T, 448><<<blocks, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// grid-stride launch: as many 256-thread blocks as fit on the 148 SMs at once
template <typename T, int D>
cudaError_t launch_key_prep_d(const KeyPrepArgs& k, long long blocks_needed, cudaStream_t stream) {
  static int per_sm = 0;
  if (per_sm == 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, key_prep_kernel<T, D>, 256, 0);
    if (e != cudaSuccess) return e;
    per_sm = std::max(per_sm, 1);
  }
  const int blocks = int(std::max(1LL, std::min<long long>(blocks_needed, 148LL * per_sm)));
  key_prep_kernel<T, D><<<blocks, 256, 0, stream>>>(k);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_key_prep_t(const KeyPrepArgs& k, long long blocks, cudaStream_t stream) {
  if (sizeof(T) == 2 && (k.d & (k.d - 1)) != 0) return cudaErrorInvalidValue;
  switch (k.d) {
    case 64: return launch_key_prep_d<T, 64>(k, blocks, stream);
    case 128: return launch_key_prep_d<T, 128>(k, blocks, stream);
    case 256: return launch_key_prep_d<T, 256>(k, blocks, stream);
    case 512: return launch_key_prep_d<T, 512>(k, blocks, stream);
    case 192: return launch_key_prep_d<T, 192>(k, blocks, stream);
    case 320: return launch_key_prep_d<T, 320>(k, blocks, stream);
    case 384: return launch_key_prep_d<T, 384>(k, blocks, stream);
    case 448: return launch_key_prep_d<T, 448>(k, blocks, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& p, bool bf16, cudaStream_t stream) {
  if (bf16 && (p.d & (p.d - 1)) != 0) return cudaErrorInvalidValue;
  const long long warps = (long long)p.B * p.C * p.Hkv;
  const int blocks = int((warps * 32 + 255) / 256);
  cudaError_t e = bf16 ? launch_kv_append_t<__nv_bfloat16>(p, blocks, stream) : launch_kv_append_t<float>(p, blocks, stream);
  count_launches(1);
  if (e != cudaSuccess) return e;
  advance_prefix_kernel<<<(p.B + 127) / 128, 128, 0, stream>>>(p.prefix_len, p.B, p.C);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_prologue(const PrologueArgs& p, bool bf16, cudaStream_t stream) {
  const int heads = p.Hq + p.Hkv + (p.global ? 0 : p.Hkv);
  const long long warps = (long long)p.B * p.C * heads;
  const int blocks = int((warps * 32 + 255) / 256);
  count_launches(1);
  return bf16 ? launch_prologue_t<__nv_bfloat16>(p, blocks, stream) : launch_prologue_t<float>(p, blocks, stream);
}

cudaError_t launch_key_prep(const KeyPrepArgs& k, bool bf16, cudaStream_t stream) {
  const int rows = (k.global ? (k.max_prefix + 3) / 4 : 0) + k.Tpad;
  const long long warps = (long long)k.B * k.Hkv * rows;
  const long long blocks = (warps * 32 + 255) / 256;
  count_launches(1);
  return bf16 ? launch_key_prep_t<__nv_bfloat16>(k, blocks, stream) : launch_key_prep_t<float>(k, blocks, stream);
}

}  // namespace canvas

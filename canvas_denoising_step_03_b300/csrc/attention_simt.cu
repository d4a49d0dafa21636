// attention_simt.cu -- decode-mode canvas attention on CUDA cores (fp32 math).
//
// The fp32 variant of the step runs here.  One CTA per (sequence b, KV head,
// canvas row i): its G warps are the G query heads that share the KV head
// (GQA), and all of them see the same key set -- the visible prefix keys of
// row i (sliding window or whole prefix) followed by all C canvas keys, i.e.
// the contiguous position range [lo, P + C).  Positions below P64 come from
// the committed prefix in place (paged cache, or the prepared global keys),
// positions from P64 on from the dense tail buffers (kernels.h).  Keys and
// values are staged in shared memory 32 (or 16) rows at a time; each warp
// keeps an online softmax (lane = key for scores, lane = channel for the
// output).
//
// Method: AI Trends summary of a DiffusionGemma 26B notebook
// (aitrends.kr/articles/94089), "섹션별 상세", decode mode (the canvas attends
// bidirectionally to the committed prefix in the KV cache and to the whole
// canvas) and the glossary entry on sliding-window attention.
#include "common.cuh"
#include "kernels.h"

namespace canvas {

namespace {

template <typename T>
__device__ __forceinline__ const T* page_row(const AttnArgs& a, const void* pool, int b, int hk, int j) {
  const int lp = j / a.page_tokens, off = j % a.page_tokens;
  const int page = (lp < a.max_pages) ? a.block_table[(size_t)b * a.max_pages + lp] : -1;
  if (page < 0 || page >= a.num_pages) return nullptr;
  return static_cast<const T*>(pool) + (((size_t)page * a.Hkv + hk) * a.page_tokens + off) * a.d;
}

template <typename T, int KB>
__global__ void __launch_bounds__(1024) attention_simt_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  const int d = a.d, G = a.Hq / a.Hkv;
  const int i = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x;
  float* sK = sm;                       // [KB][d + 1]
  float* sV = sK + KB * (d + 1);        // [KB][d]
  float* sQ = sV + KB * d;              // [G][d]

  const int P = a.prefix_len[b];
  if (P < 0 || P > a.max_prefix) return;  // reported by the key-prep kernel
  const int P64 = P & ~63;
  const int lo = (a.global || a.window <= 0) ? 0 : max(0, P + i - a.window);
  const int n_keys = (a.causal ? P + i + 1 : P + a.C) - lo;  // encode mode: canvas keys 0..i
  const size_t grp = (size_t)b * a.Hkv + hk;

  // this warp's query row
  const T* q = static_cast<const T*>(a.Qp) + (((grp * G + warp) * a.C) + i) * d;
  for (int t = lane; t < d; t += 32) sQ[warp * d + t] = to_f32(q[t]);

  const int per = d / 32;  // channels per lane (d <= 512)
  float o[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) o[k] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int k0 = 0; k0 < n_keys; k0 += KB) {
    __syncthreads();
    const int nk = min(KB, n_keys - k0);
    // stage KB keys / values as fp32
    for (int e = threadIdx.x; e < KB * d; e += nthr) {
      const int r = e / d, t = e % d;
      float kv = 0.f, vv = 0.f;
      if (r < nk) {
        const int pos = lo + k0 + r;
        const T *kr, *vr;
        float vsc = 1.f;
        if (pos < P64) {
          kr = a.global ? static_cast<const T*>(a.k_pre) + (grp * a.max_prefix + pos) * d
                        : page_row<T>(a, a.k_pre, b, hk, pos);
          vr = page_row<T>(a, a.v_pre, b, hk, pos);
          if (a.v_unit_rms) vsc = a.vs_pre[grp * a.max_prefix + pos];
        } else {
          const size_t trow = grp * a.Tpad + (pos - P64);
          kr = static_cast<const T*>(a.Kx) + trow * d;
          vr = static_cast<const T*>(a.Vx) + trow * d;
          if (a.v_unit_rms) vsc = a.vs_tail[trow];
        }
        if (kr != nullptr && vr != nullptr) {  // a bad page id is reported by the key-prep kernel
          kv = to_f32(kr[t]);
          vv = to_f32(vr[t]) * vsc;
        }
      }
      sK[r * (d + 1) + t] = kv;
      sV[r * d + t] = vv;
    }
    __syncthreads();
    // scores: lane = key
    for (int base = 0; base < nk; base += 32) {
      const int r = base + lane;
      float s = -INFINITY;
      if (r < nk) {
        float acc = 0.f;
        const float* kr = sK + r * (d + 1);
        const float* qr = sQ + warp * d;
        for (int t = 0; t < d; ++t) acc = fmaf(qr[t], kr[t], acc);
        s = acc * a.scale;
      }
      float bm = s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      const float mn = fmaxf(m, bm);
      const float alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
      const float p = (r < nk) ? expf(s - mn) : 0.f;
      float ps = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l = l * alpha + ps;
      m = mn;
#pragma unroll
      for (int k = 0; k < 16; ++k) o[k] *= alpha;
      const int cnt = min(32, nk - base);
      for (int jj = 0; jj < cnt; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const float* vr = sV + (base + jj) * d;
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if (k < per) o[k] = fmaf(pj, vr[lane + 32 * k], o[k]);
      }
    }
  }
  const float inv = 1.f / l;
  const int h = hk * G + warp;
  T* out = static_cast<T*>(a.out) + ((size_t)b * a.C + i) * a.Hq * d + (size_t)h * d;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    if (k < per) {
      const float v = o[k] * inv;
      if constexpr (sizeof(T) == 4)
        out[lane + 32 * k] = v;
      else
        out[lane + 32 * k] = __float2bfloat16_rn(v);
    }
  }
  if (a.lse != nullptr && lane == 0) a.lse[((size_t)b * a.C + i) * a.Hq + h] = m + logf(l);
}

template <typename T, int KB>
cudaError_t launch_kb(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  const size_t smem = sizeof(float) * (size_t(KB) * (a.d + 1) + size_t(KB) * a.d + size_t(G) * a.d);
  cudaError_t e = cudaFuncSetAttribute(attention_simt_kernel<T, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.C, a.Hkv, a.B);
  attention_simt_kernel<T, KB><<<grid, 32 * G, smem, stream>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_simt(const AttnArgs& a, bool bf16, cudaStream_t stream) {
  if (a.d > 256) return bf16 ? launch_kb<__nv_bfloat16, 16>(a, stream) : launch_kb<float, 16>(a, stream);
  return bf16 ? launch_kb<__nv_bfloat16, 32>(a, stream) : launch_kb<float, 32>(a, stream);
}

}  // namespace canvas

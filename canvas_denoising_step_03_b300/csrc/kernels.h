// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace canvas {

// host-side count of kernel launches (read by canvas_kernel_launches)
void count_launches(int n);

// ----------------------------------------------------------------- sampler
constexpr int kMaxSampleCluster = 8;

struct SampleArgs {
  int rows, V, chunk, cluster;
  float inv_temp, bound;
  uint64_t seed;
  uint32_t step;
  int commit_mode, canvas_len;
  const uint8_t* frozen;
  const int32_t* frozen_tokens;
  int32_t* tokens;
  uint8_t* commit_mask;
  float* entropy;
  float* confidence;
  int32_t* argmax;
  __nv_bfloat16* probs_bf16;
  float* probs_f32;
};

cudaError_t launch_sampler(const SampleArgs& a, const void* logits, bool bf16, cudaStream_t stream);

// ----------------------------------------------------------------- GEMMs
// tcgen05 bf16 GEMM: C[M,N] (fp32) = A[M,K] * op(B)
struct GemmTcArgs {
  float* C;
  int M, N, K, ldc;
  int accumulate;
  int b_mn_major;  // 0: B is [N,K] (K contiguous); 1: B is [K,N] (N contiguous)
  int two_acc;     // 1: a CTA covers 256 rows (two 128-row accumulators)
  int m_tiles, n_tiles, splits, kblocks;
  float* partials;  // [splits][M][N] when splits > 1
  int* counters;    // [m_tiles * n_tiles], zero before the launch
};
constexpr int kGemmBM = 128, kGemmBN = 256, kGemmBK = 64, kGemmStages = 3;
size_t gemm_tc_smem_bytes();
cudaError_t launch_gemm_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmTcArgs& g,
                           cudaStream_t stream);

// SIMT GEMM (fp32 path): C[M,N] = A[M,K] * op(B) (+C), TA/TB = float or bf16
cudaError_t launch_gemm_simt(const void* A, const void* B, int b_mn_major, bool bf16, float* C, int M, int N,
                             int K, int accumulate, cudaStream_t stream);

// ----------------------------------------------------------------- attention
struct PrologueArgs {
  const float* proj_q;  // [B*C, Hq*d]
  const float* proj_k;  // [B*C, Hkv*d]
  const float* proj_v;  // [B*C, Hkv*d] or null (global)
  const float* gamma_q;
  const float* gamma_k;
  const float* freq;
  const int32_t* prefix_len;
  int B, C, Hq, Hkv, d;
  float eps;
  int global;
  void* Qp;  // [B][Hkv][G][C][d]
  void* Kc;  // sliding: [B][Hkv][C][d] final canvas keys; global: raw canvas r
  void* Vc;  // sliding: [B][Hkv][C][d] canvas values; global: unused
};
cudaError_t launch_prologue(const PrologueArgs& p, bool bf16, cudaStream_t stream);

// Global layers: per key row j of the key set (prefix then canvas), the
// rotation of the raw row and its norm scalars.
struct KeyPrepArgs {
  const void* pool;          // raw r pages [num_pages][Hkv][pt][d]
  const int32_t* block_table;
  int max_pages, page_tokens, num_pages;
  const void* Rc;            // raw canvas r [B][Hkv][C][d]
  const float* gamma_k;
  const float* freq;
  const int32_t* prefix_len;
  int B, C, Hkv, d, max_prefix;
  float eps;
  void* Kt;                  // [B][Hkv][max_prefix + C][d] rotate(r)
  float* ks;                 // [B][Hkv][max_prefix + C] gamma_k * sqrt(d) / (|r| + eps)
  float* vs;                 // [B][Hkv][max_prefix + C] sqrt(d) / (|r| + eps)
};
cudaError_t launch_key_prep(const KeyPrepArgs& k, bool bf16, cudaStream_t stream);

struct AttnArgs {
  const void* Qp;            // [B][Hkv][G][C][d]
  // sliding: prefix K/V from the pools; canvas K/V from Kc/Vc
  // global : keys from Kt (+ks), values from the pool / Rc (+vs if v_unit_rms)
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  int max_pages, page_tokens, num_pages;
  const void* Kc;
  const void* Vc;
  const void* Kt;
  const float* ks;
  const float* vs;
  const int32_t* prefix_len;
  int B, C, Hq, Hkv, d, max_prefix, window;
  int global, v_unit_rms;
  float scale;
  void* out;                 // [B][C][Hq*d]
  float* lse;                // [B][C][Hq] or null
};
cudaError_t launch_attention_simt(const AttnArgs& a, bool bf16, cudaStream_t stream);

}  // namespace canvas

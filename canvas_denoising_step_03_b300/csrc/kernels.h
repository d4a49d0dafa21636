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
// a row's CTAs: up to 8, each staging up to a 64 KB slice of the row (16 CTAs
// with 32 KB slices measured slower: 75.8 against 63.5 us on 256 x 262144)
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
  // deferred normalisation (launch_sampler_slices): the vocabulary ranges
  // are the soft-embedding GEMM's K splits (kb_per or kb_per + 1 blocks of 64)
  int slices, kb_per, kb_rem;
  float* slice_state;  // [rows][slices][8]: m, Z, T, best logit, argmax (int bits)
};

// Largest vocabulary range one sampler CTA stages in shared memory (entries),
// and the most ranges per row of the deferred path.
constexpr int kSampleSliceMaxElems = 32768;
constexpr int kMaxSampleSlices = 148;

cudaError_t launch_sampler(const SampleArgs& a, const void* logits, bool bf16, cudaStream_t stream);
// deferred path: per-range states and p~ (bf16 logits), then, after the
// GEMM of p~ and E, the row outputs / decisions and the scaled split sum
cudaError_t launch_sampler_slices(const SampleArgs& a, const void* logits, cudaStream_t stream);
cudaError_t launch_soft_reduce(const SampleArgs& a, const float* partials, float* soft, int D, cudaStream_t stream);

// ----------------------------------------------------------------- GEMMs
// tcgen05 bf16 GEMM, up to three problems sharing A and K (the q / k / v
// projections of one x): C_p[M,N_p] = A[M,K] * op(B_p), fp32 (or bf16) out.
constexpr int kGemmMaxProblems = 3;
struct GemmTcArgs {
  int M, K, kblocks, splits;
  int accumulate;  // C += (one problem)
  int out_bf16;    // C holds bf16 (no accumulate)
  int b_mn_major;  // 0: B is [N,K] (K contiguous); 1: B is [K,N] (N contiguous)
  int two_acc;     // 1: a CTA covers 256 rows (two 128-row accumulators)
  int m_tiles, nprob;
  int bm;                    // rows per M tile: 256 (two accumulators when M > 128) or 128 (grouped)
  // grouped mode (non-null): M tile t belongs to group group_of_mtile[t] (-1:
  // no work), whose B rows are group * N_p .. of a [groups * N_p, K] B; the
  // rows of A are laid out so that no tile straddles two groups
  const int* group_of_mtile;
  int tile0[kGemmMaxProblems + 1];  // first 256-column tile of each problem; tile0[nprob] = all tiles
  int N[kGemmMaxProblems];
  void* C[kGemmMaxProblems];
  float* partials[kGemmMaxProblems];  // [splits][M][N_p] when splits > 1, summed by a reduce kernel
};
// A (K-major bf16), B of each problem, and the TMA store target of each
// problem (C, or the split partials)
struct GemmTcMaps {
  CUtensorMap A;
  CUtensorMap B[kGemmMaxProblems];
  CUtensorMap out[kGemmMaxProblems];
};
constexpr int kGemmBM = 128, kGemmBN = 256, kGemmBK = 64, kGemmStages = 3;
size_t gemm_tc_smem_bytes();
// reduce = false leaves a split product in its partials (g.partials[p],
// [splits][M][N_p]) for a consumer that sums them in split order itself
cudaError_t launch_gemm_tc(const GemmTcMaps& maps, const GemmTcArgs& g, cudaStream_t stream, bool reduce = true);

// SIMT GEMM (fp32 path): C[M,N] = A[M,K] * op(B) (+C), TA/TB = float or bf16
cudaError_t launch_gemm_simt(const void* A, const void* B, int b_mn_major, bool bf16, float* C, int M, int N,
                             int K, int accumulate, cudaStream_t stream);

// ----------------------------------------------------------------- attention
//
// Key sequence of one (sequence b, KV head).  Canvas row i sits at absolute
// position P + i (P = prefix_len[b]); P64 = P rounded down to a multiple of 64.
//   positions [0, P64)        committed prefix, read in place: the paged cache
//                             (sliding layers, and values of global layers) or
//                             the prepared key buffer Kt (global-layer keys);
//   positions [P64, P + C)    the "tail": the last P - P64 prefix rows followed
//                             by the C canvas rows, gathered into the dense
//                             buffers Kx / Vx [B][Hkv][Tpad][d] (row t holds
//                             position P64 + t; rows past P + C are zero).
// Every 64-key sub-block is therefore either whole in the paged / prepared
// prefix or whole in the tail buffers, and no tile ever reads a cache slot
// that holds no token.

// Tail rows: 64 * (ceil((C + 63) / 64) + 1), so a 128-key block that starts
// inside the tail never reads past the buffer.
inline int attn_tail_rows(int C) { return 64 * ((C + 63 + 63) / 64 + 1); }

struct PrologueArgs {
  // the projections, or (splits > 1) the split-K partials of each: slice s
  // of proj_x at proj_x + s * (B*C*N_x), summed in split order (s = 0, 1,
  // ...) from 0 exactly as the GEMM's own reduce would
  const float* proj_q;  // [B*C, Hq*d]
  const float* proj_k;  // [B*C, Hkv*d]
  const float* proj_v;  // [B*C, Hkv*d] or null (global)
  int splits;
  const float* gamma_q;
  const float* gamma_k;
  const float* freq;
  const int32_t* prefix_len;
  int B, C, Hq, Hkv, d, Tpad;
  float eps;
  int global;
  void* Qp;  // [B][Hkv][G][C][d]
  void* Kx;  // [B][Hkv][Tpad][d] keys of the tail rows
  void* Vx;  // [B][Hkv][Tpad][d] values of the tail rows (global: raw r)
  float* vs_tail;  // [B][Hkv][Tpad] global: sqrt(d) / (|r| + eps) of each tail row
};
cudaError_t launch_prologue(const PrologueArgs& p, bool bf16, cudaStream_t stream);

// Global-layer prefix keys Kt[j] = rotate(rms(r_j)) for j < P64, and the tail
// rows [P64, P) of both layer types (copied, or prepared from raw r), and the
// zero rows past the canvas.
struct KeyPrepArgs {
  const void* k_pool;        // [num_pages][Hkv][pt][d]: keys (sliding) / raw r (global)
  const void* v_pool;        // values (sliding) or null
  const int32_t* block_table;
  int max_pages, page_tokens, num_pages;
  const float* gamma_k;
  const float* freq;
  const int32_t* prefix_len;
  int B, C, Hkv, d, max_prefix, Tpad;
  float eps;
  int global;
  void* Kt;                  // [B][Hkv][max_prefix][d] (global)
  float* vs_pre;             // [B][Hkv][max_prefix] (global)
  void* Kx;
  void* Vx;
  float* vs_tail;
};
cudaError_t launch_key_prep(const KeyPrepArgs& k, bool bf16, cudaStream_t stream);

// Block commit: the rows of a committed block written into the paged cache
// at positions prefix_len[b] + i, then prefix_len[b] += C.
struct KvAppendArgs {
  const float* proj_k;       // [B*C, Hkv*d] x W_k^T
  const float* proj_v;       // [B*C, Hkv*d] x W_v^T (sliding) or null
  const float* gamma_k;
  const float* freq;
  int32_t* prefix_len;       // [B], advanced by C
  void* k_pool;              // [num_pages][Hkv][page_tokens][d]: final keys (sliding) / raw r (global)
  void* v_pool;              // values (sliding) or null
  const int32_t* block_table;
  int max_pages, page_tokens, num_pages;
  int B, C, Hkv, d, max_prefix;  // max_prefix: positions must stay below it
  float eps;
  int global;
};
cudaError_t launch_kv_append(const KvAppendArgs& p, bool bf16, cudaStream_t stream);

// CUDA-core attention (fp32 calls)
struct AttnArgs {
  const void* Qp;            // [B][Hkv][G][C][d]
  const void* k_pre;         // sliding: k pool (paged); global: Kt (dense)
  const void* v_pre;         // paged pool: values (sliding) / raw r (global)
  const int32_t* block_table;
  int max_pages, page_tokens, num_pages;
  const void* Kx;
  const void* Vx;
  const float* vs_pre;       // global + v_unit_rms: per-row value scale
  const float* vs_tail;
  const int32_t* prefix_len;
  int B, C, Hq, Hkv, d, max_prefix, window, Tpad;
  int global, v_unit_rms;
  int causal;                // 1: encode mode, canvas row i sees canvas keys 0..i
  float scale;
  void* out;                 // [B][C][Hq*d]
  float* lse;                // [B][C][Hq] or null
};
cudaError_t launch_attention_simt(const AttnArgs& a, bool bf16, cudaStream_t stream);

// tcgen05 attention (bf16 calls, d in {64, 128, 256, 512})
constexpr int kAttnBM = 128;       // query rows per tile (TMEM lanes)
constexpr int kAttnBN = 128;       // keys per block
struct AttnTcArgs {
  int B, C, Hq, Hkv, G, d, DV, dv_parts, q_tiles, nsplit, max_prefix, window, Tpad;
  int kpre_paged;            // 1: prefix keys from the paged pool; 0: dense Kt
  int causal;                // 1: encode mode, canvas row i sees canvas keys 0..i
  int pair;                  // 2: 4-SM kernel (two CTA pairs split the key blocks), head_dim 512;
                             // 0: one SM per 128-row tile
  const __nv_bfloat16* Qp;   // [B][Hkv][G][C][d] prepared queries (the 4-SM kernel reads half of each row)
  const int32_t* block_table;
  int max_pages, page_tokens, num_pages;
  const int32_t* prefix_len;
  const float* vs_pre;       // non-null: scale each key's softmax weight (unit-RMS values)
  const float* vs_tail;
  float c_log2;              // scale * log2(e)
  __nv_bfloat16* out;        // [B][C][Hq*d] (nsplit == 1)
  float* lse;                // [B][C][Hq] or null (nsplit == 1)
  float* part_o;             // [nsplit][B*Hkv][q_tiles*128][d] (nsplit > 1)
  float* part_ml;            // [nsplit][B*Hkv][q_tiles*128][2]
};
struct AttnTcMaps {
  CUtensorMap q, kpre, vpre, kx, vx;
  // 3D views [64-column chunk][row][64] of the same tensors, so one copy
  // brings a key box of 32 rows x all eight chunks (4-SM kernel), or a value
  // box of 64 rows x two chunks (4-SM kernel) / x all d / 64 chunks (one-SM
  // kernel)
  CUtensorMap kpre_c, kx_c, vpre_c, vx_c;
};
size_t attention_tc_smem_bytes(int d);
cudaError_t launch_attention_tc(const AttnTcMaps& maps, const AttnTcArgs& a, cudaStream_t stream);
cudaError_t launch_attention_combine(const AttnTcArgs& a, cudaStream_t stream);

// ----------------------------------------------------------------- mixture of experts
struct MoeArgs {
  int R, D, E, k, max_tiles;
  const float* scores;         // [R, E] router scores x . router_e
  const float* expert_scale;   // [E] or null (1)
  int32_t* topk_idx;           // [R, k] chosen experts, largest score first
  float* topk_w;               // [R, k] their weights
  int32_t* counts;             // [E] tokens per expert
  int32_t* offsets;            // [E + 1] first row of each expert in the grouped layout
  int32_t* cursor;             // [E] fill positions
  int32_t* group_of_mtile;     // [max_tiles] expert of each 128-row tile, -1 past the end
  int32_t* slot;               // [R, k] row of each (token, choice) in the grouped layout
  const void* x;               // [R, D] bf16 input
  void* xg;                    // [max_tiles * 128, D] bf16 rows grouped by expert
  const float* yg;             // [max_tiles * 128, D] expert outputs (grouped rows)
  const float* ys;             // [R, D] shared expert output or null
  float* out;                  // [R, D]
};
cudaError_t launch_moe_route(const MoeArgs& a, cudaStream_t stream);  // route, offsets, scatter
cudaError_t launch_moe_act(const float* gate, const float* up, void* act, long long n, cudaStream_t stream);
cudaError_t launch_moe_combine(const MoeArgs& a, cudaStream_t stream);

// ----------------------------------------------------------------- loop glue
cudaError_t launch_embed_input(const int32_t* tokens, const void* E, const float* soft, int rows, int D, int V,
                               void* x, float* x32, cudaStream_t stream);
cudaError_t launch_cast_bf16(const float* in, void* out, long long n, cudaStream_t stream);
cudaError_t launch_gelu_bf16(const float* in, void* out, long long n, cudaStream_t stream);
cudaError_t launch_count_committed(const uint8_t* mask, int n_canvas, int canvas_len, int32_t* counts,
                                   cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(cudaStream_t stream);

}  // namespace canvas

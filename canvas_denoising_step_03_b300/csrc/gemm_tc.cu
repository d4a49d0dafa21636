// gemm_tc.cu -- bf16 GEMM on the 5th-generation tensor cores (tcgen05).
//
//   C[M,N] (fp32) = A[M,K] * op(B),   A row-major (K contiguous),
//   B either [N,K] (K contiguous, "weights": C = A B^T, the pages' x @ W.T) or
//   [K,N] (N contiguous: the embedding table in the soft embedding P.E).
//
// Used for the QKV projection of the attention layer and the soft embedding
// P.E of the sampler (self-conditioning, AI Trends summary of a DiffusionGemma
// 26B notebook, aitrends.kr/articles/94089, glossary entry "자기 조건화").
//
// Up to three problems that share A and K (the q / k / v projections of one
// x) run in one launch: the grid's x dimension walks the 256-column tiles of
// problem 0, then 1, then 2.
//
// Design (one CTA per 256 x 256 output tile and K-split):
//   warp 0      TMA producer: A (two 128-row boxes) and B tiles of 64 K
//               elements, 128-byte swizzle, into a 3-stage ring;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators) and issues tcgen05.mma (M=128, N=256, K=16)
//               from one thread; tcgen05.commit frees each stage;
//   warps 2..5  epilogue: tcgen05.ld of the accumulators (each warp reads the
//               32 TMEM lanes of its quadrant), 32 x 32 fp32 boxes staged in
//               the idle ring (128-byte swizzle, two boxes per warp) and
//               written by TMA stores -- coalesced whole rows, clipped at the
//               edges of C; bf16 output packs 64 columns per box (rounded to
//               nearest even); accumulating into C (one split) adds in place.
// K is split across CTAs when the tile grid alone cannot fill the 148 SMs;
// each split writes its fp32 partial tile to the workspace and a separate
// reduce kernel sums the splits in order (so the result does not depend on
// timing), spread over the whole GPU.
// Every mbarrier wait is bounded (common.cuh): on timeout the CTA records
// CANVAS_ERR_TIMEOUT, drains and returns.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace canvas {

namespace {
constexpr int kThreads = 192;
constexpr int kABoxBytes = kGemmBM * kGemmBK * 2;          // 16 KB: 128 rows x 128 B
constexpr int kAStageBytes = 2 * kABoxBytes;                // 32 KB
constexpr int kBStageBytes = kGemmBN * kGemmBK * 2;         // 32 KB
constexpr int kTileBytes = kGemmStages * (kAStageBytes + kBStageBytes);
constexpr int kTmemCols = 512;
}  // namespace

size_t gemm_tc_smem_bytes() { return size_t(kTileBytes) + 1024 /*align*/ + 256 /*barriers*/; }

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ GemmTcMaps maps, const __grid_constant__ GemmTcArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kGemmStages * kAStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTileBytes);
  uint64_t* empty = full + kGemmStages;
  uint64_t* tmem_full = empty + kGemmStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.y, split = blockIdx.z;
  // grouped mode: this tile's group selects the B rows (uniform over the CTA,
  // decided before any barrier or TMEM allocation)
  int group = 0;
  if (g.group_of_mtile != nullptr) {
    group = g.group_of_mtile[mt];
    if (group < 0) return;
  }
  // problem of this tile (selects, not indexed loads, so the arguments stay in constant memory)
  const int prob = (g.nprob > 1 && int(blockIdx.x) >= g.tile0[1]) + (g.nprob > 2 && int(blockIdx.x) >= g.tile0[2]);
  const int nt = int(blockIdx.x) - (prob == 0 ? 0 : prob == 1 ? g.tile0[1] : g.tile0[2]);
  const int N = prob == 0 ? g.N[0] : prob == 1 ? g.N[1] : g.N[2];
  const CUtensorMap* tmA = &maps.A;
  const CUtensorMap* tmB = prob == 0 ? &maps.B[0] : prob == 1 ? &maps.B[1] : &maps.B[2];
  const CUtensorMap* tmC = prob == 0 ? &maps.out[0] : prob == 1 ? &maps.out[1] : &maps.out[2];
  float* Cf = static_cast<float*>(prob == 0 ? g.C[0] : prob == 1 ? g.C[1] : g.C[2]);
  const int kb_per = g.kblocks / g.splits, kb_rem = g.kblocks % g.splits;
  const int kb0 = split * kb_per + min(split, kb_rem);
  const int nkb = kb_per + (split < kb_rem ? 1 : 0);
  const int nacc = g.two_acc ? 2 : 1;
  const int brow0 = group * N;  // first B row of this tile's group (0 unless grouped)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    flags[0] = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(tmA);
    tma_prefetch_desc(tmB);
    tma_prefetch_desc(tmC);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint32_t bytes = uint32_t(nacc * kABoxBytes + kBStageBytes);
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kGemmStages;
        const uint32_t ph = (i / kGemmStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, flags)) break;
        issued = i + 1;
        const int kx = (kb0 + i) * kGemmBK;
        mbar_arrive_expect_tx(&full[s], bytes);
        uint8_t* a = sA + s * kAStageBytes;
        tma_load_2d(a, tmA, &full[s], kx, mt * g.bm);
        if (nacc == 2) tma_load_2d(a + kABoxBytes, tmA, &full[s], kx, mt * g.bm + 128);
        uint8_t* b = sB + s * kBStageBytes;
        if (!g.b_mn_major) {
          tma_load_2d(b, tmB, &full[s], kx, brow0 + nt * kGemmBN);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tma_load_2d(b + c * 8192, tmB, &full[s], nt * kGemmBN + 64 * c, kx);
        }
      }
      // drain: every TMA this thread issued has landed before the CTA can exit
      // (matters only after an abort; otherwise these phases are complete)
      volatile int no_abort = 0;
      for (int i = max(0, issued - kGemmStages); i < issued; ++i) {
        const int s = i % kGemmStages;
        mbar_wait(&full[s], (i / kGemmStages) & 1, &no_abort);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(128, 256, 0, g.b_mn_major);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kGemmStages;
        const uint32_t ph = (i / kGemmStages) & 1;
        if (!mbar_wait(&full[s], ph, flags)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(sA + s * kAStageBytes);
        const uint32_t b_base = smem_u32(sB + s * kBStageBytes);
#pragma unroll
        for (int kk = 0; kk < kGemmBK / 16; ++kk) {
          // K-major B: 16 elements = 32 bytes along the swizzled row.
          // MN-major B: 16 K-rows = 2 groups of 8 rows x 128 B; N chunks of
          // 64 elements sit 8 KB apart (leading byte offset).
          const uint64_t bdesc = g.b_mn_major ? smem_desc_sw128(b_base + kk * 2048, 8192, 1024)
                                              : smem_desc_sw128(b_base + kk * 32, 16, 1024);
          for (int acc = 0; acc < nacc; ++acc) {
            const uint64_t adesc = smem_desc_sw128(a_base + acc * kABoxBytes + kk * 32, 16, 1024);
            mma_bf16_ss(tmem + acc * 256, adesc, bdesc, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
      }
      mma_commit(tmem_full);
    }
  } else {
    // ---------------- epilogue: warps 2..5, quadrant = warp % 4
    const int q = warp & 3;
    mbar_wait(tmem_full, 0, flags);
    tc_fence_after();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const bool ok = flags[0] == 0;  // uniform across the epilogue warps
    const bool add = g.splits == 1 && g.accumulate != 0;
    const bool pack = g.splits == 1 && g.out_bf16 != 0;  // bf16 boxes of 64 columns
    if (ok && !add) {
      // every MMA has completed, so the ring is idle: two 4 KB boxes per warp
      uint8_t* stage = smem + (warp - 2) * 8192;
      const int z = g.splits > 1 ? split : 0;
      const int step = pack ? 2 : 1;  // 32-column TMEM chunks per box
      int nbox = 0;
      for (int acc = 0; acc < nacc; ++acc) {
        const int row0 = mt * g.bm + acc * 128 + q * 32;
        if (row0 >= g.M) break;  // uniform in the warp
        for (int cc = 0; cc < kGemmBN / 32; cc += step) {
          const int col0 = nt * kGemmBN + cc * 32;
          if (col0 >= N) break;
          uint32_t w[32];  // one 128-byte row of the box
          {
            uint32_t r[32];
            tmem_ld32(tmem + uint32_t(acc * 256 + cc * 32) + (uint32_t(q * 32) << 16), r);
            tmem_ld_wait();
            if (!pack) {
#pragma unroll
              for (int j = 0; j < 32; ++j) w[j] = r[j];
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
              tmem_ld32(tmem + uint32_t(acc * 256 + cc * 32 + 32) + (uint32_t(q * 32) << 16), r);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j)
                w[16 + j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            }
          }
          uint8_t* box = stage + (nbox & 1) * 4096;
          if (nbox >= 2) {
            if (lane == 0) bulk_wait_group_read<1>();  // the store of two boxes ago has read this one
            __syncwarp();
          }
          // row `lane` of the box; 128-byte swizzle: 16-byte chunk j sits at j ^ (row & 7)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(box + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(tmC, box, col0, row0, z);
            bulk_commit_group();
          }
          ++nbox;
        }
      }
      if (lane == 0) bulk_wait_group_all();
      __syncwarp();
    } else if (ok) {
      // C += A op(B) with a single split: read-modify-write of whole rows
      for (int acc = 0; acc < nacc; ++acc) {
        const int row = mt * g.bm + acc * 128 + q * 32 + lane;
        for (int cc = 0; cc < kGemmBN / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + uint32_t(acc * 256 + cc * 32) + (uint32_t(q * 32) << 16), r);
          tmem_ld_wait();
          const int col0 = nt * kGemmBN + cc * 32;
          if (row >= g.M || col0 >= N) continue;
          float* dst = Cf + (size_t)row * N + col0;
          const int ncol = min(32, N - col0);
          if (ncol == 32) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4* p = reinterpret_cast<float4*>(dst + j);
              const float4 o = *p;
              *p = make_float4(o.x + __uint_as_float(r[j]), o.y + __uint_as_float(r[j + 1]),
                               o.z + __uint_as_float(r[j + 2]), o.w + __uint_as_float(r[j + 3]));
            }
          } else {
            for (int j = 0; j < ncol; ++j) dst[j] += __uint_as_float(r[j]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// C[m][n] = (accumulate ? C : 0) + sum over splits s (in order) of partials[s][m][n],
// stored as fp32 or (out_bf16) rounded to bf16.  Each thread issues the loads
// of up to eight splits before adding them, so the partials stream with that
// many requests in flight per element.
__global__ void __launch_bounds__(256) gemm_split_reduce_kernel(const float4* __restrict__ partials, void* C,
                                                                 long long n4, int splits, int accumulate,
                                                                 int out_bf16) {
  for (long long e = blockIdx.x * 256LL + threadIdx.x; e < n4; e += (long long)gridDim.x * 256) {
    float4 s4 = accumulate ? static_cast<float4*>(C)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < splits; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < splits) v[j] = __ldcs(partials + (s0 + j) * n4 + e);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < splits) {
          s4.x += v[j].x;
          s4.y += v[j].y;
          s4.z += v[j].z;
          s4.w += v[j].w;
        }
    }
    if (out_bf16)
      static_cast<uint2*>(C)[e] = make_uint2(pack_bf16x2(s4.x, s4.y), pack_bf16x2(s4.z, s4.w));
    else
      static_cast<float4*>(C)[e] = s4;
  }
}

cudaError_t launch_gemm_tc(const GemmTcMaps& maps, const GemmTcArgs& g, cudaStream_t stream, bool reduce) {
  static bool attr_set = false;  // per process; the attribute is per function
  const size_t smem = gemm_tc_smem_bytes();
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(g.tile0[g.nprob], g.m_tiles, g.splits);
  gemm_bf16_tc_kernel<<<grid, kThreads, smem, stream>>>(maps, g);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || g.splits == 1 || !reduce) return e;
  for (int p = 0; p < g.nprob; ++p) {
    const long long n4 = (long long)g.M * g.N[p] / 4;  // N % 8 == 0
    const int blocks = int(std::min<long long>((n4 + 255) / 256, 148LL * 8));
    gemm_split_reduce_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(g.partials[p]), g.C[p], n4,
                                                         g.splits, g.accumulate, g.out_bf16);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace canvas

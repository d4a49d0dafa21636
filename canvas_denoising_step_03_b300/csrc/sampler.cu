// sampler.cu -- the per-position vocab sampler of a denoising step.
//
// One thread-block cluster per canvas position (row).  Each CTA of the
// cluster owns a contiguous slice of the vocabulary and reduces it to a
// (max, sum, entropy-sum) state plus the argmax; the CTAs swap their partial
// states through distributed shared memory and every CTA merges them in rank
// order (so all agree bit for bit).  CTA 0 then writes the row's entropy /
// confidence / argmax and the commit-or-renoise decision; every CTA writes
// the probabilities of its slice.  bf16 logits with slices up to 64 KB: the
// slice is staged in shared memory by bulk copies, so the logits are read
// from HBM exactly once (sample_rows_smem_kernel).  Otherwise (fp32 logits,
// larger slices) the slice is streamed from global memory twice, with an
// online state (sample_rows_kernel).
//
// Method: AI Trends summary of a DiffusionGemma 26B notebook
// (aitrends.kr/articles/94089), "섹션별 상세", sampling-loop paragraph (entropy
// per position, low-entropy positions fixed, others renoised to uniform random
// tokens); aibars news on DiffusionGemma, "블록 자동 회귀 노이즈 제거 및 자체 수정"
// (low-confidence tokens replaced by random tokens).
#include "common.cuh"
#include "kernels.h"

#include <cstring>

namespace canvas {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Online softmax state in base 2: Z = sum 2^(y - m), T = sum (y - m) 2^(y - m).
struct RowState {
  float m, Z, T;
  float bx;  // best raw logit
  int bi;    // its (lowest) index
};

__device__ __forceinline__ void state_init(RowState& s) {
  s.m = -INFINITY;
  s.Z = 0.f;
  s.T = 0.f;
  s.bx = -INFINITY;
  s.bi = 0x7fffffff;
}

// Merge b into a (associative up to rounding; used in a fixed order).
__device__ __forceinline__ void state_merge(RowState& a, const RowState& b) {
  if (b.bx > a.bx || (b.bx == a.bx && b.bi < a.bi)) {
    a.bx = b.bx;
    a.bi = b.bi;
  }
  if (b.Z == 0.f) return;
  if (a.Z == 0.f) {
    a.m = b.m;
    a.Z = b.Z;
    a.T = b.T;
    return;
  }
  const float M = fmaxf(a.m, b.m);
  const float da = a.m - M, db = b.m - M;
  const float sa = ex2_approx(da), sb = ex2_approx(db);
  a.T = sa * (a.T + da * a.Z) + sb * (b.T + db * b.Z);
  a.Z = sa * a.Z + sb * b.Z;
  a.m = M;
}

// Fold a group of 8 raw logits x[] (indices idx0 .. idx0+7, increasing within
// a thread) into s; y = x * ysc is the base-2 scaled logit.  The argmax and
// the running maximum are updated from the group maximum, so the per-element
// work is one max, one fused multiply-add, one exponential and two sums.
__device__ __forceinline__ void state_add8(RowState& s, const float (&x)[8], float ysc, int idx0) {
  float xm = x[0];
#pragma unroll
  for (int j = 1; j < 8; ++j) xm = fmaxf(xm, x[j]);
  if (xm > s.bx) {  // strict: an earlier (lower) index keeps a tie
    int jm = 7;
#pragma unroll
    for (int j = 6; j >= 0; --j)
      if (x[j] == xm) jm = j;
    s.bx = xm;
    s.bi = idx0 + jm;
  }
  const float vmax = xm * ysc;
  if (vmax > s.m) {
    if (s.Z != 0.f) {
      const float dm = s.m - vmax;
      const float sc = ex2_approx(dm);
      s.T = sc * (s.T + dm * s.Z);
      s.Z *= sc;
    }
    s.m = vmax;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float t = fmaf(x[j], ysc, -s.m);
    const float e = ex2_approx(t);
    s.Z += e;
    s.T = fmaf(t, e, s.T);
  }
}

template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
};
template <>
struct Vec8<float> {
  __device__ __forceinline__ static void load(const float* p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
};

__device__ __forceinline__ uint64_t splitmix_out(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

}  // namespace

__device__ __forceinline__ uint64_t renoise_key(uint64_t seed, uint32_t step, uint32_t row) {
  return splitmix_out(splitmix_out(splitmix_out(seed) ^ uint64_t(step)) ^ uint64_t(row));
}

// Row outputs and the commit / renoise decision (per-position commit mode).
__device__ __forceinline__ void row_decision(const SampleArgs& a, int row, const RowState& t) {
  const float H = logf(t.Z) - kLn2 * t.T / t.Z;
  const float conf = 1.0f / t.Z;
  a.entropy[row] = H;
  a.confidence[row] = conf;
  a.argmax[row] = t.bi;
  if ((a.commit_mode & 1) == 0) {
    const bool fr = a.frozen != nullptr && a.frozen[row] != 0;
    const bool commit = fr || (H < a.bound);
    int tok;
    if (fr)
      tok = a.frozen_tokens[row];
    else if (commit)
      tok = t.bi;
    else
      tok = int(renoise_key(a.seed, a.step, uint32_t(row)) % uint64_t(a.V));
    a.tokens[row] = tok;
    a.commit_mask[row] = commit ? 1 : 0;
  }
}

// Warp, CTA and cluster reduction of the row state (fixed order: every CTA of
// the cluster ends with the same bits).  Returns the row's final state.
template <int kThreads>
__device__ __forceinline__ RowState reduce_row(RowState s, RowState* warp_part, float (*cl_part)[5],
                                               uint32_t rank, uint32_t csize) {
  constexpr int kWarps = kThreads / 32;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    RowState o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
    o.Z = __shfl_xor_sync(0xffffffffu, s.Z, off);
    o.T = __shfl_xor_sync(0xffffffffu, s.T, off);
    o.bx = __shfl_xor_sync(0xffffffffu, s.bx, off);
    o.bi = __shfl_xor_sync(0xffffffffu, s.bi, off);
    RowState lo = (threadIdx.x & off) ? o : s;
    const RowState hi = (threadIdx.x & off) ? s : o;
    state_merge(lo, hi);
    s = lo;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) warp_part[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    RowState t = warp_part[0];
    for (int w = 1; w < kWarps; ++w) state_merge(t, warp_part[w]);
    const uint32_t local = smem_u32(&cl_part[rank][0]);
    for (uint32_t dst = 0; dst < csize; ++dst) {
      const uint32_t ra = mapa_shared(local, dst);
      st_cluster_f32(ra + 0, t.m);
      st_cluster_f32(ra + 4, t.Z);
      st_cluster_f32(ra + 8, t.T);
      st_cluster_f32(ra + 12, t.bx);
      st_cluster_u32(ra + 16, uint32_t(t.bi));
    }
  }
  cluster_sync_all();
  RowState t;
  state_init(t);
  for (uint32_t r = 0; r < csize; ++r) {
    RowState o;
    o.m = cl_part[r][0];
    o.Z = cl_part[r][1];
    o.T = cl_part[r][2];
    o.bx = cl_part[r][3];
    o.bi = int(__float_as_uint(cl_part[r][4]));
    state_merge(t, o);
  }
  return t;
}

// bf16 logits, the slice staged in shared memory (up to 64 KB) by bulk copies
// of 16 KB, each completing on its own mbarrier: the whole HBM read is issued
// at once, the first pass starts on the first piece while the others are in
// flight, both passes read shared memory, and three CTAs fit on an SM.  The
// partial states are exchanged with st.async (distributed shared memory
// stores that complete on the receiving CTA's mbarrier), so the reduction
// needs no cluster-wide barrier; one cluster barrier, split into an arrive
// after the exchange and a wait before exit, keeps every CTA alive until all
// stores into it have landed.
constexpr int kSmemSliceBytes = kSampleSliceMaxElems * 2;  // largest staged slice
constexpr int kPieceElems = 8192;
constexpr int kMaxPieces = kSmemSliceBytes / (2 * kPieceElems);

__device__ __forceinline__ float bf16x2_max(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  __nv_bfloat162 x, y, z, w;
  memcpy(&x, &a, 4);
  memcpy(&y, &b, 4);
  memcpy(&z, &c, 4);
  memcpy(&w, &d, 4);
  const __nv_bfloat162 m = __hmax2(__hmax2(x, y), __hmax2(z, w));
  return fmaxf(__low2float(m), __high2float(m));
}

// The first pass is split in two: the thread's maximum and the 8-element
// group holding it first (packed bf16 maxima, no exponentials), then Z and T
// about that exact maximum -- no running rescale, no data-dependent branch
// per group.  Thread t owns 16-byte chunks t + kThreads k of the slice (8
// logits each, increasing with k), read conflict-free from shared memory.
// kSlice: the staged slice's bytes (at most kSmemSliceBytes); kFull: every
// slice is exactly that long (compile-time trip counts).
template <int kThreads, int kSlice, bool kFull>
__global__ void __launch_bounds__(kThreads) sample_rows_smem_kernel(SampleArgs a,
                                                                     const __nv_bfloat16* __restrict__ logits) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kMaxK = kSlice / 16 / kThreads;                    // chunks per thread
  constexpr int kKPerPiece = kPieceElems / 8 / kThreads;            // of them in one bulk-copy piece
  static_assert(kKPerPiece >= 1 && kMaxK % kKPerPiece == 0, "piece layout");
  extern __shared__ __align__(128) uint8_t slice_raw[];
  __shared__ RowState warp_part[kWarps];
  __shared__ __align__(16) uint32_t cl_msg[kMaxSampleCluster][8];
  __shared__ uint64_t full[kMaxPieces];
  __shared__ uint64_t red_bar;
  __shared__ int abort_flag;
  const int row = blockIdx.y;
  const uint32_t rank = cluster_ctarank();
  const uint32_t csize = gridDim.x;
  const long long c0 = (long long)rank * a.chunk;
  const long long c1 = min((long long)a.V, c0 + a.chunk);
  const int n = kFull ? kSlice / 2 : (c1 > c0 ? int(c1 - c0) : 0);  // a multiple of 8
  const int nch = n / 8;
  const __nv_bfloat16* src = logits + (long long)row * a.V + c0;
  const uint4* slice4 = reinterpret_cast<const uint4*>(slice_raw);
  if (threadIdx.x == 0) {
    for (int p = 0; p < kMaxPieces; ++p) mbar_init(&full[p], 1);
    mbar_init(&red_bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
    // this thread's arrival plus the bytes of every CTA's partial state
    mbar_arrive_expect_tx(&red_bar, csize * 32u);
    for (int p = 0; p * kPieceElems < n; ++p) {
      const uint32_t cnt = uint32_t(min(kPieceElems, n - p * kPieceElems));
      mbar_arrive_expect_tx(&full[p], cnt * 2u);
      bulk_load(slice_raw + p * kPieceElems * 2, src + p * kPieceElems, cnt * 2u, &full[p]);
    }
  }
  // every CTA's barriers are initialised before any peer stores into it (the
  // initialising thread's fence.mbarrier_init releases them; the arrive
  // itself needs no memory ordering)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
  const float ysc = a.inv_temp * kLog2e;
  // (1) the thread's maximum and the first chunk that holds it
  float bv = -INFINITY;
  int bk = -1;
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    // on a timeout the status word is set and the CTA carries on, so that
    // no peer waits for it
    if (k % kKPerPiece == 0 && (k / kKPerPiece) * kPieceElems < n) mbar_wait(&full[k / kKPerPiece], 0, &abort_flag);
    const int j = int(threadIdx.x) + k * kThreads;
    if (kFull || j < nch) {
      const uint4 u = slice4[j];
      const float gm = bf16x2_max(u.x, u.y, u.z, u.w);
      if (gm > bv) {  // strict: the earlier chunk keeps a tie
        bv = gm;
        bk = k;
      }
    }
  }
  RowState s;
  state_init(s);
  if (bk >= 0) {
    const int jb = int(threadIdx.x) + bk * kThreads;
    const uint4 u = slice4[jb];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    int e = 7;
#pragma unroll
    for (int q = 3; q >= 0; --q) {
      if (__uint_as_float(w[q] & 0xffff0000u) == bv) e = 2 * q + 1;
      if (__uint_as_float(w[q] << 16) == bv) e = 2 * q;
    }
    s.bx = bv;
    s.bi = int(c0) + 8 * jb + e;
    // (2) Z and T about the thread's maximum (base 2), two logits per
    // packed fp32x2 instruction (even / odd positions in the two lanes)
    const float mt = bv * ysc;
    const uint64_t ysc2 = f2_pack(ysc, ysc), nmt2 = f2_pack(-mt, -mt);
    uint64_t Z2 = 0, T2 = 0;
#pragma unroll 4
    for (int k = 0; k < kMaxK; ++k) {
      const int j = int(threadIdx.x) + k * kThreads;
      if (kFull || j < nch) {
        const uint4 v = slice4[j];
        const uint32_t x4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t t2 = f2_fma(f2_from_bf16x2(x4[q]), ysc2, nmt2);
          const uint64_t e2 = f2_pack(ex2_approx(f2_lo(t2)), ex2_approx(f2_hi(t2)));
          Z2 = f2_add(Z2, e2);
          T2 = f2_fma(t2, e2, T2);
        }
      }
    }
    s.m = mt;
    s.Z = f2_lo(Z2) + f2_hi(Z2);
    s.T = f2_lo(T2) + f2_hi(T2);
  }
  // warp, then CTA, then cluster (every CTA merges the partial states in
  // rank order, so all end with the same bits)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    RowState o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
    o.Z = __shfl_xor_sync(0xffffffffu, s.Z, off);
    o.T = __shfl_xor_sync(0xffffffffu, s.T, off);
    o.bx = __shfl_xor_sync(0xffffffffu, s.bx, off);
    o.bi = __shfl_xor_sync(0xffffffffu, s.bi, off);
    RowState lo = (threadIdx.x & off) ? o : s;
    const RowState hi = (threadIdx.x & off) ? s : o;
    state_merge(lo, hi);
    s = lo;
  }
  if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    RowState t = warp_part[0];
    for (int w = 1; w < kWarps; ++w) state_merge(t, warp_part[w]);
    const uint32_t msg = smem_u32(&cl_msg[rank][0]), bar = smem_u32(&red_bar);
    for (uint32_t dst = 0; dst < csize; ++dst) {
      const uint32_t ra = mapa_shared(msg, dst), rb = mapa_shared(bar, dst);
      st_async_v4(ra, __float_as_uint(t.m), __float_as_uint(t.Z), __float_as_uint(t.T), __float_as_uint(t.bx), rb);
      st_async_v4(ra + 16, uint32_t(t.bi), 0u, 0u, 0u, rb);
    }
  }
  // one warp merges the partial states in rank order and publishes the row's
  // maximum and 1 / Z to the CTA
  if (threadIdx.x < 32) {
    mbar_wait(&red_bar, 0, &abort_flag);
    RowState t;
    state_init(t);
    for (uint32_t r = 0; r < csize; ++r) {
      RowState o;
      o.m = __uint_as_float(cl_msg[r][0]);
      o.Z = __uint_as_float(cl_msg[r][1]);
      o.T = __uint_as_float(cl_msg[r][2]);
      o.bx = __uint_as_float(cl_msg[r][3]);
      o.bi = int(cl_msg[r][4]);
      state_merge(t, o);
    }
    if (threadIdx.x == 0) {
      warp_part[0].m = t.m;
      warp_part[0].Z = t.Z;
      if (rank == 0) row_decision(a, row, t);
    }
  }
  __syncthreads();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const RowState t = warp_part[0];  // the row's m and Z
  // p = 2^(y - m) / Z = 2^(y - (m + log2 Z)): the normaliser folded into the
  // exponent (the fp32 rounding of m + log2 Z moves p by about 2^-19 relative)
  const float nML = -(t.m + log2f(t.Z));
  const uint64_t ysc2 = f2_pack(ysc, ysc), nML2 = f2_pack(nML, nML);
#pragma unroll 4
  for (int k = 0; k < kMaxK; ++k) {
    const int j = int(threadIdx.x) + k * kThreads;
    if (!kFull && j >= nch) break;
    const int i = 8 * j;
    const uint4 u = slice4[j];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float p[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t t2 = f2_fma(f2_from_bf16x2(w[q]), ysc2, nML2);
      p[2 * q] = ex2_approx(f2_lo(t2));
      p[2 * q + 1] = ex2_approx(f2_hi(t2));
    }
    const long long o = (long long)row * a.V + c0 + i;
    if (a.probs_bf16) {
      uint4 q;
      q.x = pack_bf16x2(p[0], p[1]);
      q.y = pack_bf16x2(p[2], p[3]);
      q.z = pack_bf16x2(p[4], p[5]);
      q.w = pack_bf16x2(p[6], p[7]);
      *reinterpret_cast<uint4*>(a.probs_bf16 + o) = q;
    }
    if (a.probs_f32) {
      float4* q = reinterpret_cast<float4*>(a.probs_f32 + o);
      q[0] = make_float4(p[0], p[1], p[2], p[3]);
      q[1] = make_float4(p[4], p[5], p[6], p[7]);
    }
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Deferred normalisation (bf16 logits, no probabilities requested, argmax
// commits): the vocabulary of a row is cut into the K ranges of the
// soft-embedding GEMM's splits, one CTA per (range, row) and no cluster.  A
// CTA stages its range in shared memory as above, reduces it to its own
// (m_s, Z_s, T_s, argmax) state, writes p~ = 2^(y - m_s) (<= 1) for its
// range and stores the state; nothing waits for another CTA.  The row's
// statistics and decision, and the factor 2^(m_s - m) / Z that turns each
// range's p~ into probabilities, are applied after the GEMM, where its split
// partials are summed (soft_reduce_kernel): P.E = sum_s 2^(m_s - m) / Z *
// (p~_s . E_s).
template <int kThreads>
__global__ void __launch_bounds__(kThreads) sample_slices_kernel(SampleArgs a,
                                                                  const __nv_bfloat16* __restrict__ logits) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kMaxK = kSmemSliceBytes / 16 / kThreads;  // 16-byte chunks per thread
  constexpr int kKPerPiece = kPieceElems / 8 / kThreads;
  static_assert(kKPerPiece >= 1 && kMaxK % kKPerPiece == 0, "piece layout");
  extern __shared__ __align__(128) uint8_t slice_raw[];
  __shared__ RowState warp_part[kWarps];
  __shared__ uint64_t full[kMaxPieces];
  __shared__ int abort_flag;
  const int row = blockIdx.y, sl = blockIdx.x;
  const long long kb0 = (long long)sl * a.kb_per + min(sl, a.kb_rem);
  const long long c0 = kb0 * 64;
  const long long c1 = min((long long)a.V, (kb0 + a.kb_per + (sl < a.kb_rem ? 1 : 0)) * 64);
  const int n = c1 > c0 ? int(c1 - c0) : 0;  // a multiple of 8, at most kSmemSliceBytes / 2
  const int nch = n / 8;
  const __nv_bfloat16* src = logits + (long long)row * a.V + c0;
  const uint4* slice4 = reinterpret_cast<const uint4*>(slice_raw);
  if (threadIdx.x == 0) {
    for (int p = 0; p < kMaxPieces; ++p) mbar_init(&full[p], 1);
    abort_flag = 0;
    fence_mbarrier_init();
    for (int p = 0; p * kPieceElems < n; ++p) {
      const uint32_t cnt = uint32_t(min(kPieceElems, n - p * kPieceElems));
      mbar_arrive_expect_tx(&full[p], cnt * 2u);
      bulk_load(slice_raw + p * kPieceElems * 2, src + p * kPieceElems, cnt * 2u, &full[p]);
    }
  }
  __syncthreads();
  const float ysc = a.inv_temp * kLog2e;
  // (1) the thread's maximum and the first chunk that holds it
  float bv = -INFINITY;
  int bk = -1;
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    if (k % kKPerPiece == 0 && (k / kKPerPiece) * kPieceElems < n) mbar_wait(&full[k / kKPerPiece], 0, &abort_flag);
    const int j = int(threadIdx.x) + k * kThreads;
    if (j < nch) {
      const uint4 u = slice4[j];
      const float gm = bf16x2_max(u.x, u.y, u.z, u.w);
      if (gm > bv) {
        bv = gm;
        bk = k;
      }
    }
  }
  RowState s;
  state_init(s);
  if (bk >= 0) {
    const int jb = int(threadIdx.x) + bk * kThreads;
    const uint4 u = slice4[jb];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    int e = 7;
#pragma unroll
    for (int q = 3; q >= 0; --q) {
      if (__uint_as_float(w[q] & 0xffff0000u) == bv) e = 2 * q + 1;
      if (__uint_as_float(w[q] << 16) == bv) e = 2 * q;
    }
    s.bx = bv;
    s.bi = int(c0) + 8 * jb + e;
    // (2) Z and T about the thread's maximum, two logits per instruction
    const float mt = bv * ysc;
    const uint64_t ysc2 = f2_pack(ysc, ysc), nmt2 = f2_pack(-mt, -mt);
    uint64_t Z2 = 0, T2 = 0;
#pragma unroll 4
    for (int k = 0; k < kMaxK; ++k) {
      const int j = int(threadIdx.x) + k * kThreads;
      if (j < nch) {
        const uint4 v = slice4[j];
        const uint32_t x4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t t2 = f2_fma(f2_from_bf16x2(x4[q]), ysc2, nmt2);
          const uint64_t e2 = f2_pack(ex2_approx(f2_lo(t2)), ex2_approx(f2_hi(t2)));
          Z2 = f2_add(Z2, e2);
          T2 = f2_fma(t2, e2, T2);
        }
      }
    }
    s.m = mt;
    s.Z = f2_lo(Z2) + f2_hi(Z2);
    s.T = f2_lo(T2) + f2_hi(T2);
  }
  // warp, then CTA (fixed order)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    RowState o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
    o.Z = __shfl_xor_sync(0xffffffffu, s.Z, off);
    o.T = __shfl_xor_sync(0xffffffffu, s.T, off);
    o.bx = __shfl_xor_sync(0xffffffffu, s.bx, off);
    o.bi = __shfl_xor_sync(0xffffffffu, s.bi, off);
    RowState lo = (threadIdx.x & off) ? o : s;
    const RowState hi = (threadIdx.x & off) ? s : o;
    state_merge(lo, hi);
    s = lo;
  }
  if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    RowState t = warp_part[0];
    for (int w = 1; w < kWarps; ++w) state_merge(t, warp_part[w]);
    float* st = a.slice_state + ((long long)row * a.slices + sl) * 8;
    reinterpret_cast<float4*>(st)[0] = make_float4(t.m, t.Z, t.T, t.bx);
    reinterpret_cast<int4*>(st)[1] = make_int4(t.bi, 0, 0, 0);
    warp_part[0].m = t.m;
  }
  __syncthreads();
  // p~ = 2^(y - m_s) (a range with no finite logit writes zeros)
  const float ms = warp_part[0].m;
  const bool live = ms != -INFINITY;
  const uint64_t ysc2 = f2_pack(ysc, ysc), nms2 = f2_pack(-ms, -ms);
  __nv_bfloat16* dst = a.probs_bf16 + (long long)row * a.V + c0;
#pragma unroll 4
  for (int k = 0; k < kMaxK; ++k) {
    const int j = int(threadIdx.x) + k * kThreads;
    if (j >= nch) break;
    const uint4 u = slice4[j];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t t2 = f2_fma(f2_from_bf16x2(w[i]), ysc2, nms2);
      q[i] = live ? pack_bf16x2(ex2_approx(f2_lo(t2)), ex2_approx(f2_hi(t2))) : 0u;
    }
    *reinterpret_cast<uint4*>(dst + 8 * j) = make_uint4(q[0], q[1], q[2], q[3]);
  }
}

// After the soft-embedding GEMM of the deferred path: a row's blocks (its D
// columns cut into blockDim-wide float4 groups) each merge the row's range
// states (warp 0: lane s holds range s, a fixed butterfly merges them, so the
// row's m, Z, T and argmax are bit-identical in every block and whichever
// order the ranges ran in); the first block writes the row outputs and
// decision.  Every thread loads its four columns' split partials before the
// merge (up to kSoftRegSplits of them held in registers) and then sums them
// in split order, each scaled by 2^(m_s - m) / Z.
constexpr int kSoftReduceThreads = 128;
constexpr int kSoftRegSplits = 16;
__global__ void __launch_bounds__(kSoftReduceThreads) soft_reduce_kernel(SampleArgs a,
                                                                         const float* __restrict__ partials,
                                                                         float* __restrict__ soft, int D) {
  __shared__ float wgt[kMaxSampleSlices];
  const int row = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;  // float4 column
  const bool col = c < D / 4;
  const long long plane = (long long)a.rows * D / 4;  // float4s per split slab
  const float4* p4 = reinterpret_cast<const float4*>(partials) + (long long)row * D / 4 + c;
  float4 v[kSoftRegSplits];
#pragma unroll
  for (int j = 0; j < kSoftRegSplits; ++j)
    if (col && j < a.slices) v[j] = __ldcs(p4 + j * plane);
  const float* st0 = a.slice_state + (long long)row * a.slices * 8;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    auto load_state = [&](int sl) {
      RowState o;
      const float4 f = reinterpret_cast<const float4*>(st0 + sl * 8)[0];
      o.m = f.x;
      o.Z = f.y;
      o.T = f.z;
      o.bx = f.w;
      o.bi = reinterpret_cast<const int4*>(st0 + sl * 8)[1].x;
      return o;
    };
    RowState t;
    state_init(t);
    for (int sl = lane; sl < a.slices; sl += 32) state_merge(t, load_state(sl));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      RowState o;
      o.m = __shfl_xor_sync(0xffffffffu, t.m, off);
      o.Z = __shfl_xor_sync(0xffffffffu, t.Z, off);
      o.T = __shfl_xor_sync(0xffffffffu, t.T, off);
      o.bx = __shfl_xor_sync(0xffffffffu, t.bx, off);
      o.bi = __shfl_xor_sync(0xffffffffu, t.bi, off);
      RowState lo = (lane & off) ? o : t;
      const RowState hi = (lane & off) ? t : o;
      state_merge(lo, hi);
      t = lo;
    }
    if (lane == 0 && blockIdx.y == 0) row_decision(a, row, t);
    for (int sl = lane; sl < a.slices; sl += 32) {
      const float ms = st0[sl * 8], zs = st0[sl * 8 + 1];
      wgt[sl] = (zs > 0.f && t.Z > 0.f) ? ex2_approx(ms - t.m) / t.Z : 0.f;
    }
  }
  __syncthreads();
  if (!col) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kSoftRegSplits; ++j) {
    if (j < a.slices) {
      const float w = wgt[j];
      acc.x = fmaf(w, v[j].x, acc.x);
      acc.y = fmaf(w, v[j].y, acc.y);
      acc.z = fmaf(w, v[j].z, acc.z);
      acc.w = fmaf(w, v[j].w, acc.w);
    }
  }
  for (int s0 = kSoftRegSplits; s0 < a.slices; s0 += 8) {
    float4 u[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (s0 + j < a.slices) u[j] = __ldcs(p4 + (s0 + j) * plane);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (s0 + j < a.slices) {
        const float w = wgt[s0 + j];
        acc.x = fmaf(w, u[j].x, acc.x);
        acc.y = fmaf(w, u[j].y, acc.y);
        acc.z = fmaf(w, u[j].z, acc.z);
        acc.w = fmaf(w, u[j].w, acc.w);
      }
    }
  }
  reinterpret_cast<float4*>(soft)[(long long)row * D / 4 + c] = acc;
}

template <typename T, int kThreads>
__global__ void __launch_bounds__(kThreads) sample_rows_kernel(SampleArgs a, const T* __restrict__ logits) {
  constexpr int kWarps = kThreads / 32;
  __shared__ RowState warp_part[kWarps];
  __shared__ float cl_part[kMaxSampleCluster][5];

  const int row = blockIdx.y;
  const uint32_t rank = cluster_ctarank();
  const uint32_t csize = gridDim.x;  // cluster spans the x dimension of the grid
  const long long c0 = (long long)rank * a.chunk;
  const long long c1 = min((long long)a.V, c0 + a.chunk);
  const T* lrow = logits + (long long)row * a.V;
  const float ysc = a.inv_temp * kLog2e;

  // every CTA of the cluster must be running before any DSMEM store below
  cluster_sync_all();
  RowState s;
  state_init(s);
  // pass 1: statistics
  for (long long i = c0 + (long long)threadIdx.x * 8; i < c1; i += (long long)kThreads * 8) {
    float x[8];
    Vec8<T>::load(lrow + i, x);
    state_add8(s, x, ysc, int(i));
  }
  const RowState t = reduce_row<kThreads>(s, warp_part, cl_part, rank, csize);
  if (threadIdx.x == 0 && rank == 0) row_decision(a, row, t);
  const float M = t.m;
  const float invZ = 1.0f / t.Z;
  // pass 2: probabilities
  for (long long i = c0 + (long long)threadIdx.x * 8; i < c1; i += (long long)kThreads * 8) {
    float x[8], p[8];
    Vec8<T>::load(lrow + i, x);
#pragma unroll
    for (int j = 0; j < 8; ++j) p[j] = ex2_approx(fmaf(x[j], ysc, -M)) * invZ;
    const long long o = (long long)row * a.V + i;
    if (a.probs_bf16) {
      uint4 u;
      u.x = pack_bf16x2(p[0], p[1]);
      u.y = pack_bf16x2(p[2], p[3]);
      u.z = pack_bf16x2(p[4], p[5]);
      u.w = pack_bf16x2(p[6], p[7]);
      *reinterpret_cast<uint4*>(a.probs_bf16 + o) = u;
    }
    if (a.probs_f32) {
      float4* q = reinterpret_cast<float4*>(a.probs_f32 + o);
      q[0] = make_float4(p[0], p[1], p[2], p[3]);
      q[1] = make_float4(p[4], p[5], p[6], p[7]);
    }
  }
}

// Categorical draw for the committed positions (commit_mode bit 1): the
// token is the smallest index k whose cumulative stored probability exceeds
// u * (sum of the stored probabilities), u = the top 24 bits of the row's
// SplitMix64 key / 2^24 (the key that would renoise the row: a position
// either commits or renoises).  One block per row; thread t sums a contiguous
// range in fp64, a block scan places the target, and the thread whose range
// holds it walks its range in index order.  Frozen and renoised rows keep
// their tokens.
template <typename P>
__device__ __forceinline__ double prob_at(const P* p, long long i);
template <>
__device__ __forceinline__ double prob_at<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
  return double(__bfloat162float(p[i]));
}
template <>
__device__ __forceinline__ double prob_at<float>(const float* p, long long i) {
  return double(p[i]);
}

template <typename P>
__global__ void __launch_bounds__(256) categorical_kernel(SampleArgs a, const P* __restrict__ probs) {
  constexpr int kT = 256;
  __shared__ double part[kT];
  __shared__ double target;
  __shared__ int found;
  const int row = blockIdx.x;
  if (a.commit_mask[row] == 0) return;
  if (a.frozen != nullptr && a.frozen[row] != 0) return;
  const P* pr = probs + (long long)row * a.V;
  const int n = (a.V + kT - 1) / kT;
  const long long i0 = (long long)threadIdx.x * n;
  const long long i1 = min((long long)a.V, i0 + n);
  double sum = 0.0;
  for (long long i = i0; i < i1; ++i) sum += prob_at<P>(pr, i);
  part[threadIdx.x] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    // exclusive prefix of the range sums, in thread (index) order
    double acc = 0.0;
    for (int t = 0; t < kT; ++t) {
      const double v = part[t];
      part[t] = acc;
      acc += v;
    }
    const uint64_t key = renoise_key(a.seed, a.step, uint32_t(row));
    target = double(key >> 40) * (1.0 / 16777216.0) * acc;
    found = -1;
  }
  __syncthreads();
  const double lo = part[threadIdx.x];
  const double hi = threadIdx.x + 1 < kT ? part[threadIdx.x + 1] : lo + sum;
  if (lo <= target && target < hi) {
    // the ranges are disjoint, so exactly one thread gets here
    double run = lo;
    int k = -1, last = -1;
    for (long long i = i0; i < i1; ++i) {
      const double v = prob_at<P>(pr, i);
      run += v;
      if (v > 0.0) last = int(i);
      if (run > target) {
        k = int(i);
        break;
      }
    }
    // the walk's sum ends an ulp short of hi: the target sits on the range's
    // last boundary, which its last positive entry closes
    found = k >= 0 ? k : last;
  }
  __syncthreads();
  if (threadIdx.x == 0) a.tokens[row] = found >= 0 ? found : a.argmax[row];
}

// Left-prefix commit mode: one thread per canvas walks its rows in order.
__global__ void commit_prefix_kernel(SampleArgs a, int n_canvas) {
  const int cv = blockIdx.x * blockDim.x + threadIdx.x;
  if (cv >= n_canvas) return;
  bool run = true;
  for (int i = 0; i < a.canvas_len; ++i) {
    const int row = cv * a.canvas_len + i;
    const bool fr = a.frozen != nullptr && a.frozen[row] != 0;
    run = run && (fr || a.entropy[row] < a.bound);
    const bool commit = fr || run;
    int tok;
    if (fr)
      tok = a.frozen_tokens[row];
    else if (commit)
      tok = a.argmax[row];
    else
      tok = int(renoise_key(a.seed, a.step, uint32_t(row)) % uint64_t(a.V));
    a.tokens[row] = tok;
    a.commit_mask[row] = commit ? 1 : 0;
  }
}

cudaError_t launch_sampler(const SampleArgs& a, const void* logits, bool bf16, cudaStream_t stream) {
  constexpr int kThreads = 256;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.cluster, a.rows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  const __nv_bfloat16* lb = static_cast<const __nv_bfloat16*>(logits);
  if (bf16 && size_t(a.chunk) * 2 <= size_t(kSmemSliceBytes)) {
    static bool attr_set = false;
    if (!attr_set) {
      e = cudaFuncSetAttribute(sample_rows_smem_kernel<kThreads, kSmemSliceBytes, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemSliceBytes);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(sample_rows_smem_kernel<kThreads, kSmemSliceBytes, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemSliceBytes);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
    cfg.dynamicSmemBytes = size_t(a.chunk) * 2;
    // every CTA's slice exactly full: compile-time trip counts
    const bool whole = (long long)a.chunk * a.cluster == a.V;
    if (whole && size_t(a.chunk) * 2 == size_t(kSmemSliceBytes))
      e = cudaLaunchKernelEx(&cfg, sample_rows_smem_kernel<kThreads, kSmemSliceBytes, true>, a, lb);
    else
      e = cudaLaunchKernelEx(&cfg, sample_rows_smem_kernel<kThreads, kSmemSliceBytes, false>, a, lb);
  } else if (bf16) {
    e = cudaLaunchKernelEx(&cfg, sample_rows_kernel<__nv_bfloat16, kThreads>, a, lb);
  } else {
    e = cudaLaunchKernelEx(&cfg, sample_rows_kernel<float, kThreads>, a, static_cast<const float*>(logits));
  }
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (a.commit_mode & 1) {
    const int n_canvas = a.rows / a.canvas_len;
    commit_prefix_kernel<<<(n_canvas + 127) / 128, 128, 0, stream>>>(a, n_canvas);
    e = cudaGetLastError();
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  if (a.commit_mode & 2) {
    if (bf16)
      categorical_kernel<__nv_bfloat16><<<a.rows, 256, 0, stream>>>(a, a.probs_bf16);
    else
      categorical_kernel<float><<<a.rows, 256, 0, stream>>>(a, a.probs_f32);
    e = cudaGetLastError();
    count_launches(1);
  }
  return e;
}

cudaError_t launch_sampler_slices(const SampleArgs& a, const void* logits, cudaStream_t stream) {
  constexpr int kThreads = 256;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(sample_slices_kernel<kThreads>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemSliceBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long elems = ((long long)a.kb_per + (a.kb_rem > 0 ? 1 : 0)) * 64;
  const size_t smem = size_t(min((long long)a.V, elems)) * 2;
  sample_slices_kernel<kThreads><<<dim3(a.slices, a.rows, 1), kThreads, smem, stream>>>(
      a, static_cast<const __nv_bfloat16*>(logits));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_soft_reduce(const SampleArgs& a, const float* partials, float* soft, int D, cudaStream_t stream) {
  const int col_blocks = (D / 4 + kSoftReduceThreads - 1) / kSoftReduceThreads;
  soft_reduce_kernel<<<dim3(a.rows, col_blocks, 1), kSoftReduceThreads, 0, stream>>>(a, partials, soft, D);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !(a.commit_mode & 1)) return e;
  const int n_canvas = a.rows / a.canvas_len;
  commit_prefix_kernel<<<(n_canvas + 127) / 128, 128, 0, stream>>>(a, n_canvas);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace canvas

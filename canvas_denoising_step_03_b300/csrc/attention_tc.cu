// attention_tc.cu -- decode-mode canvas attention on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA-fed shared memory).
//
// Method: AI Trends summary of a DiffusionGemma 26B notebook
// (aitrends.kr/articles/94089), "섹션별 상세": decode mode (the canvas attends
// bidirectionally to the committed prefix in the KV cache and to the whole
// canvas), scores q . k with the scale fixed by the scalar QK norm; the
// glossary entries on sliding-window attention and on the shared K/V
// projection of full-attention layers.
//
// Work unit (one CTA): a 128-row query tile of one (sequence b, KV head hk)
// -- the G query heads of the KV head packed as rows g * C + i (GQA) -- one
// part of the value dimension (DV = min(d, 256) columns) and one contiguous
// range of 128-key blocks (a KV split).  Keys are the position range of the
// key sequence (kernels.h); 64-key sub-blocks come either from the committed
// prefix in place (paged cache through the block table, or the dense global
// keys) or from the dense tail buffers.
//
// Roles (320 threads):
//   warp 0       TMA producer: Q tile once; then K chunks and V sub-blocks in
//                the order the MMA warp consumes them, through a ring of
//                32 KB stages (128-byte swizzle).
//   warp 1       TMEM allocation (512 columns) and the MMA issuer:
//                S_n = Q K_n^T (M=128, N=128, both operands in shared memory)
//                into one of two S buffers; O += P_n V_n (M=128, N=DV, P read
//                from TMEM where the softmax wrote it over S_n, V from shared
//                memory, MN-major).  Issue order QK0 QK1 PV0 QK2 PV1 ...
//   warps 2..9   softmax and epilogue, one query row per thread (TMEM lane)
//                and one 64-key half of each block per warp: S from TMEM,
//                masking, running max in the log2 domain (agreed between the
//                two warps of a row), P = 2^(S c - m) rounded to bf16 and
//                stored back to TMEM.
//                The accumulator is rescaled only when the running max grows
//                by more than 8 (P stays below 2^8), so most blocks never
//                touch O.
// With d = 512 the 128 x 512 fp32 accumulator would fill all of TMEM: the
// four-SM kernel further below splits the value dimension and the key blocks
// between two CTA pairs (this kernel can also split the value dimension
// across two CTAs that both form the full S); every other shape keeps the
// whole row in one CTA.
// Results: bf16 rows (and the natural-log LSE) when the key range is not
// split, else fp32 partial rows plus (max, sum) for the combine kernel.
// Every mbarrier wait is bounded (common.cuh).
#include "common.cuh"
#include "kernels.h"

namespace canvas {

namespace {

constexpr int kThreads = 320;  // TMA warp, MMA warp, 8 softmax / epilogue warps
constexpr int kStageBytes = 32768;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
// exchange area of the two softmax warps of a row quadrant: the block maxima
// of the two key halves as bf16 rounded up ([2 blocks][2 halves][128 rows]),
// then the final partial sums (fp32 [2 halves][128 rows])
constexpr int kXchgBytes = 1024;
constexpr int kBarBytes = 256;  // 18 mbarriers, the TMEM address and the abort flag

template <int D>
struct Cfg {
  static constexpr int DV = D < 256 ? D : 256;
  static constexpr int NCH = D / 64;             // 64-wide chunks of the head dimension
  static constexpr int KCH = NCH < 2 ? NCH : 2;  // chunks per K stage
  static constexpr int KST = NCH / KCH;          // K stages per block
  static constexpr int NST = D == 512 ? 3 : 5;   // ring stages
  static constexpr int QBytes = NCH * 16384;
  static constexpr int Smem = QBytes + NST * kStageBytes + 1024 + kBarBytes + kXchgBytes;
};

// bf16 bit pattern of the smallest bf16 value >= x (x finite or -inf).
__device__ __forceinline__ uint16_t bf16_bits_up(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0xffffu) != 0u && (u & 0x7f800000u) != 0x7f800000u) {
    // drop the low bits towards zero, then step away from zero for positive
    // values (towards +inf); negative values truncated are already larger
    u &= 0xffff0000u;
    if (!(u >> 31)) u += 0x10000u;
  }
  return uint16_t(u >> 16);
}

// The block sequence of one CTA (identical in every thread).
struct Seq {
  int P, P64, T, s0, n_pre, n_sub, kb0, nb, lo_max;
  bool ok;
};

// First visible prefix position of canvas row i (the host passes window 0 on
// global layers: the whole prefix is visible).
__device__ __forceinline__ int window_lo(const AttnTcArgs& a, int P, int i) {
  if (a.window <= 0) return 0;
  return min(P, max(0, P + i - a.window));
}

// rows_per_unit: query rows whose key blocks this sequence serves (one tile,
// or the two tiles of a CTA pair); qt counts units of that size.
__device__ __forceinline__ Seq make_seq(const AttnTcArgs& a, int b, int qt, int split,
                                        int rows_per_unit = kAttnBM) {
  Seq q;
  q.P = a.prefix_len[b];
  q.ok = q.P >= 0 && q.P <= a.max_prefix;
  if (!q.ok) return q;
  q.P64 = q.P & ~63;
  q.T = q.P - q.P64 + a.C;
  const int GC = a.G * a.C;
  const int R0 = qt * rows_per_unit;
  const int nrows = max(1, min(rows_per_unit, GC - R0));
  int i_min, i_max;
  if (R0 / a.C == (R0 + nrows - 1) / a.C) {
    i_min = R0 % a.C;
    i_max = (R0 + nrows - 1) % a.C;
  } else {
    i_min = 0;
    i_max = a.C - 1;
  }
  const int lo_min = window_lo(a, q.P, i_min);
  q.lo_max = window_lo(a, q.P, i_max);
  q.s0 = lo_min & ~63;
  q.n_pre = (q.P64 - q.s0) / 64;
  q.n_sub = q.n_pre + (q.T + 63) / 64;
  const int nblk = (q.n_sub + 1) / 2;
  q.kb0 = (int)((long long)split * nblk / a.nsplit);
  q.nb = (int)((long long)(split + 1) * nblk / a.nsplit) - q.kb0;
  return q;
}

// TMA row of 64-key sub-block s in the prefix (paged pool) or tail buffers.
__device__ __forceinline__ int paged_row(const AttnTcArgs& a, int b, int hk, int pos) {
  const int lp = pos / a.page_tokens;
  int page = lp < a.max_pages ? a.block_table[(size_t)b * a.max_pages + lp] : -1;
  if (page < 0 || page >= a.num_pages) {
    record_error(CANVAS_ERR_BOUNDS);
    page = 0;  // stay inside the pool; the call reports the error
  }
  return (page * a.Hkv + hk) * a.page_tokens + pos % a.page_tokens;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const __grid_constant__ AttnTcMaps maps, AttnTcArgs a) {
  using K = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* ring = smem + K::QBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + K::NST * kStageBytes);
  uint64_t* empty = full + K::NST;
  uint64_t* q_full = empty + K::NST;
  uint64_t* s_full = q_full + 1;   // [2]
  uint64_t* p_full = s_full + 2;   // [2]
  uint64_t* pv_done = p_full + 2;  // [2]
  uint64_t* drain = pv_done + 2;
  uint64_t* xbar = drain + 1;      // [4] the two softmax warps of a row quadrant
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 4);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort
  static_assert((2 * K::NST + 1 + 2 * 3 + 1 + 4) * 8 + 8 <= kBarBytes, "barrier area");
  uint16_t* xmax = reinterpret_cast<uint16_t*>(ring + K::NST * kStageBytes + kBarBytes);  // [2][2][128]
  float* xsum = reinterpret_cast<float*>(xmax);                                          // [2][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int x = blockIdx.x;
  const int dvp = x % a.dv_parts;
  x /= a.dv_parts;
  const int qt = x % a.q_tiles;
  x /= a.q_tiles;
  const int split = x % a.nsplit;
  x /= a.nsplit;
  const int hk = x % a.Hkv;
  const int b = x / a.Hkv;
  const int grp = b * a.Hkv + hk;
  const Seq sq = make_seq(a, b, qt, split);
  if (!sq.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(CANVAS_ERR_BOUNDS);
    return;  // uniform: before any barrier or TMEM allocation
  }
  const int nb = sq.nb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < K::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(&s_full[j], 1);
      mbar_init(&p_full[j], 8);  // one arrival per softmax warp
      mbar_init(&pv_done[j], 1);
    }
    mbar_init(drain, 1);
    for (int j = 0; j < 4; ++j) mbar_init(&xbar[j], 2);
    flags[0] = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.kpre);
    tma_prefetch_desc(&maps.vpre_c);
    tma_prefetch_desc(&maps.kx);
    tma_prefetch_desc(&maps.vx_c);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      mbar_arrive_expect_tx(q_full, uint32_t(K::QBytes));
      const int qrow = grp * a.G * a.C + qt * kAttnBM;
      for (int c = 0; c < K::NCH; ++c) tma_load_2d(sQ + c * 16384, &maps.q, q_full, c * 64, qrow);
      int it = 0;
      bool alive = true;
      auto acquire = [&](uint32_t bytes) -> uint8_t* {
        const int s = it % K::NST;
        if (!mbar_wait(&empty[s], ((it / K::NST) & 1) ^ 1, flags)) {
          alive = false;
          return nullptr;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        ++it;
        return ring + s * kStageBytes;
      };
      auto k_row = [&](int s, const CUtensorMap*& map) -> int {
        if (s < sq.n_pre) {
          const int pos = sq.s0 + 64 * s;
          map = &maps.kpre;
          return a.kpre_paged ? paged_row(a, b, hk, pos) : grp * a.max_prefix + pos;
        }
        map = &maps.kx;
        return grp * a.Tpad + 64 * (s - sq.n_pre);
      };
      // values through the 3D views (all DV columns of a 64-key sub-block in
      // one copy) when they cover the whole head dimension
      constexpr bool kV3 = K::DV == D;
      auto v_row = [&](int s, const CUtensorMap*& map) -> int {
        if (s < sq.n_pre) {
          map = kV3 ? &maps.vpre_c : &maps.vpre;
          return paged_row(a, b, hk, sq.s0 + 64 * s);
        }
        map = kV3 ? &maps.vx_c : &maps.vx;
        return grp * a.Tpad + 64 * (s - sq.n_pre);
      };
      auto load_k = [&](int n) {
        const int kb = sq.kb0 + n;
        for (int ks = 0; ks < K::KST && alive; ++ks) {
          uint8_t* dst = acquire(uint32_t(K::KCH * 16384));
          if (!dst) break;
          for (int u = 0; u < 2; ++u) {
            const CUtensorMap* map;
            const int row = k_row(2 * kb + u, map);
            for (int c = 0; c < K::KCH; ++c)
              tma_load_2d(dst + c * 16384 + u * 8192, map, &full[(it - 1) % K::NST], (ks * K::KCH + c) * 64, row);
          }
        }
      };
      auto load_v = [&](int n) {
        const int kb = sq.kb0 + n;
        for (int u = 0; u < 2 && alive; ++u) {
          uint8_t* dst = acquire(uint32_t(K::DV / 64 * 8192));
          if (!dst) break;
          const CUtensorMap* map;
          const int row = v_row(2 * kb + u, map);
          if (kV3)
            tma_load_3d(dst, map, &full[(it - 1) % K::NST], 0, row, 0);
          else
            for (int c = 0; c < K::DV / 64; ++c)
              tma_load_2d(dst + c * 8192, map, &full[(it - 1) % K::NST], dvp * K::DV + c * 64, row);
        }
      };
      for (int n = 0; n < nb && alive; ++n) {
        load_k(n);
        if (n >= 1) load_v(n - 1);
      }
      if (nb >= 1 && alive) load_v(nb - 1);
      // drain: every load this thread issued has landed before the CTA exits
      volatile int no_abort = 0;
      mbar_wait(q_full, 0, &no_abort);
      for (int j = max(0, it - K::NST); j < it; ++j) mbar_wait(&full[j % K::NST], (j / K::NST) & 1, &no_abort);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc_qk = idesc_bf16_f32(128, kAttnBN, 0, 0);
      const uint32_t idesc_pv = idesc_bf16_f32(128, K::DV, 0, 1);
      const uint32_t q_base = smem_u32(sQ);
      int it = 0;
      bool alive = mbar_wait(q_full, 0, flags);
      tc_fence_after();
      auto consume = [&]() -> uint32_t {
        const int s = it % K::NST;
        if (!mbar_wait(&full[s], (it / K::NST) & 1, flags)) {
          alive = false;
          return 0;
        }
        tc_fence_after();
        ++it;
        return smem_u32(ring + s * kStageBytes);
      };
      auto qk = [&](int n) {
        const uint32_t tS = tmem + 256 + (n & 1) * 128;
        for (int ks = 0; ks < K::KST && alive; ++ks) {
          const uint32_t st = consume();
          if (!alive) return;
#pragma unroll
          for (int c = 0; c < K::KCH; ++c) {
            const int ch = ks * K::KCH + c;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc_sw128(q_base + ch * 16384 + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(st + c * 16384 + kk * 32, 16, 1024);
              mma_bf16_ss(tS, ad, bd, idesc_qk, (ch | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&empty[(it - 1) % K::NST]);
        }
        mma_commit(&s_full[n & 1]);
      };
      auto pv = [&](int n) {
        const uint32_t tS = tmem + 256 + (n & 1) * 128;
        for (int u = 0; u < 2 && alive; ++u) {
          const uint32_t st = consume();
          if (!alive) return;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = smem_desc_sw128(st + kk * 2048, 8192, 1024);
            mma_bf16_ts(tmem, tS + u * 32 + kk * 8, bd, idesc_pv, (n | u | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[(it - 1) % K::NST]);
        }
        mma_commit(&pv_done[n & 1]);
      };
      if (alive && nb >= 1) qk(0);
      if (alive && nb >= 2) qk(1);
      for (int n = 0; n < nb && alive; ++n) {
        if (!mbar_wait(&p_full[n & 1], (n >> 1) & 1, flags)) break;
        tc_fence_after();
        pv(n);
        if (n + 2 < nb) qk(n + 2);
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
  } else {
    // ------------------------------------------------ softmax + epilogue
    // Eight warps: warp w reads TMEM lanes 32 (w % 4) .. +31 (one query row
    // per thread) and key half h = (w - 2) / 4 of every block (columns
    // 64 h .. 64 h + 63, one 64-key sub-block).  The two warps of a row
    // quadrant agree on the running maximum through shared memory once per
    // block (named barrier 1 + quadrant), keep their own partial sums, and
    // split the value columns of O for the rescale and the epilogue.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int lrow = quad * 32 + lane;
    const uint32_t lane_off = uint32_t(quad * 32) << 16;
    const int GC = a.G * a.C;
    const int R = qt * kAttnBM + lrow;
    const bool valid = R < GC;
    const int g = valid ? R / a.C : 0, i = valid ? R % a.C : 0;
    const int lo_row = valid ? window_lo(a, sq.P, i) : 0;
    constexpr int DVH = K::DV / 2;  // value columns this warp rescales / writes
    float m_run = -INFINITY, l = 0.f;
    bool alive = true;
    // the pair of warps of this quadrant meet on xbar[quad] once per block and
    // twice in the epilogue (phase k completes when both warps arrive);
    // bounded, so an aborted partner cannot strand a warp
    int xphase = 0;
    auto pair_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[quad]);
      const bool ok = mbar_wait(&xbar[quad], uint32_t(xphase & 1), flags);
      ++xphase;
      return ok;
    };
    for (int n = 0; n < nb; ++n) {
      if (!mbar_wait(&s_full[n & 1], (n >> 1) & 1, flags)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + 256 + (n & 1) * 128;
      // this warp's 64 keys: sub-block sb of the key sequence
      const int kb = sq.kb0 + n;
      const int sb = 2 * kb + half;
      int pos0, hi_off = 64;
      if (sb < sq.n_pre) {
        pos0 = sq.s0 + 64 * sb;
      } else {
        const int t0 = 64 * (sb - sq.n_pre);
        pos0 = sq.P64 + t0;
        hi_off = min(64, sq.T - t0);
      }
      // encode mode: canvas keys up to the row's own position
      if (a.causal && valid) hi_off = min(hi_off, sq.P + i + 1 - pos0);
      // visible offsets [lo_off, hi_off): position >= the row's window start
      // (lo_row <= P, so canvas keys pass) and, in the tail, before the padding
      const int lo_off = max(0, lo_row - pos0);
      uint32_t sv[64];
      tmem_ld32(tS + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tS + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld_wait();
      if (__any_sync(0xffffffffu, lo_off > 0 || hi_off < 64)) {
#pragma unroll
        for (int off = 0; off < 64; ++off)
          if (off < lo_off || off >= hi_off) sv[off] = __float_as_uint(-INFINITY);
      }
      // block maximum in the log2 domain (c_log2 > 0), agreed by the pair:
      // each half publishes its maximum rounded up to bf16, and both take the
      // larger published value (an upper bound of the block maximum, the same
      // bits in both warps)
      float smax = __uint_as_float(sv[0]);
#pragma unroll
      for (int c = 1; c < 64; ++c) smax = fmaxf(smax, __uint_as_float(sv[c]));
      const uint16_t mine = bf16_bits_up(smax);
      xmax[((n & 1) * 2 + half) * kAttnBM + lrow] = mine;
      if (!pair_sync()) {
        alive = false;
        break;
      }
      const uint16_t other = xmax[((n & 1) * 2 + (half ^ 1)) * kAttnBM + lrow];
      smax = fmaxf(bf16_bits_to_f32(mine), bf16_bits_to_f32(other));
      const float bmax = smax * a.c_log2;
      const float m_new = fmaxf(m_run, bmax);
      const bool need = (m_run != -INFINITY) && (m_new > m_run + kRescaleLog2);
      const float alpha = need ? exp2f(m_run - m_new) : 1.f;
      if (need) {
        l *= alpha;
        m_run = m_new;
      } else if (m_run == -INFINITY) {
        m_run = m_new;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // P = 2^(s c - m) rounded to bf16 pairs over this half's S columns
      // (keys 64 h + 32 c2 .. -> packed columns 32 h + 16 c2 ..)
      float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c2 * 32 + 2 * j;
          const float p0 = ex2_approx(fmaf(__uint_as_float(sv[c]), a.c_log2, -m_use));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sv[c + 1]), a.c_log2, -m_use));
          if (a.vs_pre == nullptr) {
            pk[j] = pack_bf16x2(p0, p1);
            // the sum uses the rounded weights, so O / l is an exact convex
            // combination of value rows with the stored weights
            l_lo += __uint_as_float(pk[j] << 16);
            l_hi += __uint_as_float(pk[j] & 0xffff0000u);
          } else {
            // unit-RMS values: weight of each key times its row scalar sc; the
            // sum divides the stored product back by sc for the same reason
            float sc[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int off = c + e;
              sc[e] = sb < sq.n_pre ? a.vs_pre[(size_t)grp * a.max_prefix + pos0 + off]
                                    : a.vs_tail[(size_t)grp * a.Tpad + (pos0 - sq.P64) + off];
            }
            pk[j] = pack_bf16x2(p0 * sc[0], p1 * sc[1]);
            const float w0 = __uint_as_float(pk[j] << 16), w1 = __uint_as_float(pk[j] & 0xffff0000u);
            l_lo += sc[0] > 0.f ? w0 / sc[0] : 0.f;
            l_hi += sc[1] > 0.f ? w1 / sc[1] : 0.f;
          }
        }
        tmem_st16(tS + half * 32 + c2 * 16, pk);
      }
      l += l_lo + l_hi;
      // rescale this warp's half of O (after P is stored): the previous
      // block's P.V must have landed first; P.V of this block waits for the
      // arrivals below
      if (__any_sync(0xffffffffu, need)) {
        if (!mbar_wait(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, flags)) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < DVH / 32; ++cc) {
          uint32_t r[32];
          const uint32_t col = uint32_t(half * DVH + cc * 32);
          tmem_ld32(tmem + lane_off + col, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          tmem_st32(tmem + lane_off + col, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[n & 1]);
    }
    if (alive && nb >= 1) {
      alive = mbar_wait(&pv_done[(nb - 1) & 1], ((nb - 1) >> 1) & 1, flags);
      tc_fence_after();
    }
    // the combine may be scheduled now (it waits for this grid to finish)
    if (warp == 2 && lane == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // ---------------- epilogue: the pair's partial sums, then each warp
    // writes its half of the row's value columns
    float l_row = l;
    if (alive) alive = pair_sync();  // both warps are past their last read of the maxima
    if (alive) {
      xsum[half * kAttnBM + lrow] = l;
      alive = pair_sync();
      l_row = l + xsum[(half ^ 1) * kAttnBM + lrow];
    }
    if (alive) {
      const int h = hk * a.G + g;
      if (a.nsplit == 1) {
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        __nv_bfloat16* dst = a.out + ((size_t)b * a.C + i) * a.Hq * a.d + (size_t)h * a.d + dvp * K::DV + half * DVH;
        for (int cc = 0; cc < DVH / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + uint32_t(half * DVH + cc * 32), r);
          tmem_ld_wait();
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
            uint4* o4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) o4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
        if (valid && dvp == 0 && half == 0 && a.lse != nullptr)
          a.lse[((size_t)b * a.C + i) * a.Hq + h] = l_row > 0.f ? (m_run + log2f(l_row)) * kLn2 : -INFINITY;
      } else {
        const size_t prow = ((size_t)split * a.B * a.Hkv + grp) * (size_t)(a.q_tiles * kAttnBM) + qt * kAttnBM + lrow;
        float* dst = a.part_o + prow * a.d + dvp * K::DV + half * DVH;
        for (int cc = 0; cc < DVH / 32; ++cc) {
          uint32_t r[32];
          if (nb >= 1) {
            tmem_ld32(tmem + lane_off + uint32_t(half * DVH + cc * 32), r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
          float4* o4 = reinterpret_cast<float4*>(dst + cc * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            o4[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                                __uint_as_float(r[4 * j + 3]));
        }
        if (dvp == 0 && half == 0) {
          a.part_ml[prow * 2] = m_run;
          a.part_ml[prow * 2 + 1] = l_row;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// d = 512 on four SMs: a cluster of two CTA pairs, no duplicated MMA work.
//
// The cluster owns 256 query rows (CTA h of each pair: rows 128 h .. 128 h +
// 127).  Pair p forms S only for key half p of every 128-key block (64 keys,
// M = 256 MMAs issued by the pair's leader, rank 2 p) and accumulates only
// value half p of O (256 columns).  The CTAs with the same rows in the two
// pairs (ranks r and r ^ 2) agree on each block's row maximum by swapping
// their half maxima, and each sends its bf16 P to the other with st.async
// into shared memory, so both pairs form O over all 128 keys:
//   O_p += P_own V[own keys, half p]   (P from TMEM, where the softmax wrote it)
//        + P_other V[other keys, half p]  (P from shared memory).
// NS S buffers: with three, the softmax of a block (with its two exchanges
// between CTAs) overlaps the MMAs of the next two blocks, a quarter of Q
// (d 0..127) sits in TMEM and the ring has three stages; with two, half of Q
// sits in TMEM and the ring has four stages (two blocks of K and V in flight).
// TMEM columns: O [0, 256), S / P NS x 64 from 256, Q at 256 + 64 NS.
// The ring is split in two: NST - VS stages of K, loaded by warp 0 in block
// order, and VS stages of V, loaded by warp 6 -- so the keys of the next
// blocks' S are fetched as soon as an S has consumed its stage, without
// queueing behind the values of the current block.  With two V stages the
// values of block n + 1 load while block n's P.V waits for its P (with one,
// every block waited for its values to arrive after the previous P.V).
template <int NS, int VS>
struct Cfg4 {
  static constexpr int NST = NS == 2 ? 4 : 3;
  static constexpr int KR = NST - VS;  // K stages [0, KR), V stages [KR, NST)
  static_assert(VS >= 1 && KR >= 2, "ring split");
  static constexpr int QT = NS == 2 ? 4 : 2;        // 64-wide chunks of Q held in TMEM
  static constexpr int QSBytes = (8 - QT) * 16384;  // the other chunks in shared memory (128 rows each)
  static constexpr int POBytes = 16384;      // the partner's P: 128 rows x 64 keys bf16
  static constexpr int Smem = QSBytes + 2 * POBytes + NST * kStageBytes + 1024 + kBarBytes + 1024;
};
constexpr int kThreads4 = 224;  // K TMA warp, MMA warp, 4 softmax / epilogue warps, V TMA warp

template <int NS, int VS>
__global__ void __launch_bounds__(kThreads4, 1)
    attention_tc4_kernel(const __grid_constant__ AttnTcMaps maps, AttnTcArgs a) {
  using K = Cfg4<NS, VS>;
  constexpr int D = 512;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sPO = smem + K::QSBytes;  // [2] partner's P
  uint8_t* ring = sPO + 2 * K::POBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + K::NST * kStageBytes);
  uint64_t* empty = full + K::NST;
  uint64_t* q_full = empty + K::NST;
  uint64_t* qt_ready = q_full + 1;
  uint64_t* s_full = qt_ready + 1;  // [NS]
  uint64_t* p_full = s_full + NS;   // [NS] (pair leader) this pair's P in TMEM
  uint64_t* px_full = p_full + NS;  // [NS] (pair leader) the other pair's P in shared memory
  uint64_t* pv_done = px_full + NS; // [2] both pairs' P.V of a block
  uint64_t* mx_full = pv_done + 2;  // [2] the partner's maxima (and, last, its sums)
  uint64_t* po_full = mx_full + 2;  // [2] the partner's P
  uint64_t* drain = po_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort
  static_assert((2 * K::NST + 2 + 3 * NS + 2 * 3 + 1) * 8 + 8 <= kBarBytes, "barrier area");
  uint32_t* xin = reinterpret_cast<uint32_t*>(ring + K::NST * kStageBytes + kBarBytes);  // [2][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pp = int(rank >> 1), h = int(rank & 1);
  const bool leader = h == 0;
  const uint32_t lead_rank = rank & 2u, partner = rank ^ 2u;
  const uint16_t pair_mask = uint16_t(3u << lead_rank);
  int x = blockIdx.x >> 2;
  const int q_pairs = (a.q_tiles + 1) / 2;
  const int qp = x % q_pairs;
  x /= q_pairs;
  const int split = x % a.nsplit;
  x /= a.nsplit;
  const int hk = x % a.Hkv;
  const int b = x / a.Hkv;
  const int grp = b * a.Hkv + hk;
  const int qt = 2 * qp + h;
  const Seq sq = make_seq(a, b, qp, split, 2 * kAttnBM);
  if (!sq.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(CANVAS_ERR_BOUNDS);
    return;  // uniform over the cluster: before any barrier or TMEM allocation
  }
  const int nb = sq.nb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < K::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(qt_ready, 8);  // the softmax warps of both CTAs of the pair
    for (int j = 0; j < NS; ++j) {
      mbar_init(&s_full[j], 1);
      mbar_init(&p_full[j], 8);
      mbar_init(&px_full[j], 8);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&pv_done[j], 2);  // one commit from each pair's leader
      mbar_init(&mx_full[j], 1);
      mbar_init(&po_full[j], 1);
    }
    mbar_init(drain, 1);
    flags[0] = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.kpre_c);
    tma_prefetch_desc(&maps.vpre_c);
    tma_prefetch_desc(&maps.kx_c);
    tma_prefetch_desc(&maps.vx_c);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of all four CTAs initialised, TMEM allocated in both pairs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t kColS = 256, kColQ = 256 + 64 * NS;

  constexpr int KR = K::KR;
  auto row_of = [&](int sb, bool key, const CUtensorMap*& map) -> int {
    if (sb < sq.n_pre) {
      const int pos = sq.s0 + 64 * sb;
      map = key ? &maps.kpre_c : &maps.vpre_c;
      return (key && !a.kpre_paged) ? grp * a.max_prefix + pos : paged_row(a, b, hk, pos);
    }
    map = key ? &maps.kx_c : &maps.vx_c;
    return grp * a.Tpad + 64 * (sb - sq.n_pre);
  };
  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producers (every CTA): K (warp 0), V (warp 6)
      const bool kp = warp == 0;
      const int nst = kp ? KR : VS, s0 = kp ? 0 : KR;
      if (kp) {
        const uint32_t lead_q = mapa_shared(smem_u32(q_full), lead_rank);
        if (leader) mbar_arrive_expect_tx(q_full, uint32_t(2 * K::QSBytes));
        const int qrow = grp * a.G * a.C + qt * kAttnBM;
        for (int c = 0; c < 8 - K::QT; ++c) tma_load_2d_pair(sQ + c * 16384, &maps.q, lead_q, (K::QT + c) * 64, qrow);
      }
      int n = 0;
      for (; n < nb; ++n) {
        const int s = s0 + n % nst;
        if (!mbar_wait(&empty[s], ((n / nst) & 1) ^ 1, flags)) break;
        if (leader) mbar_arrive_expect_tx(&full[s], uint32_t(2 * kStageBytes));
        uint8_t* dst = ring + s * kStageBytes;
        const uint32_t bar = mapa_shared(smem_u32(&full[s]), lead_rank);
        if (kp) {
          // this CTA's 32 keys of the pair's key half, all of d: 8 chunks of
          // 4 KB in one copy
          const CUtensorMap* map;
          const int row = row_of(2 * (sq.kb0 + n) + pp, true, map) + 32 * h;
          tma_load_3d_pair(dst, map, bar, 0, row, 0);
        } else {
          // all 128 keys of block n, this CTA's 128 columns of value half pp:
          // per 64-key sub-block u one copy of two 64-column chunks (16 KB at
          // u * 16 KB, chunk after chunk)
          for (int u = 0; u < 2; ++u) {
            const CUtensorMap* map;
            const int row = row_of(2 * (sq.kb0 + n) + u, false, map);
            tma_load_3d_pair(dst + u * 16384, map, bar, 0, row, pp * 4 + h * 2);
          }
        }
      }
      if (leader) {
        // drain: every stage's bytes -- both CTAs' -- have landed
        volatile int no_abort = 0;
        if (kp) mbar_wait(q_full, 0, &no_abort);
        for (int j = max(0, n - nst); j < n; ++j) mbar_wait(&full[s0 + j % nst], (j / nst) & 1, &no_abort);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer (pair leader)
      const uint32_t idesc_qk = idesc_bf16_f32(256, 64, 0, 0);
      const uint32_t idesc_pv = idesc_bf16_f32(256, 256, 0, 1);
      const uint32_t q_base = smem_u32(sQ);
      bool alive = mbar_wait(q_full, 0, flags) && mbar_wait(qt_ready, 0, flags);
      tc_fence_after();
      // K of block n: stage n % KR; V of block n: stage KR + n % VS
      auto consume = [&](int n, bool key) -> uint32_t {
        const int s = key ? n % KR : KR + n % VS;
        const uint32_t par = key ? (n / KR) & 1 : (n / VS) & 1;
        if (!mbar_wait(&full[s], par, flags)) {
          alive = false;
          return 0;
        }
        tc_fence_after();
        return smem_u32(ring + s * kStageBytes);
      };
      // descriptors advance by (byte offset >> 4) in their start-address
      // field, so each MMA adds a constant to a base computed once
      const uint64_t q_desc0 = smem_desc_sw128(q_base, 16, 1024);
      auto qk = [&](int n) {
        const uint32_t tS = tmem + kColS + (n % NS) * 64;
        const uint32_t st = consume(n, true);
        if (!alive) return;
        const uint64_t b_desc0 = smem_desc_sw128(st, 16, 1024);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = b_desc0 + uint64_t((ch * 4096 + kk * 32) >> 4);
            const uint32_t acc = (ch | kk) != 0 ? 1u : 0u;
            if (ch < K::QT)
              mma2_bf16_ts(tS, tmem + kColQ + ch * 32 + kk * 8, bd, idesc_qk, acc);
            else
              mma2_bf16_ss(tS, q_desc0 + uint64_t(((ch - K::QT) * 16384 + kk * 32) >> 4), bd, idesc_qk, acc);
          }
        }
        mma2_commit_mc(&empty[n % KR], pair_mask);
        mma2_commit_mc(&s_full[n % NS], pair_mask);
      };
      const uint64_t po_desc0 = smem_desc_sw128(smem_u32(sPO), 16, 1024);
      auto pv = [&](int n) {
        const uint32_t tS = tmem + kColS + (n % NS) * 64;
        const uint32_t st = consume(n, false);
        if (!alive) return;
        const uint64_t v_desc0 = smem_desc_sw128(st, 8192, 1024);
        const uint64_t a_desc0 = po_desc0 + uint64_t(((n & 1) * K::POBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma2_bf16_ts(tmem, tS + kk * 8, v_desc0 + uint64_t((pp * 16384 + kk * 2048) >> 4), idesc_pv,
                       (n | kk) != 0 ? 1u : 0u);
        // the other pair's keys once its P has landed in both CTAs
        if (!mbar_wait(&px_full[n % NS], (n / NS) & 1, flags)) {
          alive = false;
          return;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma2_bf16_ss(tmem, a_desc0 + uint64_t((kk * 32) >> 4),
                       v_desc0 + uint64_t(((1 - pp) * 16384 + kk * 2048) >> 4), idesc_pv, 1u);
        mma2_commit_mc(&empty[KR + n % VS], pair_mask);
        mma2_commit_mc(&pv_done[n & 1], 0xF);
      };
      for (int n = 0; n < NS && n < nb && alive; ++n) qk(n);
      for (int n = 0; n < nb && alive; ++n) {
        if (!mbar_wait(&p_full[n % NS], (n / NS) & 1, flags)) break;
        tc_fence_after();
        pv(n);
        if (n + NS < nb) qk(n + NS);
      }
      // every MMA has completed in both CTAs of the pair before either releases TMEM
      mma2_commit_mc(drain, pair_mask);
    }
    if (lane == 0) {
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort);
    }
  } else {
    // ------------------------------------------------ softmax + epilogue (every CTA)
    const int quad = warp & 3;
    const int lrow = quad * 32 + lane;
    const uint32_t lane_off = uint32_t(quad * 32) << 16;
    const int GC = a.G * a.C;
    const int R = qt * kAttnBM + lrow;
    const bool valid = R < GC;
    const int g = valid ? R / a.C : 0, i = valid ? R % a.C : 0;
    const int lo_row = valid ? window_lo(a, sq.P, i) : 0;
    const bool counter = warp == 2 && lane == 0;  // posts this CTA's expected exchange bytes
    // remote addresses; the second barrier of each pair sits 8 bytes after the first
    const uint32_t lead_p0 = mapa_shared(smem_u32(&p_full[0]), lead_rank);    // [NS]
    const uint32_t lead_px0 = mapa_shared(smem_u32(&px_full[0]), lead_rank);  // [NS]
    const uint32_t peer_mx0 = mapa_shared(smem_u32(&mx_full[0]), partner);
    const uint32_t peer_po0 = mapa_shared(smem_u32(&po_full[0]), partner);
    const uint32_t peer_xin = mapa_shared(smem_u32(xin), partner);
    const uint32_t peer_sPO = mapa_shared(smem_u32(sPO), partner);
    // the first QT chunks of this row's Q into TMEM (zeros past the last row of the group)
    {
      const uint4* src = reinterpret_cast<const uint4*>(a.Qp + ((size_t)grp * GC + (valid ? R : 0)) * D);
#pragma unroll 1
      for (int ch = 0; ch < K::QT; ++ch) {
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 u = valid ? src[ch * 8 + j] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * j] = u.x;
          w[4 * j + 1] = u.y;
          w[4 * j + 2] = u.z;
          w[4 * j + 3] = u.w;
        }
        tmem_st32(tmem + lane_off + kColQ + ch * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(qt_ready), lead_rank));
    }
    float m_run = -INFINITY, l = 0.f;
    bool alive = true;
    for (int n = 0; n < nb; ++n) {
      const int buf = n & 1;
      const uint32_t ph = (n >> 1) & 1;
      if (counter) {
        mbar_arrive_expect_tx(&mx_full[buf], 4u * kAttnBM);
        mbar_arrive_expect_tx(&po_full[buf], uint32_t(K::POBytes));
      }
      const int sbuf = n % NS;
      if (!mbar_wait(&s_full[sbuf], (n / NS) & 1, flags)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + kColS + sbuf * 64;
      const int sb = 2 * (sq.kb0 + n) + pp;
      int pos0, hi_off = 64;
      if (sb < sq.n_pre) {
        pos0 = sq.s0 + 64 * sb;
      } else {
        const int t0 = 64 * (sb - sq.n_pre);
        pos0 = sq.P64 + t0;
        hi_off = min(64, sq.T - t0);
      }
      // encode mode: canvas keys up to the row's own position
      if (a.causal && valid) hi_off = min(hi_off, sq.P + i + 1 - pos0);
      const int lo_off = max(0, lo_row - pos0);
      uint32_t sv[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld_wait();
      if (__any_sync(0xffffffffu, lo_off > 0 || hi_off < 64)) {
#pragma unroll
        for (int off = 0; off < 64; ++off)
          if (off < lo_off || off >= hi_off) sv[off] = __float_as_uint(-INFINITY);
      }
      float mx[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        mx[c] = fmaxf(fmaxf(__uint_as_float(sv[c]), __uint_as_float(sv[c + 16])),
                      fmaxf(__uint_as_float(sv[c + 32]), __uint_as_float(sv[c + 48])));
#pragma unroll
      for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
      float smax = mx[0];
      // the two key halves agree on the block maximum (rounded up to bf16)
      const uint32_t mine = bf16_bits_up(smax);
      st_async_b32(peer_xin + uint32_t((buf * kAttnBM + lrow) * 4), mine, peer_mx0 + 8u * buf);
      if (!mbar_wait(&mx_full[buf], ph, flags)) {
        alive = false;
        break;
      }
      const uint32_t other = xin[buf * kAttnBM + lrow];
      smax = fmaxf(bf16_bits_to_f32(mine), bf16_bits_to_f32(other));
      const float bmax = smax * a.c_log2;
      const float m_new = fmaxf(m_run, bmax);
      const bool need = (m_run != -INFINITY) && (m_new > m_run + kRescaleLog2);
      const float alpha = need ? exp2f(m_run - m_new) : 1.f;
      if (need) {
        l *= alpha;
        m_run = m_new;
      } else if (m_run == -INFINITY) {
        m_run = m_new;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // P = 2^(S c - m) rounded to bf16, and its row sum (the normaliser
      // matches what P.V consumes)
      uint32_t pk[32];
      float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = 2 * j;
        const float p0 = ex2_approx(fmaf(__uint_as_float(sv[c]), a.c_log2, -m_use));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sv[c + 1]), a.c_log2, -m_use));
        if (a.vs_pre == nullptr) {
          pk[j] = pack_bf16x2(p0, p1);
          l_lo += __uint_as_float(pk[j] << 16);
          l_hi += __uint_as_float(pk[j] & 0xffff0000u);
        } else {
          float sc[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int off = c + e;
            sc[e] = sb < sq.n_pre ? a.vs_pre[(size_t)grp * a.max_prefix + pos0 + off]
                                  : a.vs_tail[(size_t)grp * a.Tpad + (pos0 - sq.P64) + off];
          }
          pk[j] = pack_bf16x2(p0 * sc[0], p1 * sc[1]);
          const float w0 = __uint_as_float(pk[j] << 16), w1 = __uint_as_float(pk[j] & 0xffff0000u);
          l_lo += sc[0] > 0.f ? w0 / sc[0] : 0.f;
          l_hi += sc[1] > 0.f ? w1 / sc[1] : 0.f;
        }
      }
      l += l_lo + l_hi;
      tmem_st16(tS, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
      tmem_st16(tS + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
      // P to the partner: its buffer is free once both pairs' P.V of block n - 2 finished
      if (n >= 2 && !mbar_wait(&pv_done[buf], ((n - 2) >> 1) & 1, flags)) {
        alive = false;
        break;
      }
      {
        const uint32_t row_addr = peer_sPO + uint32_t(buf * K::POBytes + lrow * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_async_v4(row_addr + uint32_t((j ^ (lrow & 7)) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                      pk[4 * j + 3], peer_po0 + 8u * buf);
      }
      if (__any_sync(0xffffffffu, need)) {
        if (!mbar_wait(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, flags)) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + uint32_t(cc * 32), r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          tmem_st32(tmem + lane_off + uint32_t(cc * 32), r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(lead_p0 + 8u * sbuf);  // P.V over this pair's keys
      // the partner's P has landed in this CTA's shared memory
      if (!mbar_wait(&po_full[buf], ph, flags)) {
        alive = false;
        break;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(lead_px0 + 8u * sbuf);  // P.V over the other pair's keys
    }
    if (alive && nb >= 1) {
      alive = mbar_wait(&pv_done[(nb - 1) & 1], ((nb - 1) >> 1) & 1, flags);
      tc_fence_after();
    }
    // the combine may be scheduled now (it waits for this grid to finish)
    if (warp == 2 && lane == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the two key halves' sums, through the exchange slot of block nb
    float l_row = l;
    if (alive) {
      const int buf = nb & 1;
      if (counter) mbar_arrive_expect_tx(&mx_full[buf], 4u * kAttnBM);
      st_async_b32(peer_xin + uint32_t((buf * kAttnBM + lrow) * 4), __float_as_uint(l), peer_mx0 + 8u * buf);
      alive = mbar_wait(&mx_full[buf], (nb >> 1) & 1, flags);
      if (alive) l_row = l + __uint_as_float(xin[buf * kAttnBM + lrow]);
    }
    if (alive) {
      const int hq = hk * a.G + g;
      if (a.nsplit == 1) {
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        __nv_bfloat16* dst = a.out + ((size_t)b * a.C + i) * a.Hq * a.d + (size_t)hq * a.d + pp * 256;
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + uint32_t(cc * 32), r);
          tmem_ld_wait();
          if (valid) {
            uint32_t o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              o[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
            uint4* o4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) o4[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
        if (valid && pp == 0 && a.lse != nullptr)
          a.lse[((size_t)b * a.C + i) * a.Hq + hq] = l_row > 0.f ? (m_run + log2f(l_row)) * kLn2 : -INFINITY;
      } else if (qt < a.q_tiles) {
        const size_t prow = ((size_t)split * a.B * a.Hkv + grp) * (size_t)(a.q_tiles * kAttnBM) + qt * kAttnBM + lrow;
        float* dst = a.part_o + prow * a.d + pp * 256;
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t r[32];
          if (nb >= 1) {
            tmem_ld32(tmem + lane_off + uint32_t(cc * 32), r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
          float4* o4 = reinterpret_cast<float4*>(dst + cc * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            o4[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
        if (pp == 0) {
          a.part_ml[prow * 2] = m_run;
          a.part_ml[prow * 2 + 1] = l_row;
        }
      }
    }
  }
  tc_fence_before();
  cluster_sync_all();  // all four CTAs done with TMEM and with each other's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// One warp per output row (b, KV head, packed row g*C + i), eight rows per
// block: merges the KV splits' partial rows by their running max and sum.
// Lane s reads split s's (max, sum) and the warp shares them; each lane then
// owns four consecutive columns per 128-column step and issues the loads of
// every split before it adds them (in split order).
constexpr int kMaxCombineSplits = 32;
__global__ void __launch_bounds__(256) attention_combine_kernel(AttnTcArgs a) {
  // launched as a programmatic dependent of the attention kernel: wait for
  // all of its blocks and their stores before reading the partials
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int GC = a.G * a.C;
  const int lane = threadIdx.x & 31;
  const long long wrow = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wrow >= (long long)a.B * a.Hkv * GC) return;
  const int row = int(wrow % GC);
  const int grp = int(wrow / GC);
  const int b = grp / a.Hkv, hk = grp % a.Hkv;
  const int g = row / a.C, i = row % a.C;
  const size_t rows_per_split = (size_t)a.B * a.Hkv * a.q_tiles * kAttnBM;
  const size_t prow0 = (size_t)grp * a.q_tiles * kAttnBM + row;
  const int ns = min(a.nsplit, kMaxCombineSplits);
  float ms = -INFINITY, ls = 0.f;
  if (lane < ns) {
    const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (lane * rows_per_split + prow0) * 2);
    ms = ml.x;
    ls = ml.y;
  }
  float M = ms;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  // this lane's split weight 2^(m_s - M) (0 for an empty split), summed in split order
  const float wl = ms == -INFINITY ? 0.f : exp2f(ms - M);
  float L = 0.f;
  for (int sp = 0; sp < ns; ++sp) L += __shfl_sync(0xffffffffu, wl * ls, sp);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int h = hk * a.G + g;
  __nv_bfloat16* dst = a.out + ((size_t)b * a.C + i) * a.Hq * a.d + (size_t)h * a.d;
  for (int c = lane * 4; c < a.d; c += 128) {
    float4 v[kMaxCombineSplits < 8 ? kMaxCombineSplits : 8];
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < ns; s0 += 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < ns)
          v[j] = *reinterpret_cast<const float4*>(a.part_o + ((s0 + j) * rows_per_split + prow0) * a.d + c);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = __shfl_sync(0xffffffffu, wl, (s0 + j) & 31);
        if (s0 + j < ns && w != 0.f) {
          o[0] = fmaf(w, v[j].x, o[0]);
          o[1] = fmaf(w, v[j].y, o[1]);
          o[2] = fmaf(w, v[j].z, o[2]);
          o[3] = fmaf(w, v[j].w, o[3]);
        }
      }
    }
    *reinterpret_cast<uint2*>(dst + c) = make_uint2(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv));
  }
  if (lane == 0 && a.lse != nullptr)
    a.lse[((size_t)b * a.C + i) * a.Hq + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <int D>
cudaError_t launch_d(const AttnTcMaps& maps, const AttnTcArgs& a, cudaStream_t stream) {
  static bool attr_set = false;
  const int smem = Cfg<D>::Smem;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = a.B * a.Hkv * a.nsplit * a.q_tiles * a.dv_parts;
  attention_tc_kernel<D><<<grid, kThreads, smem, stream>>>(maps, a);
  count_launches(1);
  return cudaGetLastError();
}

#ifndef CANVAS_QUAD_S_BUFFERS
#define CANVAS_QUAD_S_BUFFERS 2
#endif
#ifndef CANVAS_QUAD_V_STAGES
#define CANVAS_QUAD_V_STAGES 2
#endif
cudaError_t launch_quad(const AttnTcMaps& maps, const AttnTcArgs& a, cudaStream_t stream) {
  constexpr int NS = CANVAS_QUAD_S_BUFFERS, VS = CANVAS_QUAD_V_STAGES;
  static bool attr_set = false;
  const int smem = Cfg4<NS, VS>::Smem;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(attention_tc4_kernel<NS, VS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int clusters = a.B * a.Hkv * a.nsplit * ((a.q_tiles + 1) / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * clusters, 1, 1);
  cfg.blockDim = dim3(kThreads4, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attention_tc4_kernel<NS, VS>, maps, a);
  count_launches(1);
  return e;
}

}  // namespace

size_t attention_tc_smem_bytes(int d) {
  switch (d) {
    case 64: return Cfg<64>::Smem;
    case 128: return Cfg<128>::Smem;
    case 256: return Cfg<256>::Smem;
    case 512: return Cfg<512>::Smem;
    default: return 0;
  }
}

cudaError_t launch_attention_tc(const AttnTcMaps& maps, const AttnTcArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_d<64>(maps, a, stream);
    case 128: return launch_d<128>(maps, a, stream);
    case 256: return launch_d<256>(maps, a, stream);
    case 512: return a.pair == 2 ? launch_quad(maps, a, stream) : launch_d<512>(maps, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attention_combine(const AttnTcArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.B * a.Hkv * a.G * a.C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((rows + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, attention_combine_kernel, a);
  count_launches(1);
  return e;
}

}  // namespace canvas

// api.cu -- the C ABI of libcanvas.so (declared in include/canvas.h):
// argument validation, workspace layout, tensor-map encoding and the launch
// sequence of each call.  No call allocates device memory or synchronises
// (except canvas_device_status).
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

namespace canvas {

__device__ int g_status = 0;

namespace {
std::atomic<unsigned long long> g_launches{0};
}
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

thread_local std::string t_last_error;

// A side stream (non-blocking) and a fork / join event pair per host thread
// and device, created on first use and kept for the life of the thread: work
// that does not depend on the call's earlier kernels runs beside them, and
// the call's stream waits for it before anything that needs it.  Recording
// and waiting on events brings the side stream into a stream capture like
// any fork / join.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool tried = false;
};
constexpr int kMaxSideDevices = 64;
thread_local SideStream t_side[kMaxSideDevices];

SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return nullptr;
  SideStream& x = t_side[dev];
  if (!x.tried) {
    x.tried = true;
    if (cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();  // not sticky: the calls then run everything in order on their stream
      x.s = nullptr;
    }
  }
  return x.s ? &x : nullptr;
}

// per-thread timing events (canvas_profile_events)
struct EventPair {
  cudaEvent_t start = nullptr, stop = nullptr;
};
thread_local EventPair t_events[CANVAS_KERNEL_COUNT];

// NVTX: a range around every compute call of the C ABI and one per timed
// phase inside it (host-side markers; free when no tool is attached)
const char* const kPhaseName[CANVAS_KERNEL_COUNT] = {"attention_core", "attention_prep", "sampler", "soft_emb_gemm"};
static_assert(CANVAS_KERNEL_ATTENTION == 0 && CANVAS_KERNEL_PREP == 1 && CANVAS_KERNEL_SAMPLER == 2 &&
                  CANVAS_KERNEL_SOFT_EMB == 3,
              "phase names follow the timing ids");
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

inline void mark_start(int id, cudaStream_t s) {
  nvtxRangePushA(kPhaseName[id]);
  if (t_events[id].start) cudaEventRecord(t_events[id].start, s);
}
inline void mark_stop(int id, cudaStream_t s) {
  if (t_events[id].stop) cudaEventRecord(t_events[id].stop, s);
  nvtxRangePop();
}

canvas_status fail(canvas_status code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
canvas_status fail(canvas_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

canvas_status cuda_fail(cudaError_t e, const char* where) {
  return fail(CANVAS_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define CANVAS_CUDA(call)                                   \
  do {                                                      \
    cudaError_t e_ = (call);                                \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);     \
  } while (0)

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Carves a caller-owned workspace into aligned regions.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* p) : base(static_cast<char*>(p)) {}
  template <typename T>
  T* take(size_t bytes) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align_up(off + bytes);
    return p;
  }
};

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2D bf16 tensor [rows][cols] (cols contiguous), box {box_cols, box_rows},
// 128-byte swizzle, zero fill outside the tensor.
canvas_status make_map_bf16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                            uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0)
    return fail(CANVAS_ERR_ARG, "tensor base address must be 16-byte aligned");
  if ((cols * 2) % 16 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "row pitch must be a multiple of 16 bytes");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return CANVAS_OK;
}

// The same bf16 [rows][cols] tensor seen as [cols / 64][rows][64] (dimension
// strides: row = the row pitch, chunk = 128 bytes), box {64, box_rows,
// box_chunks}: one copy lands box_chunks 64-column tiles of box_rows rows,
// tile after tile, each laid out (and 128-byte swizzled) exactly as a 2D box
// of {64, box_rows} would be.
canvas_status make_map_bf16_chunked(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                                    uint32_t box_rows, uint32_t box_chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0)
    return fail(CANVAS_ERR_ARG, "tensor base address must be 16-byte aligned");
  if (cols % 64 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "chunked view needs a multiple of 64 columns");
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled (chunked view) failed (%d)", int(r));
  return CANVAS_OK;
}

// fp32 [z][rows][cols] (row pitch ld elements, slab pitch rows * ld) for TMA
// stores of 32 x 32 boxes with the 128-byte swizzle; stores clip at every
// edge, so no box spills into the next row block or slab.
canvas_status make_map_f32_store(CUtensorMap* map, void* ptr, uint64_t z, uint64_t rows, uint64_t cols, uint64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0)
    return fail(CANVAS_ERR_ARG, "output base address must be 16-byte aligned");
  if ((ld * 4) % 16 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "output row pitch must be a multiple of 16 bytes");
  cuuint64_t dims[3] = {cols, rows, z};
  cuuint64_t strides[2] = {ld * 4, rows * ld * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled (store) failed (%d)", int(r));
  return CANVAS_OK;
}

// bf16 [z][rows][cols] for TMA stores of 32-row x 64-column boxes (128-byte rows, 128-byte swizzle)
canvas_status make_map_bf16_store(CUtensorMap* map, void* ptr, uint64_t z, uint64_t rows, uint64_t cols, uint64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0)
    return fail(CANVAS_ERR_ARG, "output base address must be 16-byte aligned");
  if ((ld * 2) % 16 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "output row pitch must be a multiple of 16 bytes");
  cuuint64_t dims[3] = {cols, rows, z};
  cuuint64_t strides[2] = {ld * 2, rows * ld * 2};
  cuuint32_t box[3] = {64, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CANVAS_ERR_CUDA, "cuTensorMapEncodeTiled (bf16 store) failed (%d)", int(r));
  return CANVAS_OK;
}

// ------------------------------------------------------------------ GEMM plan
struct GemmPlan {
  int m_tiles, n_tiles, kblocks, splits, two_acc;
  size_t partial_bytes;  // all problems, each slab 256-byte aligned
};

constexpr int kNumSms = 148;

// One launch for nprob problems C_p[M, N_p] = A[M, K] op(B_p).
GemmPlan plan_gemm_group(int M, const int* N, int nprob, int K) {
  GemmPlan p;
  p.two_acc = M > kGemmBM ? 1 : 0;
  p.m_tiles = (M + 255) / 256;
  p.n_tiles = 0;
  for (int i = 0; i < nprob; ++i) p.n_tiles += (N[i] + kGemmBN - 1) / kGemmBN;
  p.kblocks = (K + kGemmBK - 1) / kGemmBK;
  const int tiles = p.m_tiles * p.n_tiles;
  int s = tiles >= kNumSms ? 1 : kNumSms / tiles;
  // at least 8 K blocks per split: shorter splits are dominated by the
  // pipeline fill and by writing their fp32 partial tile
  s = std::min(s, std::max(1, p.kblocks / 8));
  p.splits = std::max(1, s);
  p.partial_bytes = 0;
  if (p.splits > 1)
    for (int i = 0; i < nprob; ++i) p.partial_bytes += align_up(size_t(p.splits) * M * N[i] * sizeof(float));
  return p;
}

GemmPlan plan_gemm(int M, int N, int K) { return plan_gemm_group(M, &N, 1, K); }

size_t gemm_ws_bytes(const GemmPlan& p) { return align_up(p.partial_bytes); }

// C_p[M, N_p] = A[M, K] op(B_p) (+ C_p) for p < nprob on the tensor cores, in
// one launch; C fp32, or bf16 with out_bf16 (no accumulate); ws holds the
// split partials.
canvas_status run_gemm_group(const void* A, const void* const* B, void* const* C, const int* N, int nprob,
                             int b_mn_major, int M, int K, int accumulate, int out_bf16, void* ws,
                             cudaStream_t stream, float** partials_out = nullptr, int* splits_out = nullptr) {
  if (nprob < 1 || nprob > kGemmMaxProblems) return fail(CANVAS_ERR_ARG, "GEMM: 1 to 3 problems per launch");
  const GemmPlan p = plan_gemm_group(M, N, nprob, K);
  GemmTcMaps maps;
  GemmTcArgs g;
  canvas_status st = make_map_bf16(&maps.A, A, M, K, kGemmBM, kGemmBK);
  if (st != CANVAS_OK) return st;
  Carver cv(ws);
  g.tile0[0] = 0;
  for (int i = 0; i < nprob; ++i) {
    if (b_mn_major)
      st = make_map_bf16(&maps.B[i], B[i], K, N[i], 64, 64);
    else
      st = make_map_bf16(&maps.B[i], B[i], N[i], K, kGemmBN, kGemmBK);
    if (st != CANVAS_OK) return st;
    g.partials[i] = p.splits > 1 ? cv.take<float>(size_t(p.splits) * M * N[i] * sizeof(float)) : nullptr;
    if (p.splits > 1)
      st = make_map_f32_store(&maps.out[i], g.partials[i], uint64_t(p.splits), uint64_t(M), uint64_t(N[i]),
                              uint64_t(N[i]));
    else if (out_bf16)
      st = make_map_bf16_store(&maps.out[i], C[i], 1, uint64_t(M), uint64_t(N[i]), uint64_t(N[i]));
    else
      st = make_map_f32_store(&maps.out[i], C[i], 1, uint64_t(M), uint64_t(N[i]), uint64_t(N[i]));
    if (st != CANVAS_OK) return st;
    g.C[i] = C[i];
    g.N[i] = N[i];
    g.tile0[i + 1] = g.tile0[i] + (N[i] + kGemmBN - 1) / kGemmBN;
  }
  for (int i = nprob; i < kGemmMaxProblems; ++i) {
    maps.B[i] = maps.B[0];
    maps.out[i] = maps.out[0];
    g.C[i] = nullptr;
    g.partials[i] = nullptr;
    g.N[i] = 0;
    g.tile0[i + 1] = g.tile0[i];
  }
  g.M = M;
  g.K = K;
  g.kblocks = p.kblocks;
  g.splits = p.splits;
  g.accumulate = accumulate;
  g.out_bf16 = out_bf16;
  g.b_mn_major = b_mn_major;
  g.two_acc = p.two_acc;
  g.m_tiles = p.m_tiles;
  g.bm = 256;
  g.group_of_mtile = nullptr;
  g.nprob = nprob;
  // partials_out: the caller sums a split product's partials itself
  const bool reduce = partials_out == nullptr;
  CANVAS_CUDA(launch_gemm_tc(maps, g, stream, reduce));
  if (!reduce) {
    for (int i = 0; i < nprob; ++i) partials_out[i] = p.splits > 1 ? g.partials[i] : static_cast<float*>(C[i]);
    *splits_out = p.splits;
  }
  return CANVAS_OK;
}

canvas_status run_gemm_tc(const void* A, const void* B, int b_mn_major, float* C, int M, int N, int K,
                          int accumulate, void* ws, cudaStream_t stream) {
  void* Cv = C;
  return run_gemm_group(A, &B, &Cv, &N, 1, b_mn_major, M, K, accumulate, 0, ws, stream);
}

// Grouped products: C_p[Mpad, N_p] = A[Mpad, K] B_p[group(tile), N_p rows, K]^T
// for nprob problems sharing A, every 128-row tile of A in one group
// (group_of_mtile, device; -1: no work), B_p stored as [groups * N_p, K].
// One launch, no K split; C fp32, or bf16 with out_bf16.
canvas_status run_gemm_grouped(const void* A, const void* const* B, void* const* C, const int* N, int nprob,
                               int groups, const int* group_of_mtile, int Mpad, int K, int out_bf16,
                               cudaStream_t stream) {
  if (nprob < 1 || nprob > kGemmMaxProblems || Mpad % 128 != 0)
    return fail(CANVAS_ERR_ARG, "grouped GEMM: 1 to 3 problems, rows in whole 128-row tiles");
  GemmTcMaps maps;
  GemmTcArgs g;
  canvas_status st = make_map_bf16(&maps.A, A, Mpad, K, kGemmBM, kGemmBK);
  if (st != CANVAS_OK) return st;
  g.tile0[0] = 0;
  for (int i = 0; i < nprob; ++i) {
    st = make_map_bf16(&maps.B[i], B[i], uint64_t(groups) * N[i], K, kGemmBN, kGemmBK);
    if (st != CANVAS_OK) return st;
    st = out_bf16 ? make_map_bf16_store(&maps.out[i], C[i], 1, uint64_t(Mpad), uint64_t(N[i]), uint64_t(N[i]))
                  : make_map_f32_store(&maps.out[i], C[i], 1, uint64_t(Mpad), uint64_t(N[i]), uint64_t(N[i]));
    if (st != CANVAS_OK) return st;
    g.C[i] = C[i];
    g.N[i] = N[i];
    g.partials[i] = nullptr;
    g.tile0[i + 1] = g.tile0[i] + (N[i] + kGemmBN - 1) / kGemmBN;
  }
  for (int i = nprob; i < kGemmMaxProblems; ++i) {
    maps.B[i] = maps.B[0];
    maps.out[i] = maps.out[0];
    g.C[i] = nullptr;
    g.partials[i] = nullptr;
    g.N[i] = 0;
    g.tile0[i + 1] = g.tile0[i];
  }
  g.M = Mpad;
  g.K = K;
  g.kblocks = (K + kGemmBK - 1) / kGemmBK;
  g.splits = 1;
  g.accumulate = 0;
  g.out_bf16 = out_bf16;
  g.b_mn_major = 0;
  g.two_acc = 0;
  g.m_tiles = Mpad / 128;
  g.bm = 128;
  g.group_of_mtile = group_of_mtile;
  g.nprob = nprob;
  CANVAS_CUDA(launch_gemm_tc(maps, g, stream));
  return CANVAS_OK;
}

// ------------------------------------------------------------------ attention layout
struct AttnPlan {
  int Tpad, q_tiles, dv_parts, nsplit;
};

AttnPlan plan_attn(int dtype, int B, int C, int Hq, int Hkv, int d, int max_prefix, int layer_type, int window) {
  AttnPlan p;
  const int G = Hq / Hkv;
  p.Tpad = attn_tail_rows(C);
  p.q_tiles = (G * C + kAttnBM - 1) / kAttnBM;
  p.dv_parts = d > 256 ? d / 256 : 1;
  p.nsplit = 1;
  if (dtype == CANVAS_BF16) {
    // enough CTAs to fill the SMs, at least two key blocks per split
    const int units = B * Hkv * p.q_tiles * p.dv_parts;
    int keys = max_prefix;
    if (layer_type == CANVAS_LAYER_SLIDING && window > 0) keys = std::min(keys, window + kAttnBM + 64);
    keys += 64 + p.Tpad;
    const int nblk = (keys + kAttnBN - 1) / kAttnBN;
    // (at most 32 splits: the combine holds one split per lane)
    p.nsplit = std::max(1, std::min(std::min(kNumSms / std::max(1, units), nblk / 2), 32));
  }
  return p;
}

struct AttnLayout {
  size_t proj_q, proj_k, proj_v, gemm, qp, kx, vx, vs_tail, kt, vs_pre, part_o, part_ml, total;
};

AttnLayout attn_layout(int dtype, int B, int C, int D, int Hq, int Hkv, int d, int max_prefix, int layer_type,
                       int window) {
  AttnLayout L;
  const AttnPlan pl = plan_attn(dtype, B, C, Hq, Hkv, d, max_prefix, layer_type, window);
  const size_t M = size_t(B) * C;
  const size_t es = dtype == CANVAS_BF16 ? 2 : 4;
  const bool global = layer_type == CANVAS_LAYER_GLOBAL;
  L.proj_q = M * Hq * d * 4;
  L.proj_k = M * Hkv * d * 4;
  L.proj_v = global ? 0 : M * Hkv * d * 4;
  L.gemm = 0;
  if (dtype == CANVAS_BF16) {
    const int Ns[3] = {Hq * d, Hkv * d, Hkv * d};
    L.gemm = gemm_ws_bytes(plan_gemm_group(int(M), Ns, global ? 2 : 3, D));
  }
  const size_t BH = size_t(B) * Hkv;
  L.qp = M * Hq * d * es;
  L.kx = BH * pl.Tpad * d * es;
  L.vx = L.kx;
  L.vs_tail = global ? BH * pl.Tpad * 4 : 0;
  L.kt = global ? BH * max_prefix * d * es : 0;
  L.vs_pre = global ? BH * max_prefix * 4 : 0;
  L.part_o = pl.nsplit > 1 ? size_t(pl.nsplit) * BH * pl.q_tiles * kAttnBM * d * 4 : 0;
  L.part_ml = pl.nsplit > 1 ? size_t(pl.nsplit) * BH * pl.q_tiles * kAttnBM * 2 * 4 : 0;
  L.total = align_up(L.proj_q) + align_up(L.proj_k) + align_up(L.proj_v) + align_up(L.gemm) + align_up(L.qp) +
            align_up(L.kx) + align_up(L.vx) + align_up(L.vs_tail) + align_up(L.kt) + align_up(L.vs_pre) +
            align_up(L.part_o) + align_up(L.part_ml) + kAlign;
  return L;
}

bool attn_shape_ok(int dtype, int B, int C, int D, int Hq, int Hkv, int d, int max_prefix, int layer_type) {
  if (dtype != CANVAS_BF16 && dtype != CANVAS_FP32) return false;
  if (B < 1 || C < 1 || D < 1 || Hq < 1 || Hkv < 1 || d < 2 || max_prefix < 0) return false;
  if (Hq % Hkv != 0 || Hq / Hkv > 32) return false;
  if (layer_type != CANVAS_LAYER_SLIDING && layer_type != CANVAS_LAYER_GLOBAL) return false;
  return true;
}

// ------------------------------------------------------------------ sampler layout
struct SampleLayout {
  size_t probs, argmax, gemm, states, total;
};

SampleLayout sample_layout(int dtype, int rows, int V, int D) {
  SampleLayout L;
  L.probs = size_t(rows) * V * (dtype == CANVAS_BF16 ? 2 : 4);
  L.argmax = size_t(rows) * 4;
  const GemmPlan gp = plan_gemm(rows, D, V);
  L.gemm = dtype == CANVAS_BF16 ? gemm_ws_bytes(gp) : 0;
  L.states = dtype == CANVAS_BF16 ? size_t(rows) * gp.splits * 8 * sizeof(float) : 0;
  L.total = align_up(L.probs) + align_up(L.argmax) + align_up(L.gemm) + align_up(L.states) + kAlign;
  return L;
}

// The deferred-normalisation sampler applies when nobody reads the stored
// probabilities themselves: bf16 logits, no probs_out, argmax commits, and a
// soft-embedding GEMM split along the vocabulary into ranges one CTA stages.
bool sample_deferred(int dtype, const void* probs_out, int commit_mode, const GemmPlan& gp) {
  if (dtype != CANVAS_BF16 || probs_out != nullptr || (commit_mode & 2) != 0) return false;
  if (gp.splits < 2 || gp.splits > kMaxSampleSlices) return false;
  const long long longest = (long long)(gp.kblocks / gp.splits + (gp.kblocks % gp.splits ? 1 : 0)) * 64;
  return longest <= kSampleSliceMaxElems;
}

bool ws_ok(const void* ws, size_t have, size_t need) {
  return ws != nullptr && have >= need && (reinterpret_cast<uintptr_t>(ws) % kAlign) == 0;
}

}  // namespace
}  // namespace canvas

using namespace canvas;

extern "C" {

const char* canvas_version(void) { return "canvas 0.1 (sm_103a)"; }

const char* canvas_last_error(void) { return t_last_error.c_str(); }

canvas_status canvas_profile_events(int kernel_id, void* start_event, void* stop_event) {
  if (kernel_id < 0 || kernel_id >= CANVAS_KERNEL_COUNT) return fail(CANVAS_ERR_ARG, "canvas_profile_events: kernel id");
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(CANVAS_ERR_ARG, "canvas_profile_events: pass both events or neither");
  t_events[kernel_id].start = static_cast<cudaEvent_t>(start_event);
  t_events[kernel_id].stop = static_cast<cudaEvent_t>(stop_event);
  return CANVAS_OK;
}

uint64_t canvas_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

canvas_status canvas_device_status(canvas_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(status)");
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(status)");
    return fail(canvas_status(v), "device status %d recorded by a kernel", v);
  }
  return CANVAS_OK;
}

canvas_status canvas_gelu_bf16(const float* in, void* out, size_t n, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_gelu_bf16");
  if (!in || !out) return fail(CANVAS_ERR_ARG, "canvas_gelu_bf16: null pointer");
  if (n % 8 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_gelu_bf16: n must be a multiple of 8");
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_gelu_bf16: pointers must be 16-byte aligned");
  if (n == 0) return CANVAS_OK;
  CANVAS_CUDA(launch_gelu_bf16(in, out, (long long)n, reinterpret_cast<cudaStream_t>(stream)));
  return CANVAS_OK;
}

canvas_status canvas_count_committed(const uint8_t* commit_mask, int rows, int canvas_len, int32_t* counts,
                                     canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_count_committed");
  if (!commit_mask || !counts) return fail(CANVAS_ERR_ARG, "canvas_count_committed: null pointer");
  if (rows < 1 || canvas_len < 1 || rows % canvas_len != 0)
    return fail(CANVAS_ERR_ARG, "canvas_count_committed: rows must be a multiple of canvas_len");
  CANVAS_CUDA(launch_count_committed(commit_mask, rows / canvas_len, canvas_len, counts,
                                     reinterpret_cast<cudaStream_t>(stream)));
  return CANVAS_OK;
}

float canvas_temperature_at(int step, int steps, float t_max, float t_min) {
  // linear from t_max at step 0 to t_min at step steps - 1 (one step: t_max)
  if (steps <= 1 || step <= 0) return t_max;
  if (step >= steps - 1) return t_min;
  const double f = double(step) / double(steps - 1);
  return float(double(t_max) + (double(t_min) - double(t_max)) * f);
}

canvas_status canvas_selftest_wait_timeout(canvas_stream_t stream) {
  CANVAS_CUDA(launch_wait_timeout_selftest(reinterpret_cast<cudaStream_t>(stream)));
  return CANVAS_OK;
}

size_t canvas_gemm_workspace_size(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 1) return 0;
  return gemm_ws_bytes(plan_gemm(M, N, K)) + kAlign;
}

canvas_status canvas_gemm_bf16(const void* A, const void* B, int b_layout, float* C, int M, int N, int K,
                               int accumulate, void* workspace, size_t ws_bytes, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_gemm_bf16");
  if (!A || !B || !C) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16: null pointer");
  if (M < 1 || N < 1 || K < 1) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16: bad shape");
  if (b_layout != 0 && b_layout != 1) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16: b_layout must be 0 or 1");
  if (K % 8 != 0 || N % 8 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_gemm_bf16: K and N must be multiples of 8");
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) % 16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16: A, B and C must be 16-byte aligned");
  if (!ws_ok(workspace, ws_bytes, canvas_gemm_workspace_size(M, N, K)))
    return fail(CANVAS_ERR_WORKSPACE, "canvas_gemm_bf16: workspace missing, small or misaligned");
  return run_gemm_tc(A, B, b_layout, C, M, N, K, accumulate, workspace, reinterpret_cast<cudaStream_t>(stream));
}

canvas_status canvas_gemm_bf16_to_bf16(const void* A, const void* B, int b_layout, void* C, int M, int N, int K,
                                       void* workspace, size_t ws_bytes, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_gemm_bf16_to_bf16");
  if (!A || !B || !C) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_to_bf16: null pointer");
  if (M < 1 || N < 1 || K < 1) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_to_bf16: bad shape");
  if (b_layout != 0 && b_layout != 1) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_to_bf16: b_layout must be 0 or 1");
  if (K % 8 != 0 || N % 8 != 0)
    return fail(CANVAS_ERR_UNSUPPORTED, "canvas_gemm_bf16_to_bf16: K and N must be multiples of 8");
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) % 16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_to_bf16: A, B and C must be 16-byte aligned");
  if (!ws_ok(workspace, ws_bytes, canvas_gemm_workspace_size(M, N, K)))
    return fail(CANVAS_ERR_WORKSPACE, "canvas_gemm_bf16_to_bf16: workspace missing, small or misaligned");
  void* Cv = C;
  return run_gemm_group(A, &B, &Cv, &N, 1, b_layout, M, K, 0, 1, workspace, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ loop glue
canvas_status canvas_embed_input(const int32_t* tokens, const void* E, const float* soft_emb, int rows, int D,
                                 int V, void* x, float* x32, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_embed_input");
  if (!tokens || !E || !x) return fail(CANVAS_ERR_ARG, "canvas_embed_input: null pointer");
  if (rows < 1 || D < 1 || V < 1) return fail(CANVAS_ERR_ARG, "canvas_embed_input: bad shape");
  if (D % 8 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_embed_input: D must be a multiple of 8");
  if ((reinterpret_cast<uintptr_t>(E) | reinterpret_cast<uintptr_t>(soft_emb) | reinterpret_cast<uintptr_t>(x) |
       reinterpret_cast<uintptr_t>(x32)) %
          16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_embed_input: E, soft_emb, x and x32 must be 16-byte aligned");
  CANVAS_CUDA(launch_embed_input(tokens, E, soft_emb, rows, D, V, x, x32, reinterpret_cast<cudaStream_t>(stream)));
  return CANVAS_OK;
}

canvas_status canvas_cast_bf16(const float* in, void* out, size_t n, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_cast_bf16");
  if (!in || !out) return fail(CANVAS_ERR_ARG, "canvas_cast_bf16: null pointer");
  if (n % 8 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_cast_bf16: n must be a multiple of 8");
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_cast_bf16: pointers must be 16-byte aligned");
  if (n == 0) return CANVAS_OK;
  CANVAS_CUDA(launch_cast_bf16(in, out, (long long)n, reinterpret_cast<cudaStream_t>(stream)));
  return CANVAS_OK;
}

// ------------------------------------------------------------------ GEMM without a workspace
// The split-K scratch of canvas_gemm_bf16_noalloc: one static device array,
// shared by every call on a device.  Host code cannot use the symbol as a
// pointer; its device address is looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CANVAS_GEMM_NOALLOC_SCRATCH_BYTES];

canvas_status canvas_gemm_bf16_noalloc(const void* A, const void* B, int b_layout, float* C, int M, int N, int K,
                                       int accumulate, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_gemm_bf16_noalloc");
  if (!A || !B || !C) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_noalloc: null pointer");
  if (M < 1 || N < 1 || K < 1) return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_noalloc: bad shape");
  if (b_layout != 0 && b_layout != 1)
    return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_noalloc: b_layout must be 0 or 1");
  if (K % 8 != 0 || N % 8 != 0)
    return fail(CANVAS_ERR_UNSUPPORTED, "canvas_gemm_bf16_noalloc: K and N must be multiples of 8");
  // C goes straight to the vectorised split reduce when K is split, so it is
  // checked here like A and B, before anything is enqueued
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) % 16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_gemm_bf16_noalloc: A, B and C must be 16-byte aligned");
  const size_t need = canvas_gemm_workspace_size(M, N, K);
  if (need > CANVAS_GEMM_NOALLOC_SCRATCH_BYTES)
    return fail(CANVAS_ERR_WORKSPACE,
                "canvas_gemm_bf16_noalloc: this shape needs %zu bytes of scratch, the static scratch holds %u "
                "(use canvas_gemm_bf16 with a workspace)",
                need, CANVAS_GEMM_NOALLOC_SCRATCH_BYTES);
  // device address of the static scratch, looked up once per device
  constexpr int kMaxDevices = 64;
  static void* scratch[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  CANVAS_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_gemm_bf16_noalloc: device id");
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (scratch[dev] == nullptr) {
      void* p = nullptr;
      CANVAS_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));
      scratch[dev] = p;
    }
    ws = scratch[dev];
  }
  // the scratch holds only split partials, fully rewritten by every call
  return run_gemm_tc(A, B, b_layout, C, M, N, K, accumulate, ws, reinterpret_cast<cudaStream_t>(stream));
}

size_t canvas_attention_workspace_size(int dtype, int B, int C, int D, int Hq, int Hkv, int d, int max_prefix,
                                       int layer_type) {
  if (!attn_shape_ok(dtype, B, C, D, Hq, Hkv, d, max_prefix, layer_type)) return 0;
  return attn_layout(dtype, B, C, D, Hq, Hkv, d, max_prefix, layer_type, 0).total;  // window 0: the largest plan
}

// canvas_attention (decode mode, causal = 0) and canvas_attention_encode
// (encode mode, causal = 1)
static canvas_status attention_impl(const void* x, int dtype, int B, int C, int D, const void* W_q, const void* W_k,
                             const void* W_v, int Hq, int Hkv, int d, const float* gamma_q, const float* gamma_k,
                             float eps, const float* freq, int layer_type, const canvas_kv_cache* kv,
                             const int32_t* prefix_len, int max_prefix, int window, float scale, int v_unit_rms,
                             void* out, float* lse, void* workspace, size_t ws_bytes, canvas_stream_t stream_,
                             int causal) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!attn_shape_ok(dtype, B, C, D, Hq, Hkv, d, max_prefix, layer_type))
    return fail(CANVAS_ERR_ARG, "canvas_attention: invalid shape or dtype");
  const bool global = layer_type == CANVAS_LAYER_GLOBAL;
  const bool bf16 = dtype == CANVAS_BF16;
  if (!x || !W_q || !W_k || !gamma_q || !gamma_k || !freq || !kv || !prefix_len || !out)
    return fail(CANVAS_ERR_ARG, "canvas_attention: null pointer");
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15) != 0)
    return fail(CANVAS_ERR_ARG, "canvas_attention: x and out must be 16-byte aligned");
  if (global && W_v != nullptr) return fail(CANVAS_ERR_ARG, "canvas_attention: global layers share W_v = W_k (pass NULL)");
  if (!global && W_v == nullptr) return fail(CANVAS_ERR_ARG, "canvas_attention: sliding layers need W_v");
  if (v_unit_rms && !global) return fail(CANVAS_ERR_ARG, "canvas_attention: v_unit_rms applies to global layers");
  if (!(scale > 0.f)) return fail(CANVAS_ERR_ARG, "canvas_attention: scale must be > 0");
  if (max_prefix > 0 && (!kv->k_pool || !kv->block_table)) return fail(CANVAS_ERR_ARG, "canvas_attention: cache pointers");
  if (max_prefix > 0 && !global && !kv->v_pool) return fail(CANVAS_ERR_ARG, "canvas_attention: sliding cache needs v_pool");
  if (global && kv->v_pool) return fail(CANVAS_ERR_ARG, "canvas_attention: global cache has no v_pool");
  if (max_prefix > 0 && (kv->page_tokens < 1 || kv->num_pages < 1 ||
                         (long long)kv->max_pages_per_seq * kv->page_tokens < max_prefix))
    return fail(CANVAS_ERR_ARG, "canvas_attention: cache geometry cannot hold max_prefix tokens");
  if (d % 64 != 0 || d > 512) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_attention: head_dim must be 64, 128, ..., 512");
  if (bf16 && (d & (d - 1)) != 0)
    return fail(CANVAS_ERR_UNSUPPORTED, "canvas_attention: bf16 head_dim must be 64, 128, 256 or 512");
  if (bf16 && D % 8 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_attention: d_model must be a multiple of 8");
  if (bf16 && max_prefix > 0 && kv->page_tokens % 64 != 0)
    return fail(CANVAS_ERR_UNSUPPORTED, "canvas_attention: bf16 page_tokens must be a multiple of 64");
  const AttnPlan pl = plan_attn(dtype, B, C, Hq, Hkv, d, max_prefix, layer_type, window);
  const AttnLayout L = attn_layout(dtype, B, C, D, Hq, Hkv, d, max_prefix, layer_type, window);
  if (!ws_ok(workspace, ws_bytes, L.total))
    return fail(CANVAS_ERR_WORKSPACE, "canvas_attention: workspace missing, small or misaligned (need %zu)", L.total);

  Carver cv(workspace);
  float* proj_q = cv.take<float>(L.proj_q);
  float* proj_k = cv.take<float>(L.proj_k);
  float* proj_v = cv.take<float>(L.proj_v);
  void* gws = cv.take<char>(L.gemm);
  void* Qp = cv.take<char>(L.qp);
  void* Kx = cv.take<char>(L.kx);
  void* Vx = cv.take<char>(L.vx);
  float* vs_tail = cv.take<float>(L.vs_tail);
  void* Kt = cv.take<char>(L.kt);
  float* vs_pre = cv.take<float>(L.vs_pre);
  float* part_o = cv.take<float>(L.part_o);
  float* part_ml = cv.take<float>(L.part_ml);
  const int M = B * C;
  const int G = Hq / Hkv;

  mark_start(CANVAS_KERNEL_PREP, stream);
  // 3. prefix keys of global layers, the prefix rows of the tail, zero padding:
  // independent of the projections and of the canvas rows (it writes other
  // rows of the tail buffers), so a large one (global layers with long
  // prefixes: 78 -> 62 us of preparation at prefix 32768) runs on a side
  // stream beside steps 1-2; a small one stays on the call's stream and
  // spares the fork and join
  const bool big_prep = global && (long long)B * Hkv * max_prefix * d * 2 >= (32ll << 20);
  SideStream* side = big_prep ? side_stream() : nullptr;
  cudaStream_t kstream = stream;
  if (side) {
    CANVAS_CUDA(cudaEventRecord(side->fork, stream));
    CANVAS_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
    kstream = side->s;
  }
  KeyPrepArgs k;
  k.k_pool = kv->k_pool;
  k.v_pool = kv->v_pool;
  k.block_table = kv->block_table;
  k.max_pages = kv->max_pages_per_seq;
  k.page_tokens = max_prefix > 0 ? kv->page_tokens : 64;
  k.num_pages = kv->num_pages;
  k.gamma_k = gamma_k;
  k.freq = freq;
  k.prefix_len = prefix_len;
  k.B = B;
  k.C = C;
  k.Hkv = Hkv;
  k.d = d;
  k.max_prefix = max_prefix;
  k.Tpad = pl.Tpad;
  k.eps = eps;
  k.global = global ? 1 : 0;
  k.Kt = Kt;
  k.vs_pre = vs_pre;
  k.Kx = Kx;
  k.Vx = Vx;
  k.vs_tail = vs_tail;
  CANVAS_CUDA(launch_key_prep(k, bf16, kstream));
  if (side) CANVAS_CUDA(cudaEventRecord(side->join, kstream));
  // 1. projections q = x W_q^T, k = x W_k^T, v = x W_v^T (fp32 accumulate)
  int proj_splits = 1;
  if (bf16) {
    // one launch for the two or three products (they share x)
    const void* Ws[3] = {W_q, W_k, W_v};
    void* outs[3] = {proj_q, proj_k, proj_v};
    const int Ns[3] = {Hq * d, Hkv * d, Hkv * d};
    // a split product stays in its partials: the prologue sums them
    float* parts[3] = {nullptr, nullptr, nullptr};
    const canvas_status st =
        run_gemm_group(x, Ws, outs, Ns, global ? 2 : 3, 0, M, D, 0, 0, gws, stream, parts, &proj_splits);
    if (st != CANVAS_OK) return st;
    proj_q = parts[0];
    proj_k = parts[1];
    if (!global) proj_v = parts[2];
  } else {
    CANVAS_CUDA(launch_gemm_simt(x, W_q, 0, false, proj_q, M, Hq * d, D, 0, stream));
    CANVAS_CUDA(launch_gemm_simt(x, W_k, 0, false, proj_k, M, Hkv * d, D, 0, stream));
    if (!global) CANVAS_CUDA(launch_gemm_simt(x, W_v, 0, false, proj_v, M, Hkv * d, D, 0, stream));
  }
  // 2. rms + rotate of the canvas rows (queries, canvas keys / values)
  PrologueArgs p;
  p.proj_q = proj_q;
  p.proj_k = proj_k;
  p.proj_v = global ? nullptr : proj_v;
  p.splits = proj_splits;
  p.gamma_q = gamma_q;
  p.gamma_k = gamma_k;
  p.freq = freq;
  p.prefix_len = prefix_len;
  p.B = B;
  p.C = C;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.d = d;
  p.Tpad = pl.Tpad;
  p.eps = eps;
  p.global = global ? 1 : 0;
  p.Qp = Qp;
  p.Kx = Kx;
  p.Vx = Vx;
  p.vs_tail = vs_tail;
  CANVAS_CUDA(launch_prologue(p, bf16, stream));
  // 3. (launched first, beside steps 1-2) the prefix keys
  if (side) CANVAS_CUDA(cudaStreamWaitEvent(stream, side->join, 0));
  mark_stop(CANVAS_KERNEL_PREP, stream);

  // 4. attention
  if (bf16) {
    const uint64_t BH = uint64_t(B) * Hkv;
    AttnTcMaps maps;
    canvas_status st = make_map_bf16(&maps.q, Qp, BH * G * C, d, kAttnBM, 64);
    if (st != CANVAS_OK) return st;
    st = make_map_bf16(&maps.kx, Kx, BH * pl.Tpad, d, 64, 64);
    if (st != CANVAS_OK) return st;
    st = make_map_bf16(&maps.vx, Vx, BH * pl.Tpad, d, 64, 64);
    if (st != CANVAS_OK) return st;
    if (max_prefix > 0) {
      const uint64_t pool_rows = uint64_t(kv->num_pages) * Hkv * kv->page_tokens;
      st = global ? make_map_bf16(&maps.kpre, Kt, BH * max_prefix, d, 64, 64)
                  : make_map_bf16(&maps.kpre, kv->k_pool, pool_rows, d, 64, 64);
      if (st != CANVAS_OK) return st;
      st = make_map_bf16(&maps.vpre, global ? kv->k_pool : kv->v_pool, pool_rows, d, 64, 64);
      if (st != CANVAS_OK) return st;
    } else {
      maps.kpre = maps.kx;  // never read: no prefix sub-blocks
      maps.vpre = maps.vx;
    }
    // the 4-SM kernel (head_dim 512) reads keys in boxes of 32 rows x all of
    // d and values in boxes of 64 rows x 128 columns, one copy each
    const bool quad = d == 512;
    if (quad) {
      st = make_map_bf16_chunked(&maps.kx_c, Kx, BH * pl.Tpad, d, 32, 8);
      if (st != CANVAS_OK) return st;
      st = make_map_bf16_chunked(&maps.vx_c, Vx, BH * pl.Tpad, d, 64, 2);
      if (st != CANVAS_OK) return st;
      if (max_prefix > 0) {
        const uint64_t pool_rows = uint64_t(kv->num_pages) * Hkv * kv->page_tokens;
        st = global ? make_map_bf16_chunked(&maps.kpre_c, Kt, BH * max_prefix, d, 32, 8)
                    : make_map_bf16_chunked(&maps.kpre_c, kv->k_pool, pool_rows, d, 32, 8);
        if (st != CANVAS_OK) return st;
        st = make_map_bf16_chunked(&maps.vpre_c, global ? kv->k_pool : kv->v_pool, pool_rows, d, 64, 2);
        if (st != CANVAS_OK) return st;
      } else {
        maps.kpre_c = maps.kx_c;  // never read: no prefix sub-blocks
        maps.vpre_c = maps.vx_c;
      }
    } else {
      // the one-SM kernel reads a value sub-block's d columns in one copy
      maps.kx_c = maps.kx;  // not read by the other kernels
      maps.kpre_c = maps.kpre;
      st = make_map_bf16_chunked(&maps.vx_c, Vx, BH * pl.Tpad, d, 64, uint32_t(d / 64));
      if (st != CANVAS_OK) return st;
      if (max_prefix > 0) {
        const uint64_t pool_rows = uint64_t(kv->num_pages) * Hkv * kv->page_tokens;
        st = make_map_bf16_chunked(&maps.vpre_c, global ? kv->k_pool : kv->v_pool, pool_rows, d, 64,
                                   uint32_t(d / 64));
        if (st != CANVAS_OK) return st;
      } else {
        maps.vpre_c = maps.vx_c;
      }
    }
    AttnTcArgs t;
    t.B = B;
    t.C = C;
    t.Hq = Hq;
    t.Hkv = Hkv;
    t.G = G;
    t.d = d;
    t.DV = d > 256 ? 256 : d;
    t.dv_parts = pl.dv_parts;
    t.q_tiles = pl.q_tiles;
    t.nsplit = pl.nsplit;
    t.max_prefix = max_prefix;
    t.window = global ? 0 : window;
    t.Tpad = pl.Tpad;
    t.kpre_paged = global ? 0 : 1;
    // head_dim 512: four SMs per 256 query rows (two 2-SM pairs split each
    // key block, so no S is formed twice); 2-SM MMAs do not pay at head_dim
    // 256 (166 -> 178 us), where one SM per tile stays
    t.pair = quad ? 2 : 0;
    t.causal = causal;
    t.Qp = static_cast<const __nv_bfloat16*>(Qp);
    t.block_table = kv->block_table;
    t.max_pages = kv->max_pages_per_seq;
    t.page_tokens = max_prefix > 0 ? kv->page_tokens : 64;
    t.num_pages = kv->num_pages;
    t.prefix_len = prefix_len;
    t.vs_pre = v_unit_rms ? vs_pre : nullptr;
    t.vs_tail = v_unit_rms ? vs_tail : nullptr;
    t.c_log2 = scale * 1.4426950408889634f;
    t.out = static_cast<__nv_bfloat16*>(out);
    t.lse = lse;
    t.part_o = part_o;
    t.part_ml = part_ml;
    mark_start(CANVAS_KERNEL_ATTENTION, stream);
    CANVAS_CUDA(launch_attention_tc(maps, t, stream));
    if (t.nsplit > 1) CANVAS_CUDA(launch_attention_combine(t, stream));
    mark_stop(CANVAS_KERNEL_ATTENTION, stream);
  } else {
    AttnArgs a;
    a.Qp = Qp;
    a.k_pre = global ? Kt : kv->k_pool;
    a.v_pre = global ? kv->k_pool : kv->v_pool;
    a.block_table = kv->block_table;
    a.max_pages = kv->max_pages_per_seq;
    a.page_tokens = max_prefix > 0 ? kv->page_tokens : 64;
    a.num_pages = kv->num_pages;
    a.Kx = Kx;
    a.Vx = Vx;
    a.vs_pre = vs_pre;
    a.vs_tail = vs_tail;
    a.prefix_len = prefix_len;
    a.B = B;
    a.C = C;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.max_prefix = max_prefix;
    a.window = window;
    a.Tpad = pl.Tpad;
    a.global = global ? 1 : 0;
    a.v_unit_rms = v_unit_rms ? 1 : 0;
    a.causal = causal;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    mark_start(CANVAS_KERNEL_ATTENTION, stream);
    CANVAS_CUDA(launch_attention_simt(a, bf16, stream));
    mark_stop(CANVAS_KERNEL_ATTENTION, stream);
  }
  return CANVAS_OK;
}

canvas_status canvas_attention(const void* x, int dtype, int B, int C, int D, const void* W_q, const void* W_k,
                               const void* W_v, int Hq, int Hkv, int d, const float* gamma_q, const float* gamma_k,
                               float eps, const float* freq, int layer_type, const canvas_kv_cache* kv,
                               const int32_t* prefix_len, int max_prefix, int window, float scale, int v_unit_rms,
                               void* out, float* lse, void* workspace, size_t ws_bytes, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_attention");
  return attention_impl(x, dtype, B, C, D, W_q, W_k, W_v, Hq, Hkv, d, gamma_q, gamma_k, eps, freq, layer_type, kv,
                        prefix_len, max_prefix, window, scale, v_unit_rms, out, lse, workspace, ws_bytes, stream, 0);
}

canvas_status canvas_attention_encode(const void* x, int dtype, int B, int C, int D, const void* W_q,
                                      const void* W_k, const void* W_v, int Hq, int Hkv, int d,
                                      const float* gamma_q, const float* gamma_k, float eps, const float* freq,
                                      int layer_type, const canvas_kv_cache* kv, const int32_t* prefix_len,
                                      int max_prefix, int window, float scale, int v_unit_rms, void* out, float* lse,
                                      void* workspace, size_t ws_bytes, canvas_stream_t stream) {
  NvtxRange nvtx_range("canvas_attention_encode");
  return attention_impl(x, dtype, B, C, D, W_q, W_k, W_v, Hq, Hkv, d, gamma_q, gamma_k, eps, freq, layer_type, kv,
                        prefix_len, max_prefix, window, scale, v_unit_rms, out, lse, workspace, ws_bytes, stream, 1);
}

// ------------------------------------------------------------------ block commit
static size_t kv_append_ws(int dtype, int B, int C, int D, int Hkv, int d, int layer_type, size_t* gemm_ws) {
  const size_t M = size_t(B) * C;
  const bool global = layer_type == CANVAS_LAYER_GLOBAL;
  const size_t proj = M * Hkv * d * 4;
  size_t g = 0;
  if (dtype == CANVAS_BF16) {
    const int Ns[2] = {Hkv * d, Hkv * d};
    g = gemm_ws_bytes(plan_gemm_group(int(M), Ns, global ? 1 : 2, D));
  }
  if (gemm_ws) *gemm_ws = g;
  return align_up(proj) + (global ? 0 : align_up(proj)) + align_up(g) + kAlign;
}

size_t canvas_kv_append_workspace_size(int dtype, int B, int C, int D, int Hkv, int d, int layer_type) {
  if ((dtype != CANVAS_BF16 && dtype != CANVAS_FP32) || B < 1 || C < 1 || D < 1 || Hkv < 1 || d < 2) return 0;
  if (layer_type != CANVAS_LAYER_SLIDING && layer_type != CANVAS_LAYER_GLOBAL) return 0;
  return kv_append_ws(dtype, B, C, D, Hkv, d, layer_type, nullptr);
}

canvas_status canvas_kv_append(const void* x, int dtype, int B, int C, int D, const void* W_k, const void* W_v,
                               int Hkv, int d, const float* gamma_k, float eps, const float* freq, int layer_type,
                               const canvas_kv_cache* kv, int32_t* prefix_len, int max_prefix, void* workspace,
                               size_t ws_bytes, canvas_stream_t stream_) {
  NvtxRange nvtx_range("canvas_kv_append");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t need = canvas_kv_append_workspace_size(dtype, B, C, D, Hkv, d, layer_type);
  if (need == 0) return fail(CANVAS_ERR_ARG, "canvas_kv_append: invalid shape, dtype or layer type");
  const bool global = layer_type == CANVAS_LAYER_GLOBAL;
  const bool bf16 = dtype == CANVAS_BF16;
  if (!x || !W_k || !gamma_k || !freq || !kv || !prefix_len || !kv->k_pool || !kv->block_table)
    return fail(CANVAS_ERR_ARG, "canvas_kv_append: null pointer");
  if (global && (W_v != nullptr || kv->v_pool != nullptr))
    return fail(CANVAS_ERR_ARG, "canvas_kv_append: global layers keep one raw shared pool (W_v and v_pool NULL)");
  if (!global && (W_v == nullptr || kv->v_pool == nullptr))
    return fail(CANVAS_ERR_ARG, "canvas_kv_append: sliding layers need W_v and v_pool");
  if ((reinterpret_cast<uintptr_t>(x) & 15) != 0) return fail(CANVAS_ERR_ARG, "canvas_kv_append: x must be 16-byte aligned");
  if (kv->page_tokens < 1 || kv->num_pages < 1 || kv->max_pages_per_seq < 1 || max_prefix < C ||
      (long long)kv->max_pages_per_seq * kv->page_tokens < max_prefix)
    return fail(CANVAS_ERR_ARG, "canvas_kv_append: cache geometry cannot hold max_prefix tokens");
  if (d % 64 != 0 || d > 512) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_kv_append: head_dim must be 64, 128, ..., 512");
  if (bf16 && ((d & (d - 1)) != 0 || D % 8 != 0))
    return fail(CANVAS_ERR_UNSUPPORTED, "canvas_kv_append: bf16 needs head_dim 64, 128, 256 or 512 and D a multiple of 8");
  if (!ws_ok(workspace, ws_bytes, need))
    return fail(CANVAS_ERR_WORKSPACE, "canvas_kv_append: workspace missing, small or misaligned (need %zu)", need);
  size_t gws_bytes = 0;
  kv_append_ws(dtype, B, C, D, Hkv, d, layer_type, &gws_bytes);
  const size_t M = size_t(B) * C;
  Carver cv(workspace);
  float* proj_k = cv.take<float>(M * Hkv * d * 4);
  float* proj_v = global ? nullptr : cv.take<float>(M * Hkv * d * 4);
  void* gws = cv.take<char>(gws_bytes);
  if (bf16) {
    const void* Ws[2] = {W_k, W_v};
    void* outs[2] = {proj_k, proj_v};
    const int Ns[2] = {Hkv * d, Hkv * d};
    const canvas_status st = run_gemm_group(x, Ws, outs, Ns, global ? 1 : 2, 0, int(M), D, 0, 0, gws, stream);
    if (st != CANVAS_OK) return st;
  } else {
    CANVAS_CUDA(launch_gemm_simt(x, W_k, 0, false, proj_k, int(M), Hkv * d, D, 0, stream));
    if (!global) CANVAS_CUDA(launch_gemm_simt(x, W_v, 0, false, proj_v, int(M), Hkv * d, D, 0, stream));
  }
  KvAppendArgs p;
  p.proj_k = proj_k;
  p.proj_v = proj_v;
  p.gamma_k = gamma_k;
  p.freq = freq;
  p.prefix_len = prefix_len;
  p.k_pool = const_cast<void*>(kv->k_pool);
  p.v_pool = const_cast<void*>(kv->v_pool);
  p.block_table = kv->block_table;
  p.max_pages = kv->max_pages_per_seq;
  p.page_tokens = kv->page_tokens;
  p.num_pages = kv->num_pages;
  p.B = B;
  p.C = C;
  p.Hkv = Hkv;
  p.d = d;
  p.max_prefix = max_prefix;
  p.eps = eps;
  p.global = global ? 1 : 0;
  CANVAS_CUDA(launch_kv_append(p, bf16, stream));
  return CANVAS_OK;
}

// ------------------------------------------------------------------ mixture of experts
struct MoeLayout {
  size_t scores, topk_idx, topk_w, counts, offsets, cursor, tiles, slot, xg, hg, hu, ag, yg, hs_g, hs_u, as, ys,
      gemm, total;
  int max_tiles;
};

static MoeLayout moe_layout(int R, int D, int E, int F, int k, int Fs) {
  MoeLayout L;
  // every expert's rows padded to whole 128-row tiles: at most R k + E 127 rows
  L.max_tiles = int((size_t(R) * k + size_t(E) * 127 + 127) / 128);
  const size_t Mpad = size_t(L.max_tiles) * 128;
  L.scores = size_t(R) * E * 4;
  L.topk_idx = size_t(R) * k * 4;
  L.topk_w = size_t(R) * k * 4;
  L.counts = size_t(E) * 4;
  L.offsets = size_t(E + 1) * 4;
  L.cursor = size_t(E) * 4;
  L.tiles = size_t(L.max_tiles) * 4;
  L.slot = size_t(R) * k * 4;
  L.xg = Mpad * D * 2;
  L.hg = Mpad * F * 4;
  L.hu = L.hg;
  L.ag = Mpad * F * 2;
  L.yg = Mpad * D * 4;
  L.hs_g = Fs > 0 ? size_t(R) * Fs * 4 : 0;
  L.hs_u = L.hs_g;
  L.as = Fs > 0 ? size_t(R) * Fs * 2 : 0;
  L.ys = Fs > 0 ? size_t(R) * D * 4 : 0;
  size_t g = gemm_ws_bytes(plan_gemm(R, E, D));
  if (Fs > 0) {
    const int Ns[2] = {Fs, Fs};
    g = std::max(g, gemm_ws_bytes(plan_gemm_group(R, Ns, 2, D)));
    g = std::max(g, gemm_ws_bytes(plan_gemm(R, D, Fs)));
  }
  L.gemm = g;
  L.total = align_up(L.scores) + align_up(L.topk_idx) + align_up(L.topk_w) + align_up(L.counts) +
            align_up(L.offsets) + align_up(L.cursor) + align_up(L.tiles) + align_up(L.slot) + align_up(L.xg) +
            align_up(L.hg) + align_up(L.hu) + align_up(L.ag) + align_up(L.yg) + align_up(L.hs_g) +
            align_up(L.hs_u) + align_up(L.as) + align_up(L.ys) + align_up(L.gemm) + kAlign;
  return L;
}

static bool moe_shape_ok(int R, int D, int E, int F, int k, int Fs) {
  return R >= 1 && D >= 8 && D % 8 == 0 && E >= 1 && E <= 256 && F >= 8 && F % 8 == 0 && k >= 1 && k <= 16 &&
         k <= E && Fs >= 0 && Fs % 8 == 0 && E % 8 == 0;
}

size_t canvas_moe_workspace_size(int R, int D, int E, int F, int k, int Fs) {
  if (!moe_shape_ok(R, D, E, F, k, Fs)) return 0;
  return moe_layout(R, D, E, F, k, Fs).total;
}

canvas_status canvas_moe(const void* x, int R, int D, const void* router, int E, int k, const float* expert_scale,
                         const void* W_gate, const void* W_up, const void* W_down, int F, const void* Ws_gate,
                         const void* Ws_up, const void* Ws_down, int Fs, float* out, int32_t* topk_idx,
                         float* topk_w, void* workspace, size_t ws_bytes, canvas_stream_t stream_) {
  NvtxRange nvtx_range("canvas_moe");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!moe_shape_ok(R, D, E, F, k, Fs))
    return fail(CANVAS_ERR_ARG, "canvas_moe: shape (D, F, Fs multiples of 8; E a multiple of 8 up to 256; 1 <= k <= 16, k <= E)");
  if (!x || !router || !W_gate || !W_up || !W_down || !out) return fail(CANVAS_ERR_ARG, "canvas_moe: null pointer");
  if (Fs > 0 && (!Ws_gate || !Ws_up || !Ws_down)) return fail(CANVAS_ERR_ARG, "canvas_moe: shared expert weights");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_moe: x and out must be 16-byte aligned");
  const MoeLayout L = moe_layout(R, D, E, F, k, Fs);
  if (!ws_ok(workspace, ws_bytes, L.total))
    return fail(CANVAS_ERR_WORKSPACE, "canvas_moe: workspace missing, small or misaligned (need %zu)", L.total);
  Carver cv(workspace);
  MoeArgs a;
  a.R = R;
  a.D = D;
  a.E = E;
  a.k = k;
  a.max_tiles = L.max_tiles;
  float* scores = cv.take<float>(L.scores);
  a.scores = scores;
  a.expert_scale = expert_scale;
  int32_t* idx_ws = cv.take<int32_t>(L.topk_idx);
  float* w_ws = cv.take<float>(L.topk_w);
  a.topk_idx = topk_idx ? topk_idx : idx_ws;
  a.topk_w = topk_w ? topk_w : w_ws;
  a.counts = cv.take<int32_t>(L.counts);
  a.offsets = cv.take<int32_t>(L.offsets);
  a.cursor = cv.take<int32_t>(L.cursor);
  a.group_of_mtile = cv.take<int32_t>(L.tiles);
  a.slot = cv.take<int32_t>(L.slot);
  a.x = x;
  a.xg = cv.take<char>(L.xg);
  float* hg = cv.take<float>(L.hg);
  float* hu = cv.take<float>(L.hu);
  void* ag = cv.take<char>(L.ag);
  float* yg = cv.take<float>(L.yg);
  float* hs_g = cv.take<float>(L.hs_g);
  float* hs_u = cv.take<float>(L.hs_u);
  void* as = cv.take<char>(L.as);
  float* ys = cv.take<float>(L.ys);
  void* gws = cv.take<char>(L.gemm);
  a.yg = yg;
  a.ys = Fs > 0 ? ys : nullptr;
  a.out = out;
  const int Mpad = L.max_tiles * 128;
  // 1. router scores, top-k, weights, grouped rows
  canvas_status st = run_gemm_tc(x, router, 0, scores, R, E, D, 0, gws, stream);
  if (st != CANVAS_OK) return st;
  CANVAS_CUDA(launch_moe_route(a, stream));
  // 2. the routed experts: gate and up in one grouped launch, the gated
  //    activation, down
  {
    const void* Bs[2] = {W_gate, W_up};
    void* Cs[2] = {hg, hu};
    const int Ns[2] = {F, F};
    st = run_gemm_grouped(a.xg, Bs, Cs, Ns, 2, E, a.group_of_mtile, Mpad, D, 0, stream);
    if (st != CANVAS_OK) return st;
    CANVAS_CUDA(launch_moe_act(hg, hu, ag, (long long)Mpad * F, stream));
    const void* Bd[1] = {W_down};
    void* Cd[1] = {yg};
    const int Nd[1] = {D};
    st = run_gemm_grouped(ag, Bd, Cd, Nd, 1, E, a.group_of_mtile, Mpad, F, 0, stream);
    if (st != CANVAS_OK) return st;
  }
  // 3. the shared expert on every token
  if (Fs > 0) {
    const void* Bs[2] = {Ws_gate, Ws_up};
    void* Cs[2] = {hs_g, hs_u};
    const int Ns[2] = {Fs, Fs};
    st = run_gemm_group(x, Bs, Cs, Ns, 2, 0, R, D, 0, 0, gws, stream);
    if (st != CANVAS_OK) return st;
    CANVAS_CUDA(launch_moe_act(hs_g, hs_u, as, (long long)R * Fs, stream));
    st = run_gemm_tc(as, Ws_down, 0, ys, R, D, Fs, 0, gws, stream);
    if (st != CANVAS_OK) return st;
  }
  // 4. out = sum of weighted expert outputs + shared
  CANVAS_CUDA(launch_moe_combine(a, stream));
  return CANVAS_OK;
}

size_t canvas_sample_workspace_size(int dtype, int rows, int V, int D) {
  if ((dtype != CANVAS_BF16 && dtype != CANVAS_FP32) || rows < 1 || V < 1 || D < 1) return 0;
  return sample_layout(dtype, rows, V, D).total;
}

canvas_status canvas_sample(const void* logits, int dtype, int rows, int V, const void* E, int D,
                            float entropy_bound, uint64_t seed, uint32_t step, float temperature, int commit_mode,
                            int canvas_len, const uint8_t* frozen, const int32_t* frozen_tokens, int32_t* tokens,
                            uint8_t* commit_mask, float* entropy, float* confidence, int32_t* argmax,
                            void* probs_out, int probs_dtype, float* soft_emb, void* workspace, size_t ws_bytes,
                            canvas_stream_t stream_) {
  NvtxRange nvtx_range("canvas_sample");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dtype != CANVAS_BF16 && dtype != CANVAS_FP32) return fail(CANVAS_ERR_ARG, "canvas_sample: dtype");
  if (rows < 1 || V < 1 || D < 1) return fail(CANVAS_ERR_ARG, "canvas_sample: bad shape");
  if (!logits || !E || !tokens || !commit_mask || !entropy || !confidence || !soft_emb)
    return fail(CANVAS_ERR_ARG, "canvas_sample: null pointer");
  if ((frozen == nullptr) != (frozen_tokens == nullptr))
    return fail(CANVAS_ERR_ARG, "canvas_sample: frozen and frozen_tokens go together");
  if (!(temperature > 0.f)) return fail(CANVAS_ERR_ARG, "canvas_sample: temperature must be > 0");
  if (commit_mode < 0 || commit_mode > 3) return fail(CANVAS_ERR_ARG, "canvas_sample: commit_mode");
  if (canvas_len < 1 || ((commit_mode & 1) && rows % canvas_len != 0))
    return fail(CANVAS_ERR_ARG, "canvas_sample: canvas_len");
  if (probs_out && probs_dtype != CANVAS_BF16 && probs_dtype != CANVAS_FP32)
    return fail(CANVAS_ERR_ARG, "canvas_sample: probs_dtype");
  if (V % 8 != 0 || D % 8 != 0) return fail(CANVAS_ERR_UNSUPPORTED, "canvas_sample: V and D must be multiples of 8");
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(probs_out) | reinterpret_cast<uintptr_t>(E) |
       reinterpret_cast<uintptr_t>(soft_emb)) % 16 != 0)
    return fail(CANVAS_ERR_ARG, "canvas_sample: logits, probs_out, E and soft_emb must be 16-byte aligned");
  const SampleLayout L = sample_layout(dtype, rows, V, D);
  if (!ws_ok(workspace, ws_bytes, L.total))
    return fail(CANVAS_ERR_WORKSPACE, "canvas_sample: workspace missing, small or misaligned (need %zu)", L.total);
  Carver cv(workspace);
  char* probs_ws = cv.take<char>(L.probs);
  int32_t* argmax_ws = cv.take<int32_t>(L.argmax);
  void* gws = cv.take<char>(L.gemm);
  float* states_ws = cv.take<float>(L.states);
  const bool bf16 = dtype == CANVAS_BF16;
  const GemmPlan gp = plan_gemm(rows, D, V);

  SampleArgs a;
  a.rows = rows;
  a.V = V;
  // cluster of up to 8 CTAs per row; each CTA owns a multiple of 8 columns
  int cl = 1;
  while (cl < kMaxSampleCluster && (long long)V / (cl * 2) >= 4096) cl *= 2;
  a.cluster = cl;
  a.chunk = ((V + cl - 1) / cl + 7) / 8 * 8;
  a.inv_temp = 1.0f / temperature;
  a.bound = entropy_bound;
  a.seed = seed;
  a.step = step;
  a.commit_mode = commit_mode;
  a.canvas_len = canvas_len;
  a.frozen = frozen;
  a.frozen_tokens = frozen_tokens;
  a.tokens = tokens;
  a.commit_mask = commit_mask;
  a.entropy = entropy;
  a.confidence = confidence;
  a.argmax = argmax ? argmax : argmax_ws;
  // the probabilities the soft embedding multiplies: bf16 for bf16 calls,
  // fp32 for fp32 calls; written to probs_out when its dtype matches
  a.probs_bf16 = nullptr;
  a.probs_f32 = nullptr;
  if (bf16) {
    a.probs_bf16 = (probs_out && probs_dtype == CANVAS_BF16) ? static_cast<__nv_bfloat16*>(probs_out)
                                                              : reinterpret_cast<__nv_bfloat16*>(probs_ws);
    if (probs_out && probs_dtype == CANVAS_FP32) a.probs_f32 = static_cast<float*>(probs_out);
  } else {
    a.probs_f32 = (probs_out && probs_dtype == CANVAS_FP32) ? static_cast<float*>(probs_out)
                                                             : reinterpret_cast<float*>(probs_ws);
    if (probs_out && probs_dtype == CANVAS_BF16) a.probs_bf16 = static_cast<__nv_bfloat16*>(probs_out);
  }
  a.slices = 0;
  a.kb_per = a.kb_rem = 0;
  a.slice_state = nullptr;
  if (sample_deferred(dtype, probs_out, commit_mode, gp)) {
    // per-range p~ and states; the GEMM of p~ and E leaves its split
    // partials; one pass merges the states, decides, and sums the partials
    // scaled to probabilities
    a.slices = gp.splits;
    a.kb_per = gp.kblocks / gp.splits;
    a.kb_rem = gp.kblocks % gp.splits;
    a.slice_state = states_ws;
    mark_start(CANVAS_KERNEL_SAMPLER, stream);
    CANVAS_CUDA(launch_sampler_slices(a, logits, stream));
    mark_stop(CANVAS_KERNEL_SAMPLER, stream);
    mark_start(CANVAS_KERNEL_SOFT_EMB, stream);
    float* partials = nullptr;
    int splits = 0;
    const void* Bs[1] = {E};
    void* Cs[1] = {soft_emb};
    const int Ns[1] = {D};
    const canvas_status st =
        run_gemm_group(a.probs_bf16, Bs, Cs, Ns, 1, 1, rows, V, 0, 0, gws, stream, &partials, &splits);
    if (st != CANVAS_OK) return st;
    if (splits != a.slices) return fail(CANVAS_ERR_CUDA, "canvas_sample: GEMM split plan changed");
    CANVAS_CUDA(launch_soft_reduce(a, partials, soft_emb, D, stream));
    mark_stop(CANVAS_KERNEL_SOFT_EMB, stream);
    return CANVAS_OK;
  }
  mark_start(CANVAS_KERNEL_SAMPLER, stream);
  CANVAS_CUDA(launch_sampler(a, logits, bf16, stream));
  mark_stop(CANVAS_KERNEL_SAMPLER, stream);
  // soft embedding P . E
  mark_start(CANVAS_KERNEL_SOFT_EMB, stream);
  if (bf16) {
    const canvas_status st = run_gemm_tc(a.probs_bf16, E, 1, soft_emb, rows, D, V, 0, gws, stream);
    if (st != CANVAS_OK) return st;
  } else {
    CANVAS_CUDA(launch_gemm_simt(a.probs_f32, E, 1, false, soft_emb, rows, D, V, 0, stream));
  }
  mark_stop(CANVAS_KERNEL_SOFT_EMB, stream);
  return CANVAS_OK;
}

}  // extern "C"

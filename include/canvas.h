/*
 * canvas.h -- C ABI of libcanvas.so, one canvas refinement step of
 * DiffusionGemma-style block discrete diffusion on a B300 (sm_103a).
 *
 * Two calls make up the step:
 *   canvas_attention -- one fused attention layer in decode mode: QKV
 *                       projection, scalar QK RMSNorm, split-half / partial
 *                       RoPE, bidirectional attention of the canvas over the
 *                       committed (paged) KV prefix plus the canvas itself.
 *   canvas_sample    -- the per-position vocab sampler: softmax, entropy,
 *                       argmax, confidence, entropy-bound commit / uniform
 *                       renoise, and the self-conditioning soft embedding P.E.
 * plus the glue a caller needs to assemble whole denoising steps around them:
 * bf16 GEMMs (fp32 or bf16 output), the canvas input embedding and an
 * fp32 -> bf16 cast.
 *
 * Sources (the method is described on web pages, cited by title and section):
 *   [AIT] AI Trends summary of a DiffusionGemma 26B weights notebook
 *         (aitrends.kr/articles/94089), "섹션별 상세" (the rms(), rotate() and
 *         attention-block snippets; the sampling-loop paragraph) and the
 *         glossary "용어 해설".
 *   [TC]  ThakiCloud, "DiffusionGemma 26B-A4B", "아키텍처".
 *   [AB]  aibars news on DiffusionGemma, "블록 자동 회귀 노이즈 제거 및 자체 수정".
 *
 * Conventions shared by every call:
 *   - Every pointer argument is DEVICE memory unless its comment says "host".
 *     The caller owns all memory; no call allocates device memory.
 *   - Calls are asynchronous: they validate arguments on the host, enqueue
 *     kernels on `stream` and return.  They never synchronise.  Errors found
 *     on the device (a cache page index out of range, a bounded wait that ran
 *     out) are recorded in a per-device status word that
 *     canvas_device_status() reads.
 *   - A status other than CANVAS_OK leaves a message for
 *     canvas_last_error() (thread-local).  Shapes the kernels do not cover
 *     return CANVAS_ERR_UNSUPPORTED; there is no fallback path.
 *   - Calls on different streams may run concurrently if they use distinct
 *     workspaces.  Calls that share a workspace must be stream-ordered.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 */
#ifndef CANVAS_H_
#define CANVAS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* canvas_stream_t; /* same type as cudaStream_t */

typedef enum {
  CANVAS_OK = 0,
  CANVAS_ERR_ARG = -1,          /* bad pointer, size, or combination of flags */
  CANVAS_ERR_UNSUPPORTED = -2,  /* valid request outside what the kernels cover */
  CANVAS_ERR_CUDA = -3,         /* a CUDA runtime / driver call failed */
  CANVAS_ERR_TIMEOUT = -4,      /* a bounded device-side wait ran out */
  CANVAS_ERR_WORKSPACE = -5,    /* workspace NULL, too small or misaligned */
  CANVAS_ERR_BOUNDS = -6        /* device-side index check failed (e.g. a page id) */
} canvas_status;

typedef enum { CANVAS_BF16 = 0, CANVAS_FP32 = 1 } canvas_dtype;

typedef enum {
  /* local layer: the cache holds final keys (normed, rotated) and values;
     prefix tokens more than `window` positions back are not visible */
  CANVAS_LAYER_SLIDING = 0,
  /* global (full-attention) layer: W_v = W_k, the cache holds the raw shared
     projection r; key = rotate(rms(r)) at the key's position, value = r */
  CANVAS_LAYER_GLOBAL = 1
} canvas_layer_type;

/*
 * Paged KV cache of the committed prefix.  Caller-owned device memory.
 *
 * k_pool  [num_pages][Hkv][page_tokens][d], element type = the call's dtype.
 *         Sliding layers: final keys.  Global layers: raw shared rows r.
 * v_pool  same layout: values (sliding layers); must be NULL on global layers.
 * block_table [B][max_pages_per_seq] int32: physical page of logical page p
 *         of sequence b (tokens p*page_tokens ...).  Entries for pages that hold
 *         no visible token may be -1; entries that are read must lie in
 *         [0, num_pages), else the call records CANVAS_ERR_BOUNDS.
 * page_tokens must be a multiple of 64 for bf16 calls (any size for fp32 calls).
 */
typedef struct {
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  int32_t max_pages_per_seq;
  int32_t page_tokens;
  int32_t num_pages;
} canvas_kv_cache;

/*
 * Workspace (bytes) that canvas_attention needs for this shape.  The same
 * arguments must be passed to the call.  Returns 0 for an invalid shape.
 */
size_t canvas_attention_workspace_size(int dtype, int B, int C, int D, int Hq, int Hkv, int d,
                                       int max_prefix, int layer_type);

/*
 * canvas_attention -- one attention layer of a canvas refinement step.
 *
 * Defined by [AIT] "섹션별 상세": the attention-block snippet (projection,
 * 'l (n h) -> n l h', rms() on q and k, rotate() on q and k, then cache
 * concatenation and attention), the rms() snippet (w * x * sqrt(d) /
 * (||x||_2 + eps), norm in fp32), the rotate() snippet (split-half pairs
 * t, t+d/2; angle (l + start) * freq[t mod d/2]) and the decode-mode paragraph
 * (the canvas attends bidirectionally to committed past | current canvas;
 * W_v = W_k on full-attention layers, where only K is normed and rotated);
 * the glossary entries on partial RoPE and sliding-window attention; window
 * 1,024 per [TC] "아키텍처".
 *
 *   x        [B, C, D]            canvas input, dtype (row-major), 16-byte aligned
 *   W_q      [Hq*d, D]            dtype;  q = x W_q^T
 *   W_k      [Hkv*d, D]           dtype;  k = x W_k^T
 *   W_v      [Hkv*d, D] or NULL   dtype;  NULL only on global layers (W_v = W_k)
 *   gamma_q, gamma_k [d] fp32     QK-norm weights
 *   eps                           rms epsilon, added to ||x||_2
 *   freq     [d/2] fp32           RoPE spectrum; zero entries are not rotated
 *   layer_type                    canvas_layer_type
 *   kv       host pointer to the cache descriptor (device pointers inside)
 *   prefix_len [B] int32          committed prefix length of each sequence;
 *                                 canvas position i sits at prefix_len[b] + i
 *   max_prefix                    host: upper bound of prefix_len[] (sizes grids
 *                                 and the workspace); a larger prefix_len[b]
 *                                 records CANVAS_ERR_BOUNDS
 *   window                        sliding layers: a canvas row at position p
 *                                 sees prefix keys j >= p - window; <= 0 means
 *                                 the whole prefix.  Ignored on global layers.
 *   scale                         multiplies q.k, > 0 (1.0: the QK norm already
 *                                 fixes the temperature)
 *   v_unit_rms                    0 (default).  1 on a global layer: value =
 *                                 sqrt(d) * r / (||r|| + eps) (the scalar is
 *                                 applied in fp32 to each key's softmax weight)
 *   out      [B, C, Hq*d] dtype   heads concatenated, 'n l h -> l (n h)', 16-byte aligned
 *   lse      [B, C, Hq] fp32 or NULL   natural-log softmax normaliser
 *   workspace, ws_bytes           >= canvas_attention_workspace_size(...),
 *                                 256-byte aligned; contents are scratch
 *
 * Supported: dtype BF16 with d in {64, 128, 256, 512}, D % 8 == 0; dtype FP32
 * with d <= 512.  Hq % Hkv == 0, d even, C >= 1.
 */
canvas_status canvas_attention(const void* x, int dtype, int B, int C, int D,
                               const void* W_q, const void* W_k, const void* W_v,
                               int Hq, int Hkv, int d,
                               const float* gamma_q, const float* gamma_k, float eps,
                               const float* freq, int layer_type,
                               const canvas_kv_cache* kv,
                               const int32_t* prefix_len, int max_prefix, int window,
                               float scale, int v_unit_rms,
                               void* out, float* lse,
                               void* workspace, size_t ws_bytes, canvas_stream_t stream);

/*
 * canvas_attention_encode -- the same layer in encode mode.
 *
 * Defined by [AIT] "섹션별 상세", the decode / encode paragraph: committed
 * tokens are encoded causally, like a prefill.  Every argument, layout, error
 * and the workspace are those of canvas_attention; the one difference is the
 * mask inside the block: row i attends to the visible committed prefix (as in
 * decode mode) and to block rows 0 .. i only.  A caller that commits a
 * finished canvas runs its layers in this mode and appends each layer's rows
 * to the cache with canvas_kv_append.
 */
canvas_status canvas_attention_encode(const void* x, int dtype, int B, int C, int D,
                                      const void* W_q, const void* W_k, const void* W_v,
                                      int Hq, int Hkv, int d,
                                      const float* gamma_q, const float* gamma_k, float eps,
                                      const float* freq, int layer_type,
                                      const canvas_kv_cache* kv,
                                      const int32_t* prefix_len, int max_prefix, int window,
                                      float scale, int v_unit_rms,
                                      void* out, float* lse,
                                      void* workspace, size_t ws_bytes, canvas_stream_t stream);

/* Workspace (bytes) that canvas_kv_append needs; 0 for an invalid shape. */
size_t canvas_kv_append_workspace_size(int dtype, int B, int C, int D, int Hkv, int d, int layer_type);

/*
 * canvas_kv_append -- block commit: write a committed block's cache rows.
 *
 * Defined by [AB] "블록 자동 회귀 노이즈 제거 및 자체 수정" (a denoised block is
 * committed to the KV cache) and [AIT] "섹션별 상세" (the attention-block
 * snippet: keys are normed and rotated, values are not; on full-attention
 * layers W_v = W_k and only K is normed and rotated).  Block row i of
 * sequence b is written at position p = prefix_len[b] + i:
 *   sliding layers  k_pool <- rotate(rms(x W_k^T, gamma_k)) at position p,
 *                   v_pool <- x W_v^T   (the final keys and values)
 *   global layers   k_pool <- r = x W_k^T (the raw shared row; its key is
 *                   formed from it at attention time)
 * each computed in fp32 and stored once in the call's dtype, exactly as
 * canvas_attention stores the same rows of a canvas; then prefix_len[b] += C
 * (on the device, after every row is written).
 *
 *   x        [B, C, D] dtype      the block's layer input, 16-byte aligned
 *   W_k, W_v [Hkv*d, D] dtype     W_v NULL on global layers
 *   gamma_k [d], freq [d/2] fp32, eps, layer_type: as for canvas_attention
 *   kv       host pointer to the cache descriptor; its pools are WRITTEN.
 *            The block table must map every page the new positions fall in.
 *   prefix_len [B] int32 device   read, then advanced by C
 *   max_prefix                    host: every new position must be below it
 *                                 and kv must be able to hold it; a row past
 *                                 it, or on an unmapped page, is skipped and
 *                                 records CANVAS_ERR_BOUNDS
 *   workspace, ws_bytes           >= canvas_kv_append_workspace_size(...)
 * Asynchronous on `stream`.
 */
canvas_status canvas_kv_append(const void* x, int dtype, int B, int C, int D,
                               const void* W_k, const void* W_v, int Hkv, int d,
                               const float* gamma_k, float eps, const float* freq, int layer_type,
                               const canvas_kv_cache* kv, int32_t* prefix_len, int max_prefix,
                               void* workspace, size_t ws_bytes, canvas_stream_t stream);

/* Workspace (bytes) that canvas_sample needs; 0 for an invalid shape. */
size_t canvas_sample_workspace_size(int dtype, int rows, int V, int D);

/*
 * canvas_sample -- the sampler of one denoising step, per canvas position.
 *
 * Defined by [AIT] "섹션별 상세", the sampling-loop paragraph (per-position
 * entropy; positions within the entropy bound are fixed, the rest renoised to
 * uniformly random tokens), [AB] "블록 자동 회귀 노이즈 제거 및 자체 수정"
 * (low-confidence tokens swapped for random tokens), and the self-conditioning
 * glossary entry of [AIT] (expected embedding P.E of the softmax).
 *
 *   logits   [rows, V] dtype      rows = B*C positions; 16-byte aligned
 *   E        [V, D] dtype         embedding table (row-major), 16-byte aligned
 *   entropy_bound                 commit iff entropy < bound (nats, strict)
 *   seed, step                    renoise key = m(m(m(seed) ^ step) ^ row),
 *                                 m = one SplitMix64 output; token = key mod V
 *   temperature                   logits are divided by it (> 0)
 *   commit_mode                   bit 0 -- 0: commit per position; 1: the
 *                                 longest run of qualifying positions from
 *                                 the left of each canvas of canvas_len rows.
 *                                 bit 1 -- 0: a committed (not frozen)
 *                                 position takes its argmax; 1: it takes a
 *                                 categorical draw from its stored
 *                                 probabilities p~ (the tempered softmax in
 *                                 the probability dtype below): the smallest k
 *                                 with sum_{j<=k} p~_j > u * sum_j p~_j, sums in
 *                                 fp64, u = (key >> 40) / 2^24 with key the
 *                                 row's renoise key (one key per row: a
 *                                 position either commits or renoises)
 *   canvas_len                    C (rows % C == 0 in mode 1)
 *   frozen   [rows] uint8 or NULL       1: position already committed; it keeps
 *   frozen_tokens [rows] int32 or NULL  its token and counts as committed
 *   tokens   [rows] int32         out: frozen token / argmax / renoise token
 *   commit_mask [rows] uint8      out: 1 = committed
 *   entropy, confidence [rows] fp32  out: -sum p ln p, max p
 *   argmax   [rows] int32 or NULL out: lowest index of the largest logit
 *   probs_out [rows, V] or NULL   out: softmax, in probs_dtype; 16-byte aligned
 *   probs_dtype                   CANVAS_BF16 or CANVAS_FP32
 *   soft_emb [rows, D] fp32       out: P.E, 16-byte aligned.  bf16 calls
 *                                 multiply bf16 probabilities; fp32 calls the
 *                                 fp32 ones.  A bf16 call with probs_out NULL
 *                                 and commit_mode bit 1 clear defers the
 *                                 normalisation: each vocabulary range of the
 *                                 product's K split stores bf16 2^(y - m_s)
 *                                 against its own maximum m_s, and the split
 *                                 sums are scaled by 2^(m_s - m) / Z (the same
 *                                 product; the bf16 roundings fall on the
 *                                 unnormalised values).
 *   workspace, ws_bytes           >= canvas_sample_workspace_size(...)
 *
 * Supported: V % 8 == 0, D % 8 == 0, rows >= 1.
 */
canvas_status canvas_sample(const void* logits, int dtype, int rows, int V,
                            const void* E, int D, float entropy_bound,
                            uint64_t seed, uint32_t step, float temperature,
                            int commit_mode, int canvas_len,
                            const uint8_t* frozen, const int32_t* frozen_tokens,
                            int32_t* tokens, uint8_t* commit_mask, float* entropy,
                            float* confidence, int32_t* argmax,
                            void* probs_out, int probs_dtype, float* soft_emb,
                            void* workspace, size_t ws_bytes, canvas_stream_t stream);

/* Workspace (bytes) that canvas_gemm_bf16 needs for this shape. */
size_t canvas_gemm_workspace_size(int M, int N, int K);

/*
 * canvas_gemm_bf16 -- C[M,N] (fp32) = A[M,K] . op(B)  (+ C if accumulate).
 *
 * Glue for callers that build whole layers (output projection, tied LM head)
 * and the soft-embedding product; the pages write these as plain matrix
 * products ([AIT] "섹션별 상세": x @ W.T).
 *   A  [M, K] bf16 row-major (K contiguous)
 *   B  b_layout 0: [N, K] row-major ("weights", C = A B^T)
 *      b_layout 1: [K, N] row-major (C = A B)
 *   C  [M, N] fp32 row-major, leading dimension N
 * Requires K % 8 == 0 and N % 8 == 0 (16-byte aligned rows) and A, B, C
 * 16-byte aligned (CANVAS_ERR_ARG otherwise).
 */
canvas_status canvas_gemm_bf16(const void* A, const void* B, int b_layout, float* C,
                               int M, int N, int K, int accumulate,
                               void* workspace, size_t ws_bytes, canvas_stream_t stream);

/*
 * canvas_gemm_bf16_to_bf16 -- C[M,N] (bf16) = bf16(A[M,K] . op(B)).
 *
 * The same product as canvas_gemm_bf16, accumulated in fp32 and rounded once
 * to bf16 (nearest even) where it is stored: the tied LM head of a denoising
 * step writes its logits this way, the form canvas_sample reads ([AIT]
 * "섹션별 상세", sampling-loop paragraph), without an fp32 copy of them.
 *   A, B, b_layout, M, N, K, workspace  as for canvas_gemm_bf16 (same
 *                                       workspace size)
 *   C  [M, N] bf16 row-major, leading dimension N, 16-byte aligned
 * Errors as for canvas_gemm_bf16.  Asynchronous on `stream`.
 */
canvas_status canvas_gemm_bf16_to_bf16(const void* A, const void* B, int b_layout, void* C,
                                       int M, int N, int K,
                                       void* workspace, size_t ws_bytes, canvas_stream_t stream);

/*
 * canvas_embed_input -- the canvas input of a denoising step:
 *   v[r, :] = E[tokens[r], :] + soft_emb[r, :]   (fp32)
 *   x = bf16(v), x32 = v
 * the embedding of the current tokens plus the self-conditioning soft
 * embedding P.E of the previous step ([AIT] glossary, self-conditioning; the
 * small MLP the page applies to P.E needs trained weights and is left to the
 * caller).  Glue for callers that chain steps into a loop.
 *   tokens   [rows] int32, each in [0, V) (else CANVAS_ERR_BOUNDS is recorded
 *            and the row is zero)
 *   E        [V, D] bf16, 16-byte aligned rows (D % 8 == 0)
 *   soft_emb [rows, D] fp32 or NULL (step 0: no previous step)
 *   x        [rows, D] bf16 out
 *   x32      [rows, D] fp32 out or NULL (a residual stream kept in fp32)
 */
canvas_status canvas_embed_input(const int32_t* tokens, const void* E, const float* soft_emb, int rows, int D,
                                 int V, void* x, float* x32, canvas_stream_t stream);

/*
 * canvas_cast_bf16 -- out[i] = bf16(in[i]) (round to nearest even), n % 8 == 0,
 * both 16-byte aligned.  Glue: an fp32 residual stream or fp32 logits become
 * the bf16 operands of the next call.
 */
canvas_status canvas_cast_bf16(const float* in, void* out, size_t n, canvas_stream_t stream);

/*
 * canvas_gelu_bf16 -- out[i] = bf16(gelu(in[i])), GELU in its tanh form
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), evaluated in fp32 as
 * x / (1 + exp(-2 sqrt(2/pi) (x + 0.044715 x^3))) (the same function, with
 * no cancellation for negative x) and rounded once (nearest even);
 * n % 8 == 0, both 16-byte aligned.  Glue: the
 * activation of the self-conditioning MLP ([AIT] glossary, self-conditioning:
 * the expected embedding P.E passes through a small MLP that maps zero to
 * zero before it is added to the canvas input), built as
 *   sc = W_2 . bf16(gelu(W_1 . bf16(soft_emb)))   (canvas_cast_bf16,
 *   canvas_gemm_bf16, canvas_gelu_bf16, canvas_gemm_bf16; no biases).
 */
canvas_status canvas_gelu_bf16(const float* in, void* out, size_t n, canvas_stream_t stream);

/* Workspace (bytes) that canvas_moe needs; 0 for an invalid shape. */
size_t canvas_moe_workspace_size(int R, int D, int E, int F, int k, int Fs);

/*
 * canvas_moe -- a mixture-of-experts MLP block on R tokens.
 *
 * Defined by [AIT] glossary "혼합 전문가(MoE)" (each token goes to its top-k
 * experts, which run in parallel and are summed with weights, plus a shared
 * expert every token passes through; the routing score is the exponential of
 * the router key's dot product with the input, renormalised and scaled) and
 * [TC] "아키텍처" (128 experts, 8 active + 1 shared).  The pages print no
 * expert MLP; the Gemma family's gated form is taken:
 *   s_e   = x . router_e                         (fp32 accumulation)
 *   top-k by s (equal scores: lower expert index first)
 *   w_j   = exp(s_j - s_max) / sum_{chosen} exp(s_i - s_max) * scale_e
 *   y_e   = W_down_e bf16(gelu(W_gate_e x) * (W_up_e x))   (GELU tanh form)
 *   out   = sum_j w_j y_{e_j}  (in choice order)  +  y_shared(x)
 *
 *   x        [R, D] bf16, 16-byte aligned
 *   router   [E, D] bf16 router keys
 *   expert_scale [E] fp32 or NULL (all 1)
 *   W_gate, W_up [E * F, D] bf16 (expert e: rows e*F ..), W_down [E * D, F] bf16
 *   Ws_gate, Ws_up [Fs, D], Ws_down [D, Fs] bf16: the shared expert (Fs = 0: none)
 *   out      [R, D] fp32 out, 16-byte aligned
 *   topk_idx [R, k] int32, topk_w [R, k] fp32: out, or NULL
 *   workspace, ws_bytes  >= canvas_moe_workspace_size(R, D, E, F, k, Fs)
 * Requires D, F, Fs multiples of 8, E a multiple of 8 up to 256, 1 <= k <= 16,
 * k <= E.  The experts run as grouped tensor-core GEMMs over the tokens
 * routed to them (each expert's rows padded to whole 128-row tiles).
 * Asynchronous on `stream`.
 */
canvas_status canvas_moe(const void* x, int R, int D, const void* router, int E, int k, const float* expert_scale,
                         const void* W_gate, const void* W_up, const void* W_down, int F,
                         const void* Ws_gate, const void* Ws_up, const void* Ws_down, int Fs,
                         float* out, int32_t* topk_idx, float* topk_w,
                         void* workspace, size_t ws_bytes, canvas_stream_t stream);

/*
 * canvas_count_committed -- committed positions of each canvas, for adaptive
 * stopping ("[논문리뷰] DiffusionGemma Technical Report" §1: the loop stops
 * once every position of the canvas is committed).
 *   commit_mask [rows] uint8 (canvas_sample's output), rows % canvas_len == 0
 *   counts [rows / canvas_len] int32 out: ones of each canvas's mask
 * Asynchronous on `stream`; the caller reads counts back to decide.
 */
canvas_status canvas_count_committed(const uint8_t* commit_mask, int rows, int canvas_len, int32_t* counts,
                                     canvas_stream_t stream);

/*
 * canvas_temperature_at -- host helper: the sampler temperature of denoising
 * step `step` of `steps` on a linear schedule from t_max (step 0) to t_min
 * (step steps - 1), [AIT] "섹션별 상세", sampling-loop paragraph (the
 * temperature falls from t_max to t_min over max_denoising_steps).  Pass the
 * result as canvas_sample's temperature.  steps <= 1 gives t_max.
 */
float canvas_temperature_at(int step, int steps, float t_max, float t_min);

/*
 * canvas_selftest_wait_timeout -- diagnostic; the method has no counterpart.
 *
 * Enqueues one kernel whose bounded device wait can never complete (an
 * mbarrier phase that nothing finishes), the same wait every pipelined kernel
 * of this library uses.  After the wait limit (2 s) the kernel records
 * CANVAS_ERR_TIMEOUT in the per-device status word and returns: the next
 * canvas_device_status() reports it (and clears it), and the context stays
 * usable.  Asynchronous on `stream`; CANVAS_ERR_CUDA if the launch fails.
 */
canvas_status canvas_selftest_wait_timeout(canvas_stream_t stream);

/*
 * canvas_gemm_bf16_noalloc -- canvas_gemm_bf16 without a caller workspace.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot hand the library a device buffer: code running inside a host
 * application whose allocator owns every byte of device memory and forbids
 * raw cudaMalloc, or that must not allocate after start-up (a fixed memory
 * budget, or a latency-critical path where an allocation could synchronise
 * the device).
 *
 * Same operation, arguments, layouts and result as canvas_gemm_bf16.  The
 * split-K scratch lives in one static device array of
 * CANVAS_GEMM_NOALLOC_SCRATCH_BYTES bytes inside the library; every device
 * that loads the library holds it until the process exits.  Shapes whose
 * scratch (canvas_gemm_workspace_size) exceeds that size return
 * CANVAS_ERR_WORKSPACE with a message.  No call allocates or frees device
 * memory.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All
 * calls share the one array: calls that may overlap on the GPU (different
 * streams, or different host threads, without ordering between them) race
 * on it and must be serialised by the caller.  The looked-up address is kept
 * for the life of the process: do not use this call on a device after
 * cudaDeviceReset() (the library's module, and the array with it, may be
 * loaded again at another address).  A, B and C must be 16-byte aligned
 * (CANVAS_ERR_ARG otherwise, before anything is enqueued).
 */
#define CANVAS_GEMM_NOALLOC_SCRATCH_BYTES (16u << 20)
canvas_status canvas_gemm_bf16_noalloc(const void* A, const void* B, int b_layout, float* C,
                                       int M, int N, int K, int accumulate, canvas_stream_t stream);

/*
 * Kernel timing hooks, for benchmarks.  When a pair of events is registered
 * for a kernel id, every later call on this thread records `start` on the
 * call's stream immediately before that kernel's launch and `stop` right
 * after it, so cudaEventElapsedTime gives the kernel's device time.  Events
 * are cudaEvent_t handles owned by the caller; pass NULL, NULL to clear.
 *   CANVAS_KERNEL_ATTENTION  -- the attention core of canvas_attention
 *   CANVAS_KERNEL_PREP       -- everything canvas_attention runs before it
 *                               (QKV projection, QK norm + RoPE, key prep)
 *   CANVAS_KERNEL_SAMPLER    -- the vocab reduction of canvas_sample
 *   CANVAS_KERNEL_SOFT_EMB   -- the soft-embedding GEMM of canvas_sample
 */
typedef enum {
  CANVAS_KERNEL_ATTENTION = 0,
  CANVAS_KERNEL_PREP = 1,
  CANVAS_KERNEL_SAMPLER = 2,
  CANVAS_KERNEL_SOFT_EMB = 3,
  CANVAS_KERNEL_COUNT = 4
} canvas_kernel_id;
canvas_status canvas_profile_events(int kernel_id, void* start_event, void* stop_event);

/* Number of kernels this library has launched in this process (host count). */
uint64_t canvas_kernel_launches(void);

/* Message of the last failed call on this thread ("" if none). */
const char* canvas_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device: CANVAS_OK, or the first error a kernel recorded since the
 * last read (CANVAS_ERR_BOUNDS, CANVAS_ERR_TIMEOUT, CANVAS_ERR_UNSUPPORTED).
 * This is the only call that synchronises.
 */
canvas_status canvas_device_status(canvas_stream_t stream);

/* Library version string. */
const char* canvas_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CANVAS_H_ */

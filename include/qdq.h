/*
 * qdq.h -- GB300 (sm_103a) dequantize-and-multiply kernels for GGML Q8_0 / Q4_K
 * weight matrices against f32 activations (the token-decode hot path).
 *
 * Sources (rustdoc pages of the qualia_core_db crate):
 *   "Module cuda_lane", Functions:
 *     q8_0_gemv_oracle_into / try_q8_0_cuda_gemv   -> qdq_q8_0_gemv
 *     try_q4k_soa_gemv                              -> qdq_q4k_gemv
 *     try_q4k_soa_fused_swiglu                      -> qdq_q4k_swiglu
 *     try_q4k_soa_qkv                               -> qdq_q4k_qkv
 *     try_q4k_soa_ffn_block / _ffn_block_residual   -> qdq_q4k_ffn_residual
 *     preload_q4k_soa_weights (one-time upload)     -> qdq_q8_0_pack / qdq_q4k_pack
 *   "Module cuda_lane", Goal (batch prefill-shaped GEMMs on tensor cores) and
 *   "weight_cache.rs", try_cuda_batch_gemv          -> qdq_q8_0_gemm_batch / qdq_q4k_gemm_batch /
 *                                                      qdq_q4k_swiglu_batch
 *   "QTensorEngine", dispatch_output_top1_chunked   -> qdq_q8_0_logits_argmax
 *   "QTensorEngine", dispatch_output_topk_chunked   -> qdq_topk_rows / qdq_q8_0_logits_topk
 *   "QTensorEngine", embedding_pipeline (Q6_K dequant + matmul on the GPU),
 *     dispatch_quantized_token_embedding, dispatch_gemm_into (Q6_K)
 *                                                   -> qdq_q6k_pack / _gemv / _get_rows
 *
 * Conventions for every call
 *   - W is row-major n_out x n_in (rows = outputs, the GGML convention).
 *     Activations are packed batch x n_in f32, outputs batch x n_out f32
 *     ("weight_cache.rs", try_cuda_batch_gemv doc comment).
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps a pointer after a call returns.
 *   - Every compute call is asynchronous and stream-ordered on `stream`
 *     (0 = the legacy default stream); nothing synchronises the host.
 *   - Calls return QDQ_OK or a negative status.  On a rejected argument (every
 *     status but QDQ_ERR_CUDA) nothing has been launched and every output
 *     buffer is untouched.  QDQ_ERR_CUDA from a call that launches several
 *     kernels (the FFN block, the batch GEMM, the argmax and top-k, QKV at batch > 1) can leave the
 *     kernels before the failing launch enqueued.  There is no fallback path:
 *     an unsupported shape is an error, never a silent slower route.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     start streaming its own weights while the previous kernel on the stream
 *     finishes, but it reads activations only after that kernel completed.
 *
 * Block formats (GGML, little-endian)
 *   Q8_0: 34-byte block per 32 weights: fp16 d, then int8 q[32]; w = d*q.
 *   Q4_K: 144-byte superblock per 256 weights: fp16 d, fp16 dmin, 12 bytes of
 *         eight 6-bit scales sc_j and eight 6-bit mins m_j, 128 bytes of 4-bit
 *         quants; sub-block j = weights 32j..32j+31; w = d*sc_j*q - dmin*m_j.
 *   Q6_K: 210-byte superblock per 256 weights: ql[128] (low 4 bits of each
 *         quant), qh[64] (high 2 bits), sixteen int8 scales, fp16 d (at byte
 *         208); weight e = d*scale[e/16]*(q_e - 32), q_e in 0..63, where weight
 *         128h + 32t + l (h < 2, t < 4, l < 32) takes its low 4 bits from the low
 *         (t < 2) or high (t >= 2) nibble of ql[64h + 32(t & 1) + l] and its high
 *         2 bits from bits 2t..2t+1 of qh[32h + l].
 *
 * Packed (device) formats -- produced once by qdq_*_pack, same byte count as
 * the GGML input, laid out as planes so that every kernel load is a 16-byte
 * aligned vector load:
 *   Q8_0 packed: [ q plane: n_out*n_in int8, row-major ]
 *                [ d plane: n_out*(n_in/32) fp16, row-major ]
 *   Q4_K packed: [ q plane: n_out*(n_in/2) bytes; weight e of a row is nibble
 *                  (e & 1) (0 = low) of byte e/2 ]
 *                [ header plane: n_out*(n_in/256) records of 16 bytes:
 *                  word0 = d | dmin << 16 (fp16 bits); words 1..3 form a
 *                  96-bit little-endian field with sc_j at bits 12j..12j+5
 *                  and m_j at bits 12j+6..12j+11 ]
 *   Q6_K packed: rows of qdq_q6k_packed_bytes(1, n_in) bytes (the 210/256
 *                bytes per weight padded to a multiple of 16; no padding when
 *                n_in % 2048 == 0): [ low-bit plane n_in/2 | high-bit plane
 *                n_in/4 | int8 scales n_in/16 | fp16 d n_in/128 | zeros ];
 *                32-weight block b: low bits at 16b (byte i of word c: weight
 *                8c+i in the low nibble, 8c+4+i in the high nibble), high bits
 *                at n_in/2 + 8b (byte i of word h: weights 16h+i, 16h+4+i,
 *                16h+8+i, 16h+12+i at bits 0-1, 2-3, 4-5, 6-7).
 */
#ifndef QDQ_H
#define QDQ_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------- */
#define QDQ_OK               0
#define QDQ_ERR_NULL        -1  /* a required pointer is NULL */
#define QDQ_ERR_DIMS        -2  /* a dimension is <= 0, not a whole number of blocks, or out of range */
#define QDQ_ERR_ALIGN       -3  /* a pointer does not meet the stated alignment */
#define QDQ_ERR_UNSUPPORTED -4  /* valid arguments this build does not handle (e.g. n_in too large) */
#define QDQ_ERR_CUDA        -5  /* a CUDA runtime call failed; see qdq_last_cuda_error() */
#define QDQ_ERR_ALIAS       -6  /* an output overlaps an input it may not overlap */
#define QDQ_ERR_SCRATCH     -7  /* the request does not fit the library's fixed scratch array */

/* Human-readable name of a status code (static string). */
const char *qdq_status_string(int status);
/* cudaError_t of the most recent QDQ_ERR_CUDA returned on the calling thread (0 if none). */
int qdq_last_cuda_error(void);
/* Library version string (static). */
const char *qdq_version(void);

/* ---- limits --------------------------------------------------------------- */
/* Largest supported batch for the GEMV-family calls. */
#define QDQ_MAX_GEMV_BATCH 8
/* Largest supported n_in for the GEMV-family calls (activations are staged in
 * shared memory: batch_group * n_in * 4 bytes per CTA). */
#define QDQ_MAX_GEMV_N_IN 32768

/* ---- one-time repack (the pages' preload step) ----------------------------
 * "Module cuda_lane", Functions: preload_q4k_soa_weights -- bulk upload once
 * at plan build.  Converts a row-major GGML matrix already resident on the
 * device into the packed planes above.  `ggml` and `packed` are device
 * pointers; `packed` must hold qdq_*_packed_bytes(n_out, n_in) bytes, be
 * 16-byte aligned and must not overlap `ggml`.  Q8_0 needs n_in % 32 == 0,
 * Q4_K needs n_in % 256 == 0.
 */
size_t qdq_q8_0_packed_bytes(int n_out, int n_in);   /* n_out*n_in/32*34, 0 on bad dims */
size_t qdq_q4k_packed_bytes(int n_out, int n_in);    /* n_out*n_in/256*144, 0 on bad dims */
int qdq_q8_0_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t stream);
int qdq_q4k_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t stream);

/* ---- dequantisation (verification aid) ------------------------------------
 * Writes the f32 weights of a packed matrix, row-major n_out x n_in, into
 * `out` (4-byte aligned).  Q8_0: d*q (exact in f32).  Q4_K: the single f32
 * rounding of d*sc_j*q - dmin*m_j.  Same block definitions as above.
 */
int qdq_q8_0_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t stream);
int qdq_q4k_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t stream);

/* ---- GEMV: y[b, r] = sum_k w[r, k] * x[b, k] -------------------------------
 * "Module cuda_lane", Functions: try_q8_0_cuda_gemv, q8_0_gemv_oracle_into,
 * try_q4k_soa_gemv.  W: packed (16-byte aligned).  x: batch x n_in f32,
 * 16-byte aligned.  y: batch x n_out f32, 4-byte aligned, must not overlap W
 * or x.  1 <= batch <= QDQ_MAX_GEMV_BATCH.  Error against the exact sum:
 * <= 1e-5 * sum_k |w[r,k]| |x[b,k]| for every finite input (f32 arithmetic; for
 * Q4_K also where d*sc_j*q and dmin*m_j cancel).  Batch 1 can opt into the
 * faster fixed-point arithmetic of QDQ_OPT_XS_FLOAT_X = 0, with the bound
 * stated there (the same holds for the SwiGLU, QKV and FFN calls below).
 */
int qdq_q8_0_gemv(const void *W, const float *x, float *y,
                  int n_out, int n_in, int batch, cudaStream_t stream);
int qdq_q4k_gemv(const void *W, const float *x, float *y,
                 int n_out, int n_in, int batch, cudaStream_t stream);

/* ---- fused SwiGLU expansion -------------------------------------------------
 * "Module cuda_lane", Functions: try_q4k_soa_fused_swiglu:
 *   mid[b, i] = silu(gate_i . x_b) * (up_i . x_b),  silu(z) = z / (1 + e^-z),
 * one kernel reading x once for both Q4_K matrices.  Wg, Wu: packed Q4_K
 * n_ff x n_embd.  x: batch x n_embd (16-byte aligned).  mid: batch x n_ff,
 * must not overlap any input.
 */
int qdq_q4k_swiglu(const void *Wg, const void *Wu, const float *x, float *mid,
                   int n_ff, int n_embd, int batch, cudaStream_t stream);

/* ---- Q6_K: repack, dequantisation, GEMV, embedding lookup -------------------
 * "QTensorEngine": embedding_pipeline (Q6_K embedding dequant + matmul on the
 * GPU, no CPU dequant), dispatch_quantized_token_embedding (raw quantised
 * embedding bytes uploaded, used without CPU dequant) and dispatch_gemm_into
 * (quantised GEMM into the caller's buffer, Q6_K).
 * qdq_q6k_packed_bytes: bytes of the packed matrix (0 on bad dims: n_in % 256).
 * qdq_q6k_pack: as qdq_q4k_pack, for GGML Q6_K input (n_out*n_in/256*210 bytes).
 * qdq_q6k_dequant: w = d*scale*(q - 32), exact in f32, into `out` (n_out x n_in).
 * qdq_q6k_gemv: as qdq_q8_0_gemv (same pointer, alignment, aliasing and batch
 *   rules); error <= 1e-5 * sum_k |w[r,k]| |x[b,k]| for every finite input.
 * qdq_q6k_get_rows: embedding lookup, out[i, :] = the dequantised row ids[i] of
 *   the packed n_rows x n_in matrix W, for i < n_ids (0 = nothing to do).  ids:
 *   int32 device array (4-byte aligned), read after the previous kernel on the
 *   stream; an id outside [0, n_rows) gives a row of NaN.  out: n_ids x n_in
 *   f32 (4-byte aligned), must not overlap W or ids.
 */
size_t qdq_q6k_packed_bytes(int n_out, int n_in);
int qdq_q6k_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t stream);
int qdq_q6k_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t stream);
int qdq_q6k_gemv(const void *W, const float *x, float *y, int n_out, int n_in, int batch, cudaStream_t stream);
int qdq_q6k_get_rows(const void *W, const int *ids, float *out, int n_ids, int n_rows, int n_in,
                     cudaStream_t stream);

/* ---- output projection with on-device argmax --------------------------------
 * "QTensorEngine", dispatch_output_top1_chunked (GPU block argmax, k = 1): the
 * output projection with an on-device argmax epilogue, so a decode step reads
 * back one token instead of the logits.
 *   logits[b, t] = W_t . x_b (a Q8_0 GEMV, as qdq_q8_0_gemv), then
 *   index[b] = the first t with the largest logits[b, t], value[b] = that logit
 *   (a NaN logit counts as the largest: the first NaN wins).
 * W: packed Q8_0 n_vocab x n_in (16-byte aligned).  x: batch x n_in (16-byte
 * aligned).  logits: batch x n_vocab f32 scratch the caller owns, overwritten
 * (4-byte aligned).  index (int32), value (f32): batch entries each, 4-byte
 * aligned.  No output may overlap an input or another output.  Two kernels on
 * `stream`; nothing is read back.
 */
int qdq_q8_0_logits_argmax(const void *W, const float *x, float *logits, int *index, float *value,
                           int n_vocab, int n_in, int batch, cudaStream_t stream);

/* ---- on-device top-k of the logits --------------------------------------------
 * "QTensorEngine", dispatch_output_topk_chunked (the logits stay on the GPU, a
 * top-k kernel reduces them per chunk, only K (id, logit) candidates are read
 * back).  For each of `batch` rows of n logits (row-major, 4-byte aligned):
 * index[b, j], value[b, j] (j < k, int32 / f32, 4-byte aligned) = the j-th entry
 * of the order NaN first (the first NaN first), then larger logits first, equal
 * logits (+0 == -0) by smaller index; value holds the logit's exact bits.
 * 1 <= k <= min(n, QDQ_MAX_TOPK).  workspace: qdq_topk_workspace_bytes(n, batch,
 * k) bytes of caller scratch (16-byte aligned, overwritten; the size depends on
 * the current device).  Outputs and workspace may overlap nothing.  Several
 * kernels on `stream`; k = 1 is the argmax kernel of qdq_q8_0_logits_argmax (the
 * same order), one launch, the workspace untouched.
 * qdq_q8_0_logits_topk: the Q8_0 output projection (as qdq_q8_0_logits_argmax)
 * followed by the top-k; logits: batch x n_vocab scratch the caller owns (it
 * receives the logits).  At batch 1 the projection's CTAs write the k best
 * (logit, index) keys of their own rows as they finish, and only merge kernels
 * follow; same results as the separate top-k.  k = 1 runs as
 * qdq_q8_0_logits_argmax.
 */
#define QDQ_MAX_TOPK 64
size_t qdq_topk_workspace_bytes(int n, int batch, int k);   /* 0 on bad arguments */
int qdq_topk_rows(const float *logits, int n, int batch, int k, void *workspace, int *index, float *value,
                  cudaStream_t stream);
int qdq_q8_0_logits_topk(const void *W, const float *x, float *logits, void *workspace, int *index, float *value,
                         int n_vocab, int n_in, int batch, int k, cudaStream_t stream);

/* ---- fused QKV projection ---------------------------------------------------
 * "Module cuda_lane", Functions: try_q4k_soa_qkv (one activation, one fused
 * kernel; GQA: K and V only for rows below n_kv):
 *   q[b, r] = Wq_r . x_b (r < n_q),  k[b, r] = Wk_r . x_b,  v[b, r] = Wv_r . x_b (r < n_kv).
 * Wq: packed Q4_K n_q x n_embd; Wk, Wv: packed Q4_K n_kv x n_embd, 1 <= n_kv <= n_q
 * (16-byte aligned).  x: batch x n_embd (16-byte aligned).  q: batch x n_q; k, v:
 * batch x n_kv (4-byte aligned); no output may overlap an input or another output.
 * Batch 1 is one kernel over the rows of Wq, Wk, Wv; batch 2..8 is three GEMV
 * launches.  Error bound as qdq_q4k_gemv.
 */
int qdq_q4k_qkv(const void *Wq, const void *Wk, const void *Wv, const float *x,
                float *q, float *k, float *v, int n_q, int n_kv, int n_embd, int batch,
                cudaStream_t stream);

/* ---- FFN block with on-device residual --------------------------------------
 * "Module cuda_lane", Functions: try_q4k_soa_ffn_block_residual:
 *   out = residual + W_down . swiglu(W_gate x, W_up x)
 * (pre-norm-free: x is used as given).  Two kernels on `stream`; `mid` stays
 * on the device.  Wg, Wu: packed Q4_K n_ff x n_embd; Wd: packed Q4_K
 * n_embd x n_ff.  x, residual, out: batch x n_embd.  mid_workspace: caller-
 * owned batch x n_ff f32 scratch, 16-byte aligned, overwritten.  out may be
 * exactly `residual` (in-place residual add) but may not overlap anything else.
 */
int qdq_q4k_ffn_residual(const void *Wg, const void *Wu, const void *Wd,
                         const float *x, const float *residual, float *out,
                         float *mid_workspace, int n_embd, int n_ff, int batch,
                         cudaStream_t stream);

/* ---- FFN block without caller scratch (allocates nothing) -------------------
 * No counterpart on the reference pages: an addition for callers that may not
 * allocate device memory -- e.g. a plug-in whose host application owns all GPU
 * memory through its own pool, or a decode loop that must not pay for
 * cudaMalloc/cudaFree.  Same operation, arguments and error behaviour as
 * qdq_q4k_ffn_residual, but `mid` lives in a fixed device array inside the
 * library (QDQ_NOALLOC_FFN_MAX_MID floats, 1 MiB, held by every GPU that loads
 * the library until the process exits); nothing is allocated.
 *   - batch * n_ff > QDQ_NOALLOC_FFN_MAX_MID returns QDQ_ERR_SCRATCH.
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the one array: calls that overlap on the GPU (other
 *     streams, other threads) race on it and must be serialised by the caller.
 */
#define QDQ_NOALLOC_FFN_MAX_MID 262144
int qdq_q4k_ffn_residual_noalloc(const void *Wg, const void *Wu, const void *Wd,
                                 const float *x, const float *residual, float *out,
                                 int n_embd, int n_ff, int batch, cudaStream_t stream);

/* ---- batch-prefill GEMMs on tensor cores -----------------------------------
 * "Module cuda_lane", Goal (tensor-core GEMM for batch prefill-shaped work)
 * and "weight_cache.rs", try_cuda_batch_gemv (hidden packed batch x n_in,
 * W row-major n_out x n_in, out batch x n_out; the reference pads to 16 and
 * trims, this call masks instead):
 *   Y[m, r] = sum_k bf16(X[m, k]) * bf16(w[r, k])   (f32 accumulation)
 * with w the exact f32 dequantised weight (Q8_0 d*q; Q4_K RN(d*sc*q - dmin*m)).
 * W: packed Q8_0 / Q4_K (16-byte aligned).  X: M x n_in f32 (16-byte aligned).
 * Y: M x n_out f32 (16-byte aligned), must not overlap W, X or workspace.
 * workspace: caller-owned scratch of qdq_gemm_batch_workspace_bytes(M, n_out,
 * n_in) bytes (0 when no device can be queried), 256-byte aligned, overwritten
 * with X rounded to bf16 when M > 32 (unused for M <= 32, where the kernel
 * rounds X itself; qdq_q4k_swiglu_batch: M > 16 and M <= 16).  K is split across the CTAs of a thread-block cluster when
 * the output tiles alone cannot fill the SMs; the splits' partial tiles are
 * added in shared memory, in a fixed order.
 * Requires n_in % 64 == 0 (Q4_K: % 256) and n_out % 128 == 0; M >= 1 (tail
 * masked).  Results do not depend on the order in which CTAs run (split-K
 * partials are added in a fixed order).
 * Error against the exact sum: <= 4e-3 * sum_k |w[r,k]| |X[m,k]|.
 * qdq_q4k_swiglu_batch: the SwiGLU expansion for M tokens ("Module cuda_lane",
 * try_q4k_soa_fused_swiglu, prefill-shaped): mid[m, i] = silu(g[m, i]) * u[m, i]
 * with g, u the two GEMMs above against Wg, Wu (packed Q4_K n_ff x n_embd), in
 * one kernel; workspace of qdq_q4k_swiglu_batch_workspace_bytes(M, n_ff, n_embd).
 */
size_t qdq_gemm_batch_workspace_bytes(int M, int n_out, int n_in);
int qdq_q8_0_gemm_batch(const void *W, const float *X, float *Y, void *workspace,
                        int n_out, int n_in, int M, cudaStream_t stream);
int qdq_q4k_gemm_batch(const void *W, const float *X, float *Y, void *workspace,
                       int n_out, int n_in, int M, cudaStream_t stream);
size_t qdq_q4k_swiglu_batch_workspace_bytes(int M, int n_ff, int n_embd);
int qdq_q4k_swiglu_batch(const void *Wg, const void *Wu, const float *X, float *mid, void *workspace,
                         int n_ff, int n_embd, int M, cudaStream_t stream);

/* ---- pipeline health -------------------------------------------------------
 * Every wait inside the tensor-core pipeline is bounded (2 s wall clock); a
 * wait that runs out makes its CTA stop early instead of hanging, and counts
 * here.  Returns the count since the previous call and resets it (-1 on a
 * CUDA error).  Synchronous: it waits for the device.
 */
int qdq_pipeline_timeouts(void);

/* ---- debug build: device-side guards ----------------------------------------
 * A library built with -DQDQ_CHECKS (ggml_quantized_dequant_gb300._build.build(checks=True),
 * libqdq_checked.so) guards its shared-memory row buffers, weight-row and
 * activation indices, output indices and bulk-copy alignment inside the kernels:
 * an index out of bounds skips that access and sets a bit of a device status word
 * (QDQ_CHECK_* in the library's internal header: 1 shared memory, 2 weight row,
 * 4 output, 8 copy alignment) instead of trapping.  qdq_check_status waits for the
 * device, returns the or of the bits since its previous call and clears them (-1
 * on a CUDA error); in the normal build it returns 0.  qdq_checks_enabled: 1 in
 * the debug build, else 0.
 */
int qdq_check_status(void);
int qdq_checks_enabled(void);

/* ---- launch round trip -------------------------------------------------------
 * "QTensorEngine", bench_empty_submit_roundtrip (the fixed submit-to-completion
 * latency, measured with no compute): launches one empty kernel (one thread) on
 * `stream`; a caller times n of these each followed by a synchronisation.
 */
int qdq_noop(cudaStream_t stream);

/* ---- launch options (same work, different launch shape; for measurement) -- */
#define QDQ_OPT_PDL          1  /* 1 (default): programmatic dependent launch on; 0: plain launches */
#define QDQ_OPT_L2_PREFETCH  2  /* L2 prefetch of weight rows.  0 (default): automatic -- the batch-1 direct-load kernel
                                   prefetches nothing, the ring kernel's Q8_0 GEMV prefetches the rows its first ring fill
                                   leaves out when they fit in half the L2; 1: every GEMV CTA prefetches all its rows first;
                                   2: every ring-kernel CTA prefetches the rows its first ring fill leaves out; 3: no prefetch */
#define QDQ_OPT_CTAS_PER_SM  3  /* GEMV-family CTAs per SM, 1..4; 0 (default): automatic (batch-1 direct-load kernel: as
                                   many as fit; ring kernel: 2 for the FFN kernels, else 1; batch 2..8: 1) */
#define QDQ_OPT_XS_GROUPS    4  /* batch-1 GEMV groups of slice warps per CTA, 0 = automatic (default: 1 in the
                                   direct-load kernel), 1..16 */
#define QDQ_OPT_XS_STAGES    5  /* batch-1 GEMV: ring slots per consumer group (ring kernel), or the register depth
                                   1 / 2 (direct-load kernel); 0 = automatic (default), 1..16 */
/* Arithmetic of the batch-1 kernels (qdq_q8_0_gemv and qdq_q4k_gemv at batch 1,
 * qdq_q4k_swiglu, qdq_q4k_qkv, the output projections and both FFN calls at batch 1):
 *   1 (default): weights converted exactly to f32 and multiplied with f32 FMAs
 *     (Q4_K: quants shifted by the sub-block's integer offset before they are
 *     summed): within 1e-5 sum |w||x| of the exact sum for every finite input.
 *   0 (opt-in, faster): each 32-activation block becomes 24-bit block fixed
 *     point X_j = rint(x_j 2^e), |X_j| <= 2^22, and block dot products are
 *     exact integer byte dot products, scaled in f32.  Error against the exact
 *     sum <= 2^-22 sum_blocks max_j |x_j| sum_j |w_j| + f32 rounding: a bound
 *     relative to each block's largest activation, so it exceeds
 *     1e-5 sum |w||x| where a row's weights sit on the small activations of
 *     blocks whose largest activation they skip.  A block with an inf or NaN
 *     activation gives NaN outputs. */
#define QDQ_OPT_XS_FLOAT_X   6
/* Batch-1 kernel of the f32 arithmetic: 0 (default) the direct-load kernel (weights straight into
 * registers, small CTAs of one group of slice warps, as many per SM as fit); 1 the shared-memory
 * ring kernel (a producer warp streams weights into a ring sized to half an SM, so that the next
 * kernel's CTA can start streaming beside it).  Same results within the stated bound; the
 * fixed-point arithmetic always runs in the ring kernel. */
#define QDQ_OPT_BATCH1_KERNEL 7
/* Sets a process-wide option; returns the previous value, or QDQ_ERR_DIMS for a bad key/value. */
int qdq_set_option(int key, int value);

#ifdef __cplusplus
}
#endif

#endif /* QDQ_H */

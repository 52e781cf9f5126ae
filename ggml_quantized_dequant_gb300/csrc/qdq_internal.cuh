// Internal helpers shared by the qdq kernels (not part of the public ABI).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "qdq.h"

namespace qdq {

// ---------------------------------------------------------------- host side

// Process-wide launch options (see QDQ_OPT_* in qdq.h).
int opt_pdl();
int opt_l2_prefetch();
int opt_ctas_per_sm();
// The CTAs-per-SM option, or `dflt` where it is left automatic (0).
inline int ctas_per_sm_or(int dflt) {
  const int v = opt_ctas_per_sm();
  return v > 0 ? v : dflt;
}
int opt_xs_groups();
int opt_xs_stages();
int opt_xs_float_x();
int opt_batch1_kernel();

// Per-device facts queried once (SM count, opt-in shared memory).
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
  int smem_per_sm;
  int reserved_smem_per_block;
  int regs_per_sm;
  int l2_bytes;
};

// Dynamic shared memory for a streaming GEMV CTA: at least `need`, and when
// programmatic dependent launch is on, enough that an SM holds this kernel's
// CTAs plus one CTA of the next kernel but no more -- so the next kernel's
// weight prefetch runs exactly one kernel ahead instead of flooding L2.
size_t gemv_smem_bytes(const DeviceInfo &di, size_t need);

// Grid of a streaming GEMV: CTAs-per-SM x SMs, but no more CTAs than tasks of
// `rows_per_task` output rows.
inline int gemv_grid(const DeviceInfo &di, int n_out, int rows_per_task) {
  const int g = di.sm_count * ctas_per_sm_or(1);
  const int max_g = (n_out + rows_per_task - 1) / rows_per_task;
  return g < max_g ? g : max_g;
}
// Returns 0 and fills `out` for the current device, or a cudaError_t.
cudaError_t device_info(DeviceInfo *out);


// Records a CUDA error for qdq_last_cuda_error() and returns QDQ_ERR_CUDA.
int fail_cuda(cudaError_t e);

// Raises `func`'s dynamic shared-memory cap on the current device to at least
// `bytes` (once per kernel and device; thread-safe).
cudaError_t allow_dynamic_smem(const void *func, int bytes);

// Launch `kernel` with optional programmatic dependent launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opt_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// True when [a, a+na) and [b, b+nb) overlap (byte ranges).
inline bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return na && nb && pa < pb + nb && pb < pa + na;
}
inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Argument checks of the FFN block (qdq_q4k_ffn_residual); `mid` NULL skips the
// checks of the intermediate buffer (the allocation-free entry point owns it).
int check_ffn_residual(const void *Wg, const void *Wu, const void *Wd, const float *x, const float *residual,
                       const float *out, const float *mid, int n_embd, int n_ff, int batch);

// Kernel launchers (defined in the per-kernel translation units).
int launch_q8_0_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t s);
int launch_q4k_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t s);
int launch_q8_0_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t s);
int launch_q4k_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t s);
int launch_q8_0_gemv(const void *W, const float *x, float *y, int n_out, int n_in, int batch,
                     cudaStream_t s);
// Q4_K GEMV family.  mode 0: y = W x;  mode 1: y = silu(Wg x) * (Wu x) (W2 = Wu);
// mode 2: y = residual + W x.
int launch_q4k_gemv(int mode, const void *W, const void *W2, const float *x, const float *residual,
                    float *y, int n_out, int n_in, int batch, cudaStream_t s);
// Batch-1 "x-stationary" GEMV fast path (qdq_gemv_xs.cu); fmt 0 = Q8_0,
// 1 = Q4_K with mode 0/1/2 as launch_q4k_gemv, 2 = Q6_K (mode 0).
bool gemv_xs_supported(int n_in, int batch, int fmt);
// Fused Q4_K QKV projection at batch 1 (n_in as gemv_xs_supported allows for Q4_K).
int launch_gemv_xs_qkv(const void *Wq, const void *Wk, const void *Wv, const float *x, float *q, float *k, float *v,
                       int n_q, int n_kv, int n_in, cudaStream_t s);
int launch_gemv_xs(int fmt, int mode, const void *W, const void *W2, const float *x, const float *residual,
                   float *y, int n_out, int n_in, cudaStream_t s);
// Top-k of each row of a logits matrix (qdq_topk.cu); the workspace holds the
// candidate keys of two merge rounds.
size_t topk_workspace_bytes(int n, int batch, int k);
int launch_topk_rows(const float *logits, int n, int batch, int k, void *workspace, int *index, float *value,
                     cudaStream_t s);
// The merge rounds alone, for one row whose `count` candidate keys (each CTA's k best,
// in any order) are at the start of the workspace (the batch-1 projection writes them).
int launch_topk_merge(int count, int k, void *workspace, const float *logits, int n, int *index, float *value,
                      cudaStream_t s);
// Batch-1 direct-load GEMV (qdq_gemv_dl.cu), f32 arithmetic; same fmt / mode as launch_gemv_xs.
int launch_gemv_dl(int fmt, int mode, const void *W, const void *W2, const float *x, const float *residual, float *y,
                   int n_out, int n_in, cudaStream_t s);
int launch_gemv_dl_qkv(const void *Wq, const void *Wk, const void *Wv, const float *x, float *q, float *k, float *v,
                       int n_q, int n_kv, int n_in, cudaStream_t s);
// Batch-1 Q8_0 GEMV whose CTAs also write the k best keys (topk_key) of their rows to
// cand[cta * k ...]; *n_cand = CTAs * k.
int launch_gemv_dl_topk(const void *W, const float *x, float *y, int n_out, int n_in, uint64_t *cand, int k,
                        int *n_cand, cudaStream_t s);
// Upper bound of the CTAs launch_gemv_dl_topk runs on the current device (0 on error).
int gemv_dl_max_ctas();
// Q6_K (qdq_q6k.cu): repack, dequantisation, embedding-row lookup, GEMV (batch 1..8).
int launch_q6k_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t s);
int launch_q6k_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t s);
int launch_q6k_get_rows(const void *W, const int *ids, float *out, int n_ids, int n_rows, int n_in, cudaStream_t s);
int launch_q6k_gemv(const void *W, const float *x, float *y, int n_out, int n_in, int batch, cudaStream_t s);
// Pipeline-timeout counters of the translation units that run bounded waits:
// each returns its count since the last call and resets it (-1 on CUDA error).
int read_gemm_timeouts();
int read_xs_timeouts();
int read_dl_timeouts();
// Tensor-core batch GEMMs (qdq_gemm_tc.cu).  The workspace holds X in bf16, the
// split-K partial tiles and one ticket per output tile; gemm_workspace_bytes is its
// size for `na` weight matrices on the current device (0 on a CUDA error).
size_t gemm_workspace_bytes(int M, int n_out, int n_in, int na);
int launch_q8_0_gemm_batch(const void *W, const float *X, float *Y, void *workspace, int n_out,
                           int n_in, int M, cudaStream_t s);
int launch_q4k_gemm_batch(const void *W, const float *X, float *Y, void *workspace, int n_out,
                          int n_in, int M, cudaStream_t s);
int launch_q4k_swiglu_batch(const void *Wg, const void *Wu, const float *X, float *mid, void *workspace, int n_ff,
                            int n_embd, int M, cudaStream_t s);

// ---------------------------------------------------------------- device side

// Debug-build guards (compiled with -DQDQ_CHECKS): a guarded access whose index
// is out of bounds is skipped and its check bit is or-ed into this translation
// unit's status word (qdq_check_status reads and clears them all); nothing traps.
// In the normal build QDQ_GUARD is `true` and costs nothing.
#define QDQ_CHECK_SMEM 1u     // a shared-memory index past its buffer
#define QDQ_CHECK_ROW 2u      // a weight row or activation index past its matrix
#define QDQ_CHECK_OUT 4u      // an output index past its buffer
#define QDQ_CHECK_ALIGN 8u    // a bulk copy not 16-byte aligned or sized
#ifdef QDQ_CHECKS
static __device__ unsigned int g_check_status = 0;
#define QDQ_GUARD(cond, bit) ((cond) ? true : (atomicOr(&g_check_status, (bit)), false))
// Defines this translation unit's reader of its status word (read and clear).
#define QDQ_CHECK_READER(name)                                                           \
  int name() {                                                                           \
    unsigned int v = 0, zero = 0;                                                        \
    if (cudaMemcpyFromSymbol(&v, g_check_status, sizeof(v)) != cudaSuccess) return -1; \
    if (cudaMemcpyToSymbol(g_check_status, &zero, sizeof(zero)) != cudaSuccess) return -1; \
    return int(v);                                                                       \
  }
#else
#define QDQ_GUARD(cond, bit) true
#define QDQ_CHECK_READER(name) \
  int name() { return 0; }
#endif
int read_checks_dl();
int read_checks_xs();
int read_checks_gemm();
int read_checks_topk();
int read_checks_q6k();

// A logit and its index as a 64-bit key whose unsigned order is the top-k order: a
// NaN above every number, then larger values, equal values (+0 = -0) by smaller
// index.  The high word maps the float to an order-preserving integer (every NaN
// to the largest), the low word is the complement of the index; key 0 is below
// every real key.
__device__ __forceinline__ uint64_t topk_key(float v, uint32_t index) {
  uint32_t o;
  if (v != v) {
    o = 0xFFFFFFFFu;
  } else {
    uint32_t b = __float_as_uint(v);
    if ((b & 0x7FFFFFFFu) == 0) b = 0;  // -0 sorts as +0
    o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  return (uint64_t(o) << 32) | uint64_t(~index);
}

// Warp-wide bitonic sort of 64 keys, descending: lane l holds positions l (a) and
// 32 + l (b).  Strides below 32 are shuffles, the 32 stride a register swap.
__device__ __forceinline__ uint64_t shfl_xor_key(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, uint32_t(v), m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, uint32_t(v >> 32), m);
  return (uint64_t(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t key_cmpx(uint64_t mine, uint64_t other, int p, int j, int k) {
  const bool take_max = ((p & j) == 0) == ((p & k) == 0);  // lower position of a descending run keeps the max
  return take_max ? (mine > other ? mine : other) : (mine < other ? mine : other);
}
__device__ __forceinline__ void warp_merge_desc(uint64_t &a, uint64_t &b, int lane, int k) {
  // the bitonic merge steps of stage k (k = 64: a bitonic sequence -> descending)
  int j = k >> 1;
  if (j == 32) {
    const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
    j = 16;
  }
  for (; j > 0; j >>= 1) {
    const uint64_t oa = shfl_xor_key(a, j), ob = shfl_xor_key(b, j);
    a = key_cmpx(a, oa, lane, j, k);
    b = key_cmpx(b, ob, lane + 32, j, k);
  }
}
__device__ __forceinline__ void warp_sort64_desc(uint64_t &a, uint64_t &b, int lane) {
#pragma unroll 1
  for (int k = 2; k <= 64; k <<= 1) {
    if (k == 64) {
      warp_merge_desc(a, b, lane, 64);
    } else {
      for (int j = k >> 1; j > 0; j >>= 1) {
        const uint64_t oa = shfl_xor_key(a, j), ob = shfl_xor_key(b, j);
        a = key_cmpx(a, oa, lane, j, k);
        b = key_cmpx(b, ob, lane + 32, j, k);
      }
    }
  }
}
// (ta, tb) <- the 64 largest of two descending 64-key lists (ta, tb) and (a, b), descending:
// the element-wise maximum of one list and the other reversed is bitonic and holds them.
__device__ __forceinline__ void warp_top64_merge(uint64_t &ta, uint64_t &tb, uint64_t a, uint64_t b, int lane) {
  const uint64_t ra = shfl_xor_key(b, 31), rb = shfl_xor_key(a, 31);  // positions 63 - l and 31 - l of (a, b)
  ta = ta > ra ? ta : ra;
  tb = tb > rb ? tb : rb;
  warp_merge_desc(ta, tb, lane, 64);
}

// Programmatic dependent launch: let the next grid on the stream start early.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until every prerequisite grid has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Named barrier over `threads` threads (a multiple of 32); barrier 0 is __syncthreads.
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bulk L2 prefetch of [p, p+bytes): p and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetch the byte range [lo, hi) of a buffer whose valid extent is
// [base, base+total) into L2, rounded inward to 16-byte boundaries, in chunks.
__device__ __forceinline__ void prefetch_range_l2(const uint8_t *base, uint64_t total, uint64_t lo,
                                                  uint64_t hi) {
  lo = (lo + 15) & ~uint64_t(15);
  hi = hi < total ? hi : total;
  hi &= ~uint64_t(15);
  constexpr uint64_t kChunk = 32768;
  for (uint64_t a = lo; a < hi; a += kChunk) {
    const uint64_t n = (hi - a) < kChunk ? (hi - a) : kChunk;
    bulk_prefetch_l2(base + a, static_cast<uint32_t>(n));
  }
}

// ---- shared-memory pipelines (mbarrier + bulk async copies) -----------------
// Every wait is bounded by a wall-clock limit: a wait that runs out returns
// false and the caller winds its CTA down instead of hanging.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_try_wait, but the thread may sleep (up to about a millisecond) until the
// phase completes instead of returning at once: waiting warps leave the issue
// slots to the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity; false if the wall-clock limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(a, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk async copy global -> shared, completing on an mbarrier (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  if (!QDQ_GUARD(((smem_u32(dst) | uint32_t(reinterpret_cast<uintptr_t>(src)) | bytes) & 15u) == 0, QDQ_CHECK_ALIGN))
    return;
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// 128-bit coherent load of data an earlier kernel wrote.  A volatile asm with a
// memory clobber stays after a preceding griddepcontrol.wait; __ldg (ld.global.nc)
// is an invariant load the compiler may hoist above that wait.
__device__ __forceinline__ float4 ld_after_wait(const float4 *p) {
  float4 v;
  asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// 32-bit coherent load of data an earlier kernel wrote (see ld_after_wait).
__device__ __forceinline__ int ld_s32_after_wait(const int *p) {
  int v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 128-bit read-only load that does not allocate in L1 (streamed weights).
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Packed f32x2 arithmetic (sm_100+ builtins): two floats per instruction.
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 f2_bits(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// Exact small-integer -> f32 conversions without conversion instructions.  A
// value v placed in mantissa bits [p, p+k) of a float whose exponent makes bit
// p worth 1 reads as 2^(23-p) + v; subtracting 2^(23-p) (a packed f32x2 add)
// leaves v exactly.  Each select is one LOP3 with the mask as an immediate and
// the exponent pattern in a per-lane register: a LOP3 cannot take two uniform
// operands, so patterns kept in uniform registers would cost a move per use.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t c) {  // (a & MASK) | c
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
}
template <uint32_t MASK>
__device__ __forceinline__ uint32_t lop3_sel_xor(uint32_t a, uint32_t c) {  // MASK ? (a ^ c) : c
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
}

// Exponent patterns (and the matching subtraction constants), passed as kernel
// parameters and moved into per-lane registers once per thread (lane_magic).
struct Magic {
  uint32_t s8_0, s8_1;                // Q8_0: byte 0 / byte 1 of a half, sign bit flipped: 2^23, 2^15 (+128)
  uint32_t u4_0, u4_1, u4_2, u4_3;    // Q4_K: nibble 0..3 of a half: 2^23, 2^19, 2^15, 2^11
  uint32_t sc, m;                     // Q4_K header: 6-bit scale at bit 0 (2^23), 6-bit min at bit 6 (2^17)
  float2 b_s8, b_u4_01, b_u4_23, b_scm;  // subtraction constants
  float2 b_s8p;                       // Q8_0, byte-permute form: -(2^23 + 128) twice
  float2 b_q6;                        // Q6_K: -(2^23 + 32) twice (an unsigned byte at 2^23, minus the offset 32)
};
inline Magic make_magic() {
  Magic k;
  k.s8_0 = 0x4B000080u;
  k.s8_1 = 0x47008000u;
  k.u4_0 = 0x4B000000u;
  k.u4_1 = 0x49000000u;
  k.u4_2 = 0x47000000u;
  k.u4_3 = 0x45000000u;
  k.sc = 0x4B000000u;
  k.m = 0x48000000u;
  k.b_s8 = make_float2(-8388736.0f, -32896.0f);     // -(2^23 + 128), -(2^15 + 128)
  k.b_u4_01 = make_float2(-8388608.0f, -524288.0f);  // -2^23, -2^19
  k.b_u4_23 = make_float2(-32768.0f, -2048.0f);      // -2^15, -2^11
  k.b_scm = make_float2(-8388608.0f, -131072.0f);    // -2^23, -2^17
  k.b_s8p = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  k.b_q6 = make_float2(-8388640.0f, -8388640.0f);    // -(2^23 + 32)
  return k;
}
__device__ __forceinline__ uint32_t lane_reg(uint32_t v) { return __shfl_sync(0xffffffffu, v, threadIdx.x & 31); }
__device__ __forceinline__ float lane_regf(float v) { return __shfl_sync(0xffffffffu, v, threadIdx.x & 31); }
__device__ __forceinline__ Magic lane_magic(const Magic &k) {
  Magic r;
  r.s8_0 = lane_reg(k.s8_0);
  r.s8_1 = lane_reg(k.s8_1);
  r.u4_0 = lane_reg(k.u4_0);
  r.u4_1 = lane_reg(k.u4_1);
  r.u4_2 = lane_reg(k.u4_2);
  r.u4_3 = lane_reg(k.u4_3);
  r.sc = lane_reg(k.sc);
  r.m = lane_reg(k.m);
  r.b_s8 = f2(lane_regf(k.b_s8.x), lane_regf(k.b_s8.y));
  r.b_u4_01 = f2(lane_regf(k.b_u4_01.x), lane_regf(k.b_u4_01.y));
  r.b_u4_23 = f2(lane_regf(k.b_u4_23.x), lane_regf(k.b_u4_23.y));
  r.b_scm = f2(lane_regf(k.b_scm.x), lane_regf(k.b_scm.y));
  r.b_s8p = f2(lane_regf(k.b_s8p.x), lane_regf(k.b_s8p.y));
  r.b_q6 = f2(lane_regf(k.b_q6.x), lane_regf(k.b_q6.y));
  return r;
}

// Four signed int8 in `w` -> exact floats as two pairs (q0,q1), (q2,q3): the sign bits
// flipped (q + 128 per byte), then each byte permuted under the exponent bits of 2^23
// (one byte permute per quant, no shifts) and 2^23 + 128 taken off.  In the batch-1 GEMV
// this measured 6 % faster per up projection than select-and-xor operations on the ALU.
__device__ __forceinline__ void s8x4_to_f2(uint32_t w, const Magic &k, float2 &q01, float2 &q23) {
  const uint32_t u = w ^ 0x80808080u;
  q01 = __fadd2_rn(f2_bits(__byte_perm(u, k.u4_0, 0x7650), __byte_perm(u, k.u4_0, 0x7651)), k.b_s8p);
  q23 = __fadd2_rn(f2_bits(__byte_perm(u, k.u4_0, 0x7652), __byte_perm(u, k.u4_0, 0x7653)), k.b_s8p);
}
// The same by bit selects with the sign flip (one LOP3 per quant): what the tensor-core
// GEMM's dequantising warps use (the byte-permute form measured 1-2 % slower there).
__device__ __forceinline__ void s8x4_to_f2_sel(uint32_t w, const Magic &k, float2 &q01, float2 &q23) {
  const uint32_t hi = w >> 16;
  q01 = __fadd2_rn(f2_bits(lop3_sel_xor<0x000000FFu>(w, k.s8_0), lop3_sel_xor<0x0000FF00u>(w, k.s8_1)), k.b_s8);
  q23 = __fadd2_rn(f2_bits(lop3_sel_xor<0x000000FFu>(hi, k.s8_0), lop3_sel_xor<0x0000FF00u>(hi, k.s8_1)), k.b_s8);
}

// Eight unsigned nibbles of `w` (nibble i = bits 4i..4i+3) -> four exact float pairs.
__device__ __forceinline__ void u4x8_to_f2(uint32_t w, const Magic &k, float2 q[4]) {
  const uint32_t h = w >> 16;
  q[0] = __fadd2_rn(f2_bits(lop3_and_or<0x000Fu>(w, k.u4_0), lop3_and_or<0x00F0u>(w, k.u4_1)), k.b_u4_01);
  q[1] = __fadd2_rn(f2_bits(lop3_and_or<0x0F00u>(w, k.u4_2), lop3_and_or<0xF000u>(w, k.u4_3)), k.b_u4_23);
  q[2] = __fadd2_rn(f2_bits(lop3_and_or<0x000Fu>(h, k.u4_0), lop3_and_or<0x00F0u>(h, k.u4_1)), k.b_u4_01);
  q[3] = __fadd2_rn(f2_bits(lop3_and_or<0x0F00u>(h, k.u4_2), lop3_and_or<0xF000u>(h, k.u4_3)), k.b_u4_23);
}

// As u4x8_to_f2 with the subtraction constants given: with b01 = b_u4_01 - (mu, mu)
// and b23 = b_u4_23 - (mu, mu) for an integer mu in [0, 15] the pairs hold q - mu, exactly.
__device__ __forceinline__ void u4x8_to_f2_shifted(uint32_t w, const Magic &k, float2 b01, float2 b23,
                                                   float2 q[4]) {
  const uint32_t h = w >> 16;
  q[0] = __fadd2_rn(f2_bits(lop3_and_or<0x000Fu>(w, k.u4_0), lop3_and_or<0x00F0u>(w, k.u4_1)), b01);
  q[1] = __fadd2_rn(f2_bits(lop3_and_or<0x0F00u>(w, k.u4_2), lop3_and_or<0xF000u>(w, k.u4_3)), b23);
  q[2] = __fadd2_rn(f2_bits(lop3_and_or<0x000Fu>(h, k.u4_0), lop3_and_or<0x00F0u>(h, k.u4_1)), b01);
  q[3] = __fadd2_rn(f2_bits(lop3_and_or<0x0F00u>(h, k.u4_2), lop3_and_or<0xF000u>(h, k.u4_3)), b23);
}

// Q6_K packed block of 32 weights (the layout qdq_q6k_pack writes): `ql` holds
// the low 4 bits -- byte b of word c has weight 8c+b in its low nibble and
// weight 8c+4+b in its high nibble -- and `qh` the high 2 bits -- byte b of word
// h has those of weights 16h+b, 16h+4+b, 16h+8+b, 16h+12+b at bits 0-1, 2-3,
// 4-5, 6-7.  Returns the exact floats q - 32 of weights (2p, 2p+1) in v[p].
__device__ __forceinline__ void q6k_block_to_f2(uint4 ql, uint2 qh, const Magic &k, float2 v[16]) {
  const uint32_t lw[4] = {ql.x, ql.y, ql.z, ql.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t H = (c >> 1) ? qh.y : qh.x;
    const uint32_t hlo = (c & 1) ? H : (H << 4);        // high bits of weights 8c..8c+3 at bits 4-5
    const uint32_t hhi = (c & 1) ? (H >> 2) : (H << 2);  // of weights 8c+4..8c+7
    const uint32_t ev = (lw[c] & 0x0F0F0F0Fu) | (hlo & 0x30303030u);         // bytes = q of 8c..8c+3
    const uint32_t od = ((lw[c] >> 4) & 0x0F0F0F0Fu) | (hhi & 0x30303030u);  // bytes = q of 8c+4..8c+7
    // each byte permuted under the exponent bits of 2^23 (k.u4_0), then 2^23 + 32 taken off: one
    // byte permute per quant and no shifts (12 % faster than masks and shifts on the ALU)
    v[4 * c + 0] = __fadd2_rn(f2_bits(__byte_perm(ev, k.u4_0, 0x7650), __byte_perm(ev, k.u4_0, 0x7651)), k.b_q6);
    v[4 * c + 1] = __fadd2_rn(f2_bits(__byte_perm(ev, k.u4_0, 0x7652), __byte_perm(ev, k.u4_0, 0x7653)), k.b_q6);
    v[4 * c + 2] = __fadd2_rn(f2_bits(__byte_perm(od, k.u4_0, 0x7650), __byte_perm(od, k.u4_0, 0x7651)), k.b_q6);
    v[4 * c + 3] = __fadd2_rn(f2_bits(__byte_perm(od, k.u4_0, 0x7652), __byte_perm(od, k.u4_0, 0x7653)), k.b_q6);
  }
}

// Bytes of one packed Q6_K row of n_in weights: the low-bit plane (n_in/2), the
// high-bit plane (n_in/4), the int8 scales (n_in/16) and the fp16 d (n_in/128),
// padded to a multiple of 16 bytes.
__host__ __device__ __forceinline__ int64_t q6k_row_bytes(int n_in) {
  return (int64_t(n_in) / 256 * 210 + 15) / 16 * 16;
}

// Q4_K header field (sc in bits 0..5, m in bits 6..11) -> (sc, m) as floats.
__device__ __forceinline__ float2 q4k_field_to_f2(uint32_t f, const Magic &k) {
  return __fadd2_rn(f2_bits(lop3_and_or<0x3Fu>(f, k.sc), lop3_and_or<0xFC0u>(f, k.m)), k.b_scm);
}

// Shift of a Q4_K sub-block with D = d*sc_j, Dm = dmin*m_j: mu is the integer in
// [0, 15] nearest Dm / D (0 when D is 0 or of the other sign), and R = Dm - D*mu
// (one rounding).  Each weight is then w = D*(q - mu) - R, where either |R| <= D/2
// (up to the quotient's approximation) or every term has the sign of w, so that
// |D*(q - mu)| <= 2|w| and |R| <= |w| for every weight of the sub-block.  A dot
// product formed as D*sum((q - mu) x) - R*sum(x) therefore has an f32 error that is
// a small multiple of sum |w||x| -- also where D*q and Dm cancel (w near 0), which
// the plain regrouping D*sum(q x) - Dm*sum(x) does not give.
__device__ __forceinline__ float q4k_mu(float2 DDm) {
  const float mu = rintf(__fdividef(DDm.y, DDm.x));
  return fminf(fmaxf(mu, 0.f), 15.f);  // a NaN quotient (0 / 0) gives 0
}

// Reduce v[0..3] (one partial per row per lane) over the warp by recursive
// halving; afterwards lane 8k holds the warp total of row k.
__device__ __forceinline__ void butterfly4_rows(float v[4], int lane) {
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = up ? v[i] : v[i + 2];
      const float keep = up ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool up = lane & 8;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 4);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace qdq

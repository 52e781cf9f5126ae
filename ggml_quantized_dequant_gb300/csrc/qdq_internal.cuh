// Internal helpers shared by the qdq kernels (not part of the public ABI).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "qdq.h"

namespace qdq {

// ---------------------------------------------------------------- host side

// Per-device facts queried once (SM count, opt-in shared memory).
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
  int smem_per_sm;
  int reserved_smem_per_block;
};

// Dynamic shared memory for a streaming GEMV CTA: at least `need`, and when
// programmatic dependent launch is on, enough that an SM holds this kernel's
// CTAs plus one CTA of the next kernel but no more -- so the next kernel's
// weight prefetch runs exactly one kernel ahead instead of flooding L2.
size_t gemv_smem_bytes(const DeviceInfo &di, size_t need);
// Returns 0 and fills `out` for the current device, or a cudaError_t.
cudaError_t device_info(DeviceInfo *out);

// Process-wide launch options (see QDQ_OPT_* in qdq.h).
int opt_pdl();
int opt_l2_prefetch();
int opt_ctas_per_sm();

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
int launch_q8_0_gemm_batch(const void *W, const float *X, float *Y, void *workspace, int n_out,
                           int n_in, int M, cudaStream_t s);

// ---------------------------------------------------------------- device side

// Programmatic dependent launch: let the next grid on the stream start early.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until every prerequisite grid has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// 128-bit read-only load that does not allocate in L1 (streamed weights).
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Packed f32x2 arithmetic (sm_100+): two lanes per instruction.
struct f2 {
  unsigned long long v;
};
__device__ __forceinline__ f2 f2_make(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r.v) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ f2 f2_from_u32(uint32_t a, uint32_t b) {
  f2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r.v) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void f2_split(f2 a, float &lo, float &hi) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

// Four signed int8 in `w` -> exact floats as two pairs (q0,q1), (q2,q3).
// A byte placed in mantissa bits [p, p+8) of a float whose exponent makes bit
// p worth 1 reads as 2^(23-p) + (byte ^ 0x80); one packed subtraction of the
// constants 2^(23-p) + 128 leaves q exactly (no conversion instructions).
__device__ __forceinline__ void s8x4_to_f2(uint32_t w, f2 &q01, f2 &q23) {
  const f2 bias = f2_make(-8388736.0f, -32896.0f);  // -(2^23 + 128), -(2^15 + 128)
  const uint32_t hi = w >> 16;
  const uint32_t a = ((w ^ 0x80u) & 0xFFu) | 0x4B000000u;      // 2^23 + (q0 + 128)
  const uint32_t b = ((w ^ 0x8000u) & 0xFF00u) | 0x47000000u;  // 2^15 + (q1 + 128)
  const uint32_t c = ((hi ^ 0x80u) & 0xFFu) | 0x4B000000u;
  const uint32_t d = ((hi ^ 0x8000u) & 0xFF00u) | 0x47000000u;
  q01 = f2_add(f2_from_u32(a, b), bias);
  q23 = f2_add(f2_from_u32(c, d), bias);
}

// Activation staging in shared memory: rows of floats cut into 128-byte lines
// of eight 16-byte chunks; chunk c of line l is stored at position c ^ (l & 7),
// so the eight lanes of one 128-bit shared-memory phase that read the same
// chunk of eight consecutive lines hit eight different bank groups.
__device__ __forceinline__ int swz_chunk(int line, int chunk) { return (line << 3) | (chunk ^ (line & 7)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace qdq

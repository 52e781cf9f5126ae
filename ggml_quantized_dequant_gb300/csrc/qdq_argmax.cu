// On-device argmax over each row of a logits matrix: the epilogue of the output
// projection, so that a decode step reads back one index and one value per token
// instead of the whole vocabulary of logits.
//
// "QTensorEngine", dispatch_output_top1_chunked (the output projection plus a
// GPU block argmax, k = 1, that saves the logits readback).  One cluster of
// eight CTAs per batch row: each CTA scans an eighth of the row (the logits come
// from L2, where the projection just wrote them) with sixteen loads in flight per
// thread, reduces it, and CTA 0 of the cluster combines the eight results through
// distributed shared memory after a cluster barrier.  The first maximal index
// wins; a NaN counts as larger than every number (the first NaN wins), the
// numpy.argmax convention.  The combination rule is associative and commutative,
// so the result does not depend on the order of the partial reductions.
#include "qdq_internal.cuh"

namespace qdq {

namespace {

constexpr int kArgmaxThreads = 1024;
constexpr int kArgmaxCluster = 8;
constexpr int kUnroll = 16;

// (value, index) that wins between two candidates
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  const bool na = a != a, nb = b != b;
  if (na != nb) return na;
  if (!na && a != b) return a > b;
  return ia < ib;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void block_reduce(float &best, int &bi, float *sv, int *si) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, best, bi)) {
      best = ov;
      bi = oi;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    best = sv[lane];
    bi = si[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, best, bi)) {
        best = ov;
        bi = oi;
      }
    }
  }
}

__global__ void __launch_bounds__(kArgmaxThreads) argmax_rows_kernel(const float *logits, int n, int *index,
                                                                     float *value) {
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
  __shared__ float s_best;
  __shared__ int s_idx;
  pdl_launch_dependents();
  pdl_wait();  // the logits come from the previous kernel
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const float *row = logits + int64_t(blockIdx.y) * n;
  const int lo = int(int64_t(rank) * n / kArgmaxCluster), hi = int(int64_t(rank + 1) * n / kArgmaxCluster);
  float best = -__int_as_float(0x7f800000);  // -inf
  int bi = n;                                 // no candidate yet
  for (int i0 = lo + threadIdx.x; i0 < hi; i0 += kUnroll * kArgmaxThreads) {
    float v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {  // all loads of the round first
      const int i = i0 + u * kArgmaxThreads;
      if (i < hi) asm volatile("ld.global.f32 %0, [%1];" : "=f"(v[u]) : "l"(row + i) : "memory");
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kArgmaxThreads;
      if (i < hi && better(v[u], i, best, bi)) {
        best = v[u];
        bi = i;
      }
    }
  }
  block_reduce(best, bi, sv, si);
  if (threadIdx.x == 0) {
    s_best = best;
    s_idx = bi;
  }
  cluster_sync();  // every CTA's result is in its shared memory
  if (rank == 0 && threadIdx.x == 0) {
    for (int r = 1; r < kArgmaxCluster; ++r) {
      uint32_t a_v, a_i;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_v) : "r"(smem_u32(&s_best)), "r"(r));
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a_i) : "r"(smem_u32(&s_idx)), "r"(r));
      float ov;
      int oi;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(ov) : "r"(a_v) : "memory");
      asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(oi) : "r"(a_i) : "memory");
      if (better(ov, oi, best, bi)) {
        best = ov;
        bi = oi;
      }
    }
    index[blockIdx.y] = bi;
    value[blockIdx.y] = best;
  }
  cluster_sync();  // no CTA leaves while CTA 0 may still read its shared memory
}

}  // namespace

int launch_argmax_rows(const float *logits, int n, int batch, int *index, float *value, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kArgmaxCluster, batch);
  cfg.blockDim = dim3(kArgmaxThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opt_pdl() ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kArgmaxCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, argmax_rows_kernel, logits, n, index, value);
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace qdq

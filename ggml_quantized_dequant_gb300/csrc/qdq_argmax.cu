// On-device argmax over each row of a logits matrix: the epilogue of the output
// projection, so that a decode step reads back one index and one value per token
// instead of the whole vocabulary of logits.
//
// "QTensorEngine", dispatch_output_top1_chunked (the output projection plus a
// GPU block argmax, k = 1, that saves the logits readback).  One CTA per batch row: the logits
// of one row (a few hundred KB) come from L2, where the projection just wrote
// them.  The first maximal index wins; a NaN counts as larger than every
// number (the first NaN wins), the numpy.argmax convention.
#include "qdq_internal.cuh"

namespace qdq {

namespace {

constexpr int kArgmaxThreads = 1024;

// (value, index) that wins between two candidates
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  const bool na = a != a, nb = b != b;
  if (na != nb) return na;
  if (!na && a != b) return a > b;
  return ia < ib;
}

__global__ void __launch_bounds__(kArgmaxThreads) argmax_rows_kernel(const float *logits, int n, int *index,
                                                                     float *value) {
  pdl_launch_dependents();
  pdl_wait();  // the logits come from the previous kernel
  const float *row = logits + int64_t(blockIdx.x) * n;
  float best = -__int_as_float(0x7f800000);  // -inf
  int bi = n;                                 // no candidate yet
  for (int i = threadIdx.x; i < n; i += kArgmaxThreads) {
    const float v = row[i];
    if (better(v, i, best, bi)) {
      best = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, best, bi)) {
      best = ov;
      bi = oi;
    }
  }
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
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
    if (lane == 0) {
      index[blockIdx.x] = bi;
      value[blockIdx.x] = best;
    }
  }
}

}  // namespace

int launch_argmax_rows(const float *logits, int n, int batch, int *index, float *value, cudaStream_t s) {
  const cudaError_t e = launch(argmax_rows_kernel, dim3(batch), dim3(kArgmaxThreads), 0, s, logits, n, index, value);
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace qdq

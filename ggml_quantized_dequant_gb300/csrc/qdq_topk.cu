// On-device top-k over each row of a logits matrix: the top-k epilogue of the
// output projection, so that a decode step reads back k (id, logit) candidates
// instead of the whole vocabulary of logits.
//
// "QTensorEngine", dispatch_output_topk_chunked: the logits stay on the GPU, a
// top-k kernel reduces them per chunk, and only the merged K candidates are read
// back.  The same here: the row is cut into chunks of 1024 logits, each chunk is
// sorted in shared memory and keeps its k best; the candidates are then merged by
// the same sort, 4096 at a time, until one chunk holds them all.
//
// Order (the k = 1 case is the argmax epilogue): a NaN comes before every number
// (the first NaN first), then larger values first, equal values (+0 and -0 are
// equal) by smaller index.  Each logit becomes a 64-bit key whose unsigned order
// is that order: the high word maps the float to an order-preserving integer
// (every NaN to the largest), the low word is the complement of the index.  A
// chunk past the row's end is padded with key 0, below every real key.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kChunk1 = 1024;  // logits per first-round chunk
constexpr int kThreads1 = 512;
constexpr int kChunk2 = 4096;  // candidate keys per merge chunk
constexpr int kThreads2 = 1024;

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

// Sorts keys[0..N) (N a power of two) into descending order; every thread of the
// CTA calls it.
template <int N, int THREADS>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t *keys) {
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < N / 2; i += THREADS) {
        const int a = 2 * i - (i & (j - 1));  // i with a zero bit inserted at bit log2(j)
        const int b = a + j;
        const bool desc = (a & k) == 0;
        const uint64_t ka = keys[a], kb = keys[b];
        if ((ka < kb) == desc) {
          keys[a] = kb;
          keys[b] = ka;
        }
      }
      __syncthreads();
    }
  }
}

// Round 1: chunk blockIdx.x of batch row blockIdx.y -> its k best keys at
// out[(row * gridDim.x + chunk) * k ...].
__global__ void __launch_bounds__(kThreads1) topk_chunk_kernel(const float *logits, int n, int k, uint64_t *out) {
  __shared__ uint64_t keys[kChunk1];
  pdl_launch_dependents();
  pdl_wait();  // the logits come from the previous kernel
  const int row = blockIdx.y;
  const int64_t base = int64_t(blockIdx.x) * kChunk1;
  const float *lr = logits + int64_t(row) * n;
  for (int i = threadIdx.x; i < kChunk1; i += kThreads1) {
    const int64_t idx = base + i;
    float v = 0.f;
    if (idx < n) asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(lr + idx) : "memory");
    keys[i] = idx < n ? topk_key(v, uint32_t(idx)) : 0ull;
  }
  __syncthreads();
  bitonic_sort_desc<kChunk1, kThreads1>(keys);
  uint64_t *o = out + (int64_t(row) * gridDim.x + blockIdx.x) * k;
  for (int j = threadIdx.x; j < k; j += kThreads1) o[j] = keys[j];
}

// Merge rounds: chunk blockIdx.x of the `count` candidate keys of batch row
// blockIdx.y -> its k best.  With one chunk left (gridDim.x == 1) and `index`
// non-NULL, writes the final (index, value) pairs instead, the value read back
// from the logits so that its bits are exactly the logit's.
__global__ void __launch_bounds__(kThreads2) topk_merge_kernel(const uint64_t *in, int count, int k, uint64_t *out,
                                                               const float *logits, int n, int *index,
                                                               float *value) {
  __shared__ uint64_t keys[kChunk2];
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.y;
  const int64_t base = int64_t(blockIdx.x) * kChunk2;
  const uint64_t *ir = in + int64_t(row) * count;
  for (int i = threadIdx.x; i < kChunk2; i += kThreads2) {
    const int64_t idx = base + i;
    uint64_t v = 0;
    if (idx < count) asm volatile("ld.global.u64 %0, [%1];" : "=l"(v) : "l"(ir + idx) : "memory");
    keys[i] = v;
  }
  __syncthreads();
  bitonic_sort_desc<kChunk2, kThreads2>(keys);
  if (index != nullptr) {
    for (int j = threadIdx.x; j < k; j += kThreads2) {
      const uint32_t id = ~uint32_t(keys[j] & 0xFFFFFFFFull);
      float v;
      asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(logits + int64_t(row) * n + id) : "memory");
      index[int64_t(row) * k + j] = int(id);
      value[int64_t(row) * k + j] = v;
    }
  } else {
    uint64_t *o = out + (int64_t(row) * gridDim.x + blockIdx.x) * k;
    for (int j = threadIdx.x; j < k; j += kThreads2) o[j] = keys[j];
  }
}

int64_t chunks1(int n) { return (int64_t(n) + kChunk1 - 1) / kChunk1; }

}  // namespace

size_t topk_workspace_bytes(int n, int batch, int k) {
  return 2 * size_t(batch) * size_t(chunks1(n)) * size_t(k) * sizeof(uint64_t);
}

int launch_topk_rows(const float *logits, int n, int batch, int k, void *workspace, int *index, float *value,
                     cudaStream_t s) {
  uint64_t *buf[2];
  buf[0] = static_cast<uint64_t *>(workspace);
  buf[1] = buf[0] + size_t(batch) * size_t(chunks1(n)) * size_t(k);
  const int nch = int(chunks1(n));
  cudaError_t e = launch(topk_chunk_kernel, dim3(nch, batch), dim3(kThreads1), 0, s, logits, n, k, buf[0]);
  if (e != cudaSuccess) return fail_cuda(e);
  int count = nch * k, cur = 0;  // candidate keys per batch row in buf[cur]
  while (count > kChunk2) {
    const int m = (count + kChunk2 - 1) / kChunk2;
    e = launch(topk_merge_kernel, dim3(m, batch), dim3(kThreads2), 0, s, static_cast<const uint64_t *>(buf[cur]),
               count, k, buf[cur ^ 1], static_cast<const float *>(nullptr), 0, static_cast<int *>(nullptr),
               static_cast<float *>(nullptr));
    if (e != cudaSuccess) return fail_cuda(e);
    count = m * k;
    cur ^= 1;
  }
  e = launch(topk_merge_kernel, dim3(1, batch), dim3(kThreads2), 0, s, static_cast<const uint64_t *>(buf[cur]), count,
             k, static_cast<uint64_t *>(nullptr), logits, n, index, value);
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace qdq

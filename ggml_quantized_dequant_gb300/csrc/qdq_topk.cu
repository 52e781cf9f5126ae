// On-device top-k over each row of a logits matrix: the top-k epilogue of the
// output projection, so that a decode step reads back k (id, logit) candidates
// instead of the whole vocabulary of logits.
//
// "QTensorEngine", dispatch_output_topk_chunked: the logits stay on the GPU, a
// top-k kernel reduces them per chunk, and only the merged K candidates are read
// back.  The same here: the row is cut into chunks of 1024 logits, each chunk keeps
// its k best (sorted); the chunks' sorted lists are then folded 32 at a time by
// bitonic merges until one list holds the row's k best.
//
// Order (the k = 1 case is the argmax epilogue): a NaN comes before every number
// (the first NaN first), then larger values first, equal values (+0 and -0 are
// equal) by smaller index.  Each logit becomes a 64-bit key whose unsigned order
// is that order: the high word maps the float to an order-preserving integer
// (every NaN to the largest), the low word is the complement of the index.  A
// chunk past the row's end is padded with key 0, below every real key.
//
// Sorting is warp-wide only: bitonic networks over 64 keys held two per lane (lane l
// has positions l and 32 + l; strides below 32 are shuffles, the 32 stride a swap
// between a lane's two registers), and sorted 64-key lists are combined by bitonic
// merges, never by a block-wide sort.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kChunk1 = 1024;  // logits per first-round chunk

// First pass: chunk blockIdx.x of batch row blockIdx.y -> its k best keys, sorted best
// first, at out[(row * gridDim.x + chunk) * k ...].  Each of the 16 warps sorts its 64
// logits (a warp-wide bitonic sort), and the warps' sorted lists are folded pairwise
// through shared memory as in the merge rounds.
__global__ void __launch_bounds__(kChunk1 / 2) topk_chunk_kernel(const float *logits, int n, int k, uint64_t *out) {
  __shared__ uint64_t sl[kChunk1 / 128][64];
  pdl_launch_dependents();
  pdl_wait();  // the logits come from the previous kernel
  const int row = blockIdx.y;
  const int64_t base = int64_t(blockIdx.x) * kChunk1;
  const float *lr = logits + int64_t(row) * n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ia = base + 64 * warp + lane, ib = ia + 32;
  float va = 0.f, vb = 0.f;
  if (ia < n) asm volatile("ld.global.f32 %0, [%1];" : "=f"(va) : "l"(lr + ia) : "memory");
  if (ib < n) asm volatile("ld.global.f32 %0, [%1];" : "=f"(vb) : "l"(lr + ib) : "memory");
  uint64_t a = ia < n ? topk_key(va, uint32_t(ia)) : 0ull;
  uint64_t b = ib < n ? topk_key(vb, uint32_t(ib)) : 0ull;
  warp_sort64_desc(a, b, lane);
  for (int half = kChunk1 / 128; half >= 1; half >>= 1) {
    if (warp >= half && warp < 2 * half) {
      sl[warp - half][lane] = a;
      sl[warp - half][lane + 32] = b;
    }
    __syncthreads();
    if (warp < half) warp_top64_merge(a, b, sl[warp][lane], sl[warp][lane + 32], lane);
    __syncthreads();
  }
  if (warp == 0) {  // the k best are positions 0..k-1 of warp 0's list
    uint64_t *o = out + (int64_t(row) * gridDim.x + blockIdx.x) * k;
    if (lane < k) o[lane] = a;
    if (lane + 32 < k) o[lane + 32] = b;
  }
}

// Merge rounds: the candidate lists (k keys each, sorted best first: the chunks' or the
// projection CTAs' k best) of batch row blockIdx.y hold the row's k best, which are the
// k best of their union.  They are folded with bitonic merges of sorted lists instead of
// being sorted again (the element-wise maximum of one sorted list and the other reversed
// is bitonic and holds the 64 largest of the two; one bitonic merge sorts it).  A round:
// CTA b takes lists 32b .. 32b + 31, one per warp, and folds them pairwise through shared
// memory into one sorted list of k keys; rounds repeat until one CTA per row is left,
// which writes the (index, value) pairs, the value read back from the logits so that
// its bits are exactly the logit's.
__global__ void __launch_bounds__(1024) topk_fold_kernel(const uint64_t *in, int nlists, int k, uint64_t *out,
                                                         const float *logits, int n, int *index, float *value) {
  __shared__ uint64_t sl[16][64];
  pdl_launch_dependents();
  pdl_wait();  // the lists come from the previous kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.y;
  const int c = blockIdx.x * 32 + warp;  // this warp's list: positions lane, lane + 32 (key 0 past k)
  uint64_t ta = 0ull, tb = 0ull;
  if (c < nlists) {
    const uint64_t *p = in + (int64_t(row) * nlists + c) * k;
    if (lane < k) asm volatile("ld.global.u64 %0, [%1];" : "=l"(ta) : "l"(p + lane) : "memory");
    if (lane + 32 < k) asm volatile("ld.global.u64 %0, [%1];" : "=l"(tb) : "l"(p + lane + 32) : "memory");
  }
  for (int half = 16; half >= 1; half >>= 1) {
    if (warp >= half && warp < 2 * half) {
      sl[warp - half][lane] = ta;
      sl[warp - half][lane + 32] = tb;
    }
    __syncthreads();
    if (warp < half) warp_top64_merge(ta, tb, sl[warp][lane], sl[warp][lane + 32], lane);
    __syncthreads();
  }
  if (warp != 0) return;
  if (index == nullptr) {
    uint64_t *o = out + (int64_t(row) * gridDim.x + blockIdx.x) * k;
    if (lane < k) o[lane] = ta;
    if (lane + 32 < k) o[lane + 32] = tb;
    return;
  }
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    if (j >= k) break;
    const uint64_t key = h ? tb : ta;
    const uint32_t id = ~uint32_t(key & 0xFFFFFFFFull);
    float v = __int_as_float(0x7fffffff);
    if (QDQ_GUARD(id < uint32_t(n), QDQ_CHECK_ROW))
      asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(logits + int64_t(row) * n + id) : "memory");
    index[int64_t(row) * k + j] = int(id);
    value[int64_t(row) * k + j] = v;
  }
}

int64_t chunks1(int n) { return (int64_t(n) + kChunk1 - 1) / kChunk1; }

}  // namespace

QDQ_CHECK_READER(read_checks_topk)

size_t topk_workspace_bytes(int n, int batch, int k) {
  // the chunked path: two rounds of ceil(n / 1024) * k keys per row; the batch-1 output
  // projection: one key list per CTA of k keys, and the merge round after it
  const size_t chunked = 2 * size_t(batch) * size_t(chunks1(n)) * size_t(k);
  const size_t fused = 2 * size_t(gemv_dl_max_ctas()) * size_t(k);
  return (chunked > fused ? chunked : fused) * sizeof(uint64_t);
}

namespace {
// Fold rounds over `count` candidate keys (count / k lists) per batch row in buf0, buf1
// the other half of the ping-pong, down to one CTA per row, which writes the pairs.
int merge_rounds(int count, int batch, int k, uint64_t *buf0, uint64_t *buf1, const float *logits, int n, int *index,
                 float *value, cudaStream_t s) {
  uint64_t *buf[2] = {buf0, buf1};
  int cur = 0, nlists = count / k;
  cudaError_t e = cudaSuccess;
  while (nlists > 32) {
    const int m = (nlists + 31) / 32;
    e = launch(topk_fold_kernel, dim3(m, batch), dim3(1024), 0, s, buf[cur], nlists, k, buf[cur ^ 1],
               static_cast<const float *>(nullptr), 0, static_cast<int *>(nullptr), static_cast<float *>(nullptr));
    if (e != cudaSuccess) return fail_cuda(e);
    nlists = m;
    cur ^= 1;
  }
  e = launch(topk_fold_kernel, dim3(1, batch), dim3(1024), 0, s, buf[cur], nlists, k, static_cast<uint64_t *>(nullptr),
             logits, n, index, value);
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}
}  // namespace

int launch_topk_rows(const float *logits, int n, int batch, int k, void *workspace, int *index, float *value,
                     cudaStream_t s) {
  uint64_t *buf0 = static_cast<uint64_t *>(workspace);
  uint64_t *buf1 = buf0 + size_t(batch) * size_t(chunks1(n)) * size_t(k);
  const int nch = int(chunks1(n));
  const cudaError_t e = launch(topk_chunk_kernel, dim3(nch, batch), dim3(kChunk1 / 2), 0, s, logits, n, k, buf0);
  if (e != cudaSuccess) return fail_cuda(e);
  return merge_rounds(nch * k, batch, k, buf0, buf1, logits, n, index, value, s);
}

int launch_topk_merge(int count, int k, void *workspace, const float *logits, int n, int *index, float *value,
                      cudaStream_t s) {
  uint64_t *buf0 = static_cast<uint64_t *>(workspace);
  return merge_rounds(count, 1, k, buf0, buf0 + count, logits, n, index, value, s);
}

}  // namespace qdq

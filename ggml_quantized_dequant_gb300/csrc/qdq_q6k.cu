// GGML Q6_K on the device: the one-time repack, the bit-exact dequantisation,
// the embedding-row lookup and the batch 2..8 GEMV (batch 1 runs in
// qdq_gemv_xs.cu).
//
// "QTensorEngine": the embedding pipeline ("GPU-side Q6_K embedding dequant +
// matmul (zero CPU dequant)", dispatch_quantized_token_embedding) and
// dispatch_gemm_into ("Quantized GEMM into caller out ... (Q6_K)").
//
// GGML Q6_K superblock, 210 bytes for 256 weights: ql[128] (low 4 bits of each
// quant) @0, qh[64] (high 2 bits) @128, sixteen int8 scales @192, fp16 d @208.
// Weight e (0..255) belongs to the 16-weight sub-block e/16 and equals
// d * scale[e/16] * (q_e - 32), q_e in 0..63.  In GGML order the superblock is
// two halves h of 128 weights; weight 128h + 32t + l (t = 0..3, l = 0..31)
// takes its low 4 bits from the low (t < 2) or high (t >= 2) nibble of
// ql[64h + 32(t & 1) + l] and its high 2 bits from bits 2t..2t+1 of qh[32h + l].
//
// Packed row (the kernels' layout): [ low-bit plane n_in/2 | high-bit plane
// n_in/4 | scales n_in/16 | d n_in/128 | zero padding to 16 bytes ].  Block b of
// 32 weights owns bytes 16b.. of the low plane, 8b.. of the high plane, 2b.. of
// the scales and (b/8)*2.. of d; inside it the bits are placed as
// q6k_block_to_f2 reads them, so one 16-byte and one 8-byte load carry a lane's
// 32 quants.  Only the padding adds bytes (none when n_in % 2048 == 0).
//
// Exactness: d has at most 11 significant bits, |scale| <= 128, |q - 32| <= 32,
// so d * scale and (d * scale) * (q - 32) are exact in f32.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t items, int threads) {
  int64_t g = (items + threads - 1) / threads;
  if (g > 65535LL * 16) g = 65535LL * 16;
  return int(g < 1 ? 1 : g);
}

// One thread per GGML superblock.
__global__ void q6k_pack_kernel(const uint8_t *__restrict__ g, uint8_t *__restrict__ packed, int64_t n_super,
                                int nsb_row, int n_in, int64_t row_bytes) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_super;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint8_t *src = g + i * 210;
    const int64_t row = i / nsb_row;
    const int sb = int(i - row * nsb_row);
    uint8_t *dst_row = packed + row * row_bytes;
    uint8_t q[256];
    for (int h = 0; h < 2; ++h)
      for (int t = 0; t < 4; ++t)
        for (int l = 0; l < 32; ++l) {
          const uint32_t b = src[64 * h + 32 * (t & 1) + l];
          const uint32_t lo = t < 2 ? (b & 0x0Fu) : (b >> 4);
          const uint32_t hi = (uint32_t(src[128 + 32 * h + l]) >> (2 * t)) & 3u;
          q[128 * h + 32 * t + l] = uint8_t(lo | (hi << 4));
        }
    for (int bl = 0; bl < 8; ++bl) {  // the superblock's eight 32-weight blocks
      const uint8_t *qb = q + 32 * bl;
      const int blk = 8 * sb + bl;
      uint8_t *lo = dst_row + 16 * blk;
      uint8_t *hi = dst_row + n_in / 2 + 8 * blk;
      for (int c = 0; c < 4; ++c)
        for (int b = 0; b < 4; ++b) lo[4 * c + b] = uint8_t((qb[8 * c + b] & 0x0F) | ((qb[8 * c + 4 + b] & 0x0F) << 4));
      for (int h = 0; h < 2; ++h)
        for (int b = 0; b < 4; ++b)
          hi[4 * h + b] = uint8_t((qb[16 * h + b] >> 4) | ((qb[16 * h + 4 + b] >> 4) << 2) |
                                  ((qb[16 * h + 8 + b] >> 4) << 4) | ((qb[16 * h + 12 + b] >> 4) << 6));
    }
    uint8_t *sc = dst_row + n_in / 2 + n_in / 4 + 16 * sb;
    for (int j = 0; j < 16; ++j) sc[j] = src[192 + j];
    uint8_t *d = dst_row + n_in / 2 + n_in / 4 + n_in / 16 + 2 * sb;
    d[0] = src[208];
    d[1] = src[209];
    if (sb == nsb_row - 1)  // the row's padding
      for (int64_t p = int64_t(n_in) / 256 * 210; p < row_bytes; ++p) dst_row[p] = 0;
  }
}

// Block `blk` of a packed Q6_K row: quants (as q6k_block_to_f2 wants them), the two
// sub-block scales times d (exact), for weights 0..15 and 16..31 of the block.
struct Q6Block {
  uint4 ql;
  uint2 qh;
  float ds0, ds1;
};
__device__ __forceinline__ Q6Block q6k_load_block(const uint8_t *row, int n_in, int blk) {
  Q6Block b;
  b.ql = ldg_stream(row + 16 * blk);
  b.qh = *reinterpret_cast<const uint2 *>(row + n_in / 2 + 8 * blk);
  const uint16_t s = *reinterpret_cast<const uint16_t *>(row + n_in / 2 + n_in / 4 + 2 * blk);
  const float d = __half2float(*reinterpret_cast<const __half *>(row + n_in / 2 + n_in / 4 + n_in / 16 + 2 * (blk / 8)));
  b.ds0 = __fmul_rn(d, float(int8_t(s & 0xFF)));
  b.ds1 = __fmul_rn(d, float(int8_t(s >> 8)));
  return b;
}

// One thread per 32-weight block: w = (d * scale) * (q - 32), exact.
__global__ void q6k_dequant_kernel(const uint8_t *__restrict__ W, float *__restrict__ out, int64_t n_blocks,
                                   int nblk_row, int n_in, int64_t row_bytes, const Magic mg_param) {
  const Magic mg = lane_magic(mg_param);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_blocks;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = i / nblk_row;
    const int blk = int(i - row * nblk_row);
    const Q6Block b = q6k_load_block(W + row * row_bytes, n_in, blk);
    float2 v[16];
    q6k_block_to_f2(b.ql, b.qh, mg, v);
    float *o = out + row * n_in + 32 * blk;
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const float ds = p < 8 ? b.ds0 : b.ds1;
      o[2 * p] = __fmul_rn(ds, v[p].x);
      o[2 * p + 1] = __fmul_rn(ds, v[p].y);
    }
  }
}

// Embedding lookup: out[i, :] = dequantised row ids[i] (a NaN row for an id
// outside [0, n_rows)).  One warp per 32-weight block column strip.
__global__ void q6k_get_rows_kernel(const uint8_t *__restrict__ W, const int *ids, float *__restrict__ out,
                                    int n_ids, int n_rows, int n_in, int64_t row_bytes, const Magic mg_param) {
  const Magic mg = lane_magic(mg_param);
  pdl_launch_dependents();
  pdl_wait();  // the ids may come from the previous kernel
  const int nblk = n_in / 32;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < int64_t(n_ids) * nblk;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int r = int(i / nblk), blk = int(i - int64_t(r) * nblk);
    if (!QDQ_GUARD(r < n_ids, QDQ_CHECK_OUT)) continue;
    const int id = ld_s32_after_wait(ids + r);
    float *o = out + int64_t(r) * n_in + 32 * blk;
    if (id < 0 || id >= n_rows) {
#pragma unroll
      for (int k = 0; k < 32; ++k) o[k] = __int_as_float(0x7fffffff);
      continue;
    }
    const Q6Block b = q6k_load_block(W + int64_t(id) * row_bytes, n_in, blk);
    float2 v[16];
    q6k_block_to_f2(b.ql, b.qh, mg, v);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const float ds = p < 8 ? b.ds0 : b.ds1;
      o[2 * p] = __fmul_rn(ds, v[p].x);
      o[2 * p + 1] = __fmul_rn(ds, v[p].y);
    }
  }
}

// Batch 2..8 GEMV: one CTA per SM over a contiguous row range, x for NB batch
// rows staged in shared memory, one warp per row at a time, lane l taking the
// row's 32-weight blocks l, l + 32, ...; per block the two sub-block sums are
// scaled by d * scale once (error relative to sum |w||x|, no offset term).
template <int NB>
__global__ void __launch_bounds__(kThreads) q6k_gemv_kernel(const uint8_t *__restrict__ W, const float *__restrict__ x,
                                                            float *__restrict__ y, int n_out, int n_in,
                                                            int64_t row_bytes, const Magic mg_param) {
  extern __shared__ float4 smem4[];
  float *xs = reinterpret_cast<float *>(smem4);
  const Magic mg = lane_magic(mg_param);
  const int r_begin = int(int64_t(blockIdx.x) * n_out / gridDim.x);
  const int r_end = int(int64_t(blockIdx.x + 1) * n_out / gridDim.x);
  pdl_launch_dependents();
  pdl_wait();
  for (int i = threadIdx.x; i < NB * n_in / 4; i += kThreads)
    reinterpret_cast<float4 *>(xs)[i] = ld_after_wait(reinterpret_cast<const float4 *>(x) + i);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = n_in / 32;
  for (int r = r_begin + warp; r < r_end; r += kThreads / 32) {
    const uint8_t *row = W + int64_t(r) * row_bytes;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    for (int blk = lane; blk < nblk; blk += 32) {
      const Q6Block qb = q6k_load_block(row, n_in, blk);
      float2 v[16];
      q6k_block_to_f2(qb.ql, qb.qh, mg, v);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float4 *xb = reinterpret_cast<const float4 *>(xs + int64_t(b) * n_in + 32 * blk);
        float2 s0 = f2(0.f, 0.f), s1 = f2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const float4 xv = xb[p];
          float2 &s = p < 4 ? s0 : s1;
          s = __ffma2_rn(v[2 * p], f2(xv.x, xv.y), s);
          s = __ffma2_rn(v[2 * p + 1], f2(xv.z, xv.w), s);
        }
        acc[b] = fmaf(qb.ds1, s1.x + s1.y, fmaf(qb.ds0, s0.x + s0.y, acc[b]));
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float v = warp_sum(acc[b]);
      if (lane == 0) y[int64_t(b) * n_out + r] = v;
    }
  }
}

template <int NB>
int launch_nb(const uint8_t *W, const float *x, float *y, int n_out, int n_in, cudaStream_t s, const DeviceInfo &di) {
  const size_t smem = size_t(NB) * n_in * sizeof(float);
  auto kern = q6k_gemv_kernel<NB>;
  if (smem > 48 * 1024) {
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const int grid = gemv_grid(di, n_out, 1);
  const cudaError_t e = launch(kern, dim3(grid), dim3(kThreads), smem, s, W, x, y, n_out, n_in,
                               q6k_row_bytes(n_in), make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace

QDQ_CHECK_READER(read_checks_q6k)

int launch_q6k_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t s) {
  const int64_t nsb = int64_t(n_out) * (n_in / 256);
  q6k_pack_kernel<<<grid_for(nsb, 128), 128, 0, s>>>(static_cast<const uint8_t *>(ggml),
                                                      static_cast<uint8_t *>(packed), nsb, n_in / 256, n_in,
                                                      q6k_row_bytes(n_in));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

int launch_q6k_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t s) {
  const int64_t n = int64_t(n_out) * (n_in / 32);
  q6k_dequant_kernel<<<grid_for(n, kThreads), kThreads, 0, s>>>(static_cast<const uint8_t *>(W), out, n, n_in / 32,
                                                                 n_in, q6k_row_bytes(n_in), make_magic());
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

int launch_q6k_get_rows(const void *W, const int *ids, float *out, int n_ids, int n_rows, int n_in, cudaStream_t s) {
  const int64_t n = int64_t(n_ids) * (n_in / 32);
  const cudaError_t e = launch(q6k_get_rows_kernel, dim3(grid_for(n, kThreads)), dim3(kThreads), 0, s,
                               static_cast<const uint8_t *>(W), ids, out, n_ids, n_rows, n_in, q6k_row_bytes(n_in),
                               make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

int launch_q6k_gemv(const void *Wv, const float *x, float *y, int n_out, int n_in, int batch, cudaStream_t s) {
  if (gemv_xs_supported(n_in, batch, 2)) return launch_gemv_xs(2, 0, Wv, nullptr, x, nullptr, y, n_out, n_in, s);
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  const uint8_t *W = static_cast<const uint8_t *>(Wv);
  // batch rows per launch: as many as the activations of fit in shared memory
  int per = int(int64_t(di.max_smem_optin) / (int64_t(n_in) * 4));
  if (per < 1) return QDQ_ERR_UNSUPPORTED;
  if (per > QDQ_MAX_GEMV_BATCH) per = QDQ_MAX_GEMV_BATCH;
  for (int b0 = 0; b0 < batch; b0 += per) {
    const int nb = (batch - b0) < per ? (batch - b0) : per;
    const float *xb = x + int64_t(b0) * n_in;
    float *yb = y + int64_t(b0) * n_out;
    int rc;
    switch (nb) {
      case 1: rc = launch_nb<1>(W, xb, yb, n_out, n_in, s, di); break;
      case 2: rc = launch_nb<2>(W, xb, yb, n_out, n_in, s, di); break;
      case 3: rc = launch_nb<3>(W, xb, yb, n_out, n_in, s, di); break;
      case 4: rc = launch_nb<4>(W, xb, yb, n_out, n_in, s, di); break;
      case 5: rc = launch_nb<5>(W, xb, yb, n_out, n_in, s, di); break;
      case 6: rc = launch_nb<6>(W, xb, yb, n_out, n_in, s, di); break;
      case 7: rc = launch_nb<7>(W, xb, yb, n_out, n_in, s, di); break;
      default: rc = launch_nb<8>(W, xb, yb, n_out, n_in, s, di); break;
    }
    if (rc != QDQ_OK) return rc;
  }
  return QDQ_OK;
}

}  // namespace qdq

// Q8_0 dequant-GEMV: y[b, r] = sum_blk d[r, blk] * sum_{k<32} q[r, blk, k] * x[b, 32 blk + k].
//
// "Module cuda_lane", Functions: try_q8_0_cuda_gemv (native Q8_0 GEMV) and
// q8_0_gemv_oracle_into (decode a row-major GGML Q8_0 matrix, multiply by x).
//
// Design (HBM-bound streaming kernel):
//  * grid = SMs x CTAs-per-SM; CTA i owns the contiguous row range
//    [i*n_out/G, (i+1)*n_out/G), i.e. one contiguous slice of the q plane and
//    of the d plane.  Its first thread bulk-prefetches both slices into L2
//    before waiting on the previous kernel (programmatic dependent launch),
//    so weight streaming overlaps the previous kernel's tail.
//  * x (batch x n_in f32) is staged once per CTA in XOR-swizzled shared
//    memory; 16-byte reads by consecutive lanes are bank-conflict free.
//  * a warp task is R consecutive rows; lane l reads 16-byte chunks l, l+32,
//    ... of each row with non-allocating 128-bit loads and the matching fp16
//    scale (shared by two lanes).
//  * int8 -> f32 exactly, without conversion instructions: a byte b placed in
//    mantissa bits [p, p+8) of a float whose exponent makes bit p worth 1
//    gives 2^(23-p) + (b ^ 0x80); subtracting the constant 2^(23-p) + 128
//    recovers q exactly.  Products and partial sums use packed f32x2 FMA.
//  * per 16-weight chunk the partial sum s = sum q*x is scaled by d once:
//    d is common to the chunk and positive or negative alike, so the error is
//    bounded by that of sum |q||x| times |d| = sum |w||x|.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 2;  // rows per warp task

template <int NB>
__global__ void __launch_bounds__(kThreads) q8_0_gemv_kernel(const uint8_t *__restrict__ W,
                                                             const float *__restrict__ x,
                                                             float *__restrict__ y, int n_out, int n_in,
                                                             int l2_prefetch) {
  extern __shared__ float4 xs[];
  const int64_t q_bytes = int64_t(n_out) * n_in;
  const int64_t d_row_bytes = n_in / 16;  // n_in/32 fp16 scales
  const int r_begin = int(int64_t(blockIdx.x) * n_out / gridDim.x);
  const int r_end = int(int64_t(blockIdx.x + 1) * n_out / gridDim.x);

  if (l2_prefetch && threadIdx.x == 0) {
    prefetch_range_l2(W, q_bytes, int64_t(r_begin) * n_in, int64_t(r_end) * n_in);
    prefetch_range_l2(W + q_bytes, int64_t(n_out) * d_row_bytes, int64_t(r_begin) * d_row_bytes,
                      int64_t(r_end) * d_row_bytes);
  }
  pdl_launch_dependents();
  pdl_wait();

  const int lines_per_row = n_in >> 5;
  {
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const int n4 = NB * lines_per_row * 8;
    for (int i = threadIdx.x; i < n4; i += kThreads) xs[swz_chunk(i >> 3, i & 7)] = x4[i];
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = n_in >> 4;
  const int ntask = (r_end - r_begin + kRows - 1) / kRows;
  const __half *dplane = reinterpret_cast<const __half *>(W + q_bytes);

  for (int task = warp; task < ntask; task += kWarps) {
    const int r0 = r_begin + task * kRows;
    const uint8_t *qrow[kRows];
    const __half *drow[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int row = min(r0 + r, r_end - 1);  // a missing last row re-reads the previous one; result dropped
      qrow[r] = W + int64_t(row) * n_in;
      drow[r] = dplane + int64_t(row) * (n_in >> 5);
    }
    f2 acc[kRows][NB];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = f2_make(0.f, 0.f);

    int ch = lane;
    uint4 qv[kRows];
    float dv[kRows];
    if (ch < nch) {
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        qv[r] = ldg_stream(qrow[r] + int64_t(ch) * 16);
        dv[r] = __half2float(__ldg(drow[r] + (ch >> 1)));
      }
    }
    while (ch < nch) {
      // issue the next chunk's loads before using this one
      const int nx = ch + 32;
      uint4 qn[kRows];
      float dn[kRows];
      if (nx < nch) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          qn[r] = ldg_stream(qrow[r] + int64_t(nx) * 16);
          dn[r] = __half2float(__ldg(drow[r] + (nx >> 1)));
        }
      }
      f2 qf[kRows][8];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        s8x4_to_f2(qv[r].x, qf[r][0], qf[r][1]);
        s8x4_to_f2(qv[r].y, qf[r][2], qf[r][3]);
        s8x4_to_f2(qv[r].z, qf[r][4], qf[r][5]);
        s8x4_to_f2(qv[r].w, qf[r][6], qf[r][7]);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int line = b * lines_per_row + (ch >> 1);
        const int c0 = (ch & 1) << 2;
        f2 s[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) s[r] = f2_make(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 xv = xs[swz_chunk(line, c0 + i)];
          const f2 x01 = f2_make(xv.x, xv.y), x23 = f2_make(xv.z, xv.w);
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            s[r] = f2_fma(qf[r][2 * i], x01, s[r]);
            s[r] = f2_fma(qf[r][2 * i + 1], x23, s[r]);
          }
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) acc[r][b] = f2_fma(f2_make(dv[r], dv[r]), s[r], acc[r][b]);
      }
      if (nx < nch) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          qv[r] = qn[r];
          dv[r] = dn[r];
        }
      }
      ch = nx;
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float lo, hi;
        f2_split(acc[r][b], lo, hi);
        const float v = warp_sum(lo + hi);
        if (lane == 0 && r0 + r < r_end) y[int64_t(b) * n_out + r0 + r] = v;
      }
    }
  }
}

template <int NB>
int launch_nb(const uint8_t *W, const float *x, float *y, int n_out, int n_in, cudaStream_t s,
              const DeviceInfo &di) {
  const size_t smem = gemv_smem_bytes(di, size_t(NB) * n_in * sizeof(float));
  auto kern = q8_0_gemv_kernel<NB>;
  if (smem > 48 * 1024) {
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  int grid = di.sm_count * opt_ctas_per_sm();
  const int max_grid = (n_out + kRows - 1) / kRows;
  if (grid > max_grid) grid = max_grid;
  const cudaError_t e = launch(kern, dim3(grid), dim3(kThreads), smem, s, W, x, y, n_out, n_in,
                               opt_l2_prefetch());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace

int launch_q8_0_gemv(const void *Wv, const float *x, float *y, int n_out, int n_in, int batch,
                     cudaStream_t s) {
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  const uint8_t *W = static_cast<const uint8_t *>(Wv);
  // batch groups: each group's activations must fit in shared memory
  const int budget = di.max_smem_optin < 200 * 1024 ? di.max_smem_optin : 200 * 1024;
  int per = budget / (n_in * int(sizeof(float)));
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

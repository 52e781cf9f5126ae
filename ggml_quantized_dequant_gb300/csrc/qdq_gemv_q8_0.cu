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
//  * x (batch x n_in f32) is staged once per CTA in shared memory with one
//    16-byte pad per 16 floats, so 16-byte reads by consecutive lanes are
//    bank-conflict free.
//  * a warp task is 2 consecutive rows; lane l reads 16-byte chunks l, l+32,
//    ... of both rows with non-allocating 128-bit loads and the matching fp16
//    scale (shared by two lanes).  A CTA's tasks x lane-iterations ("units")
//    are split into equal contiguous ranges, one per warp, and each lane keeps
//    P units of loads in flight in a register ring (about 8 KB per warp), so
//    the kernel is not latency-bound.  Rows straddling two warps' ranges get
//    two shared-memory adds, which commute, so results stay deterministic.
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

// x staging: chunk c (16 floats) of batch row b at float offset (b * nch + c) * kXStride;
// the 80-byte stride puts the 16-byte reads of eight consecutive chunks in
// eight different bank groups (5c mod 8 is a permutation), with no index math.
constexpr int kXStride = 20;

template <int NB, int P>
__global__ void __launch_bounds__(kThreads) q8_0_gemv_kernel(const uint8_t *__restrict__ W,
                                                             const float *__restrict__ x,
                                                             float *__restrict__ y, int n_out, int n_in,
                                                             int l2_prefetch, const Magic mg_param) {
  extern __shared__ float4 smem4[];
  const Magic mg = lane_magic(mg_param);
  const int64_t q_bytes = int64_t(n_out) * n_in;
  const int64_t d_row_bytes = n_in / 16;  // n_in/32 fp16 scales
  const int r_begin = int(int64_t(blockIdx.x) * n_out / gridDim.x);
  const int r_end = int(int64_t(blockIdx.x + 1) * n_out / gridDim.x);
  const int nrows = r_end - r_begin;

  if (l2_prefetch && threadIdx.x == 0) {
    prefetch_range_l2(W, q_bytes, int64_t(r_begin) * n_in, int64_t(r_end) * n_in);
    prefetch_range_l2(W + q_bytes, int64_t(n_out) * d_row_bytes, int64_t(r_begin) * d_row_bytes,
                      int64_t(r_end) * d_row_bytes);
  }
  pdl_launch_dependents();

  const int nch = n_in >> 4;  // 16-weight chunks per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int itpt = (nch + 31) >> 5;  // lane iterations per row pair ("units" per task)
  const int ntask = (nrows + kRows - 1) / kRows;
  const int total = ntask * itpt;
  // contiguous, balanced unit ranges per warp; a range is never shorter than a task,
  // so at most two warps contribute to any row (their two shared-memory adds commute)
  int per = (total + kWarps - 1) / kWarps;
  if (per < itpt) per = itpt;
  const int k0 = min(warp * per, total);
  const int k1 = min(k0 + per, total);
  const uint16_t *dplane = reinterpret_cast<const uint16_t *>(W + q_bytes);
  const int dpr = n_in >> 5;  // scales per row

  // load cursor (task lt, iteration li) with per-task row pointers; the weight
  // ring is filled before waiting on the previous kernel, which only x depends on
  int lt = k0 / itpt, li = k0 - lt * itpt;
  const uint8_t *lq[kRows];
  const uint16_t *ld[kRows];
  auto set_rows = [&]() {
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int row = r_begin + min(kRows * lt + r, nrows - 1);  // a missing last row repeats; dropped later
      lq[r] = W + int64_t(row) * n_in + lane * 16;
      ld[r] = dplane + int64_t(row) * dpr + (lane >> 1);
    }
  };
  uint4 qb[P][kRows];
  uint16_t db[P][kRows];  // raw fp16 bits, converted where used
  auto load = [&](int slot) {
    if (lane + 32 * li < nch) {
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        qb[slot][r] = ldg_stream(lq[r] + li * 512);
        db[slot][r] = __ldg(ld[r] + li * 16);
      }
    }
    if (++li == itpt) {
      li = 0;
      ++lt;
      set_rows();
    }
  };
  if (k0 < k1) {
    set_rows();
#pragma unroll
    for (int p = 0; p < P; ++p)
      if (k0 + p < k1) load(p);
  }

  pdl_wait();
  float *xs = reinterpret_cast<float *>(smem4);
  float *ysm = xs + size_t(NB) * nch * kXStride;  // nrows x NB partial sums
  {
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    for (int i = threadIdx.x; i < NB * nch * 4; i += kThreads)
      *reinterpret_cast<float4 *>(xs + (i >> 2) * kXStride + (i & 3) * 4) = x4[i];
    for (int i = threadIdx.x; i < nrows * NB; i += kThreads) ysm[i] = 0.f;
  }
  __syncthreads();

  if (k0 < k1) {
    int ct = k0 / itpt, ci = k0 - ct * itpt;  // compute cursor
    float2 acc[kRows][NB];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = f2(0.f, 0.f);

    for (int kb = k0; kb < k1; kb += P) {
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const int k = kb + p;
        if (k < k1) {
          const int ch = lane + 32 * ci;
          if (ch < nch) {
            float2 qf[kRows][8];
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
              s8x4_to_f2(qb[p][r].x, mg, qf[r][0], qf[r][1]);
              s8x4_to_f2(qb[p][r].y, mg, qf[r][2], qf[r][3]);
              s8x4_to_f2(qb[p][r].z, mg, qf[r][4], qf[r][5]);
              s8x4_to_f2(qb[p][r].w, mg, qf[r][6], qf[r][7]);
            }
            float dv[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r) dv[r] = __half2float(__ushort_as_half(db[p][r]));
            const float *xc = xs + ch * kXStride;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              float2 s0[kRows], s1[kRows];  // two independent chains per row
#pragma unroll
              for (int r = 0; r < kRows; ++r) s0[r] = s1[r] = f2(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 xv = *reinterpret_cast<const float4 *>(xc + b * nch * kXStride + 4 * i);
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                  s0[r] = __ffma2_rn(qf[r][2 * i], f2(xv.x, xv.y), s0[r]);
                  s1[r] = __ffma2_rn(qf[r][2 * i + 1], f2(xv.z, xv.w), s1[r]);
                }
              }
#pragma unroll
              for (int r = 0; r < kRows; ++r)
                acc[r][b] = __ffma2_rn(f2(dv[r], dv[r]), __fadd2_rn(s0[r], s1[r]), acc[r][b]);
            }
          }
          if (k + P < k1) load(p);
          if (++ci == itpt || k + 1 == k1) {  // this warp's share of task ct is complete
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                const float v = warp_sum(acc[r][b].x + acc[r][b].y);
                const int row = kRows * ct + r;
                if (lane == 0 && row < nrows) atomicAdd(&ysm[row * NB + b], v);
                acc[r][b] = f2(0.f, 0.f);
              }
            }
            if (ci == itpt) {
              ci = 0;
              ++ct;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nrows * NB; i += kThreads) {
    const int row = i / NB, b = i - row * NB;
    y[int64_t(b) * n_out + r_begin + row] = ysm[i];
  }
}

template <int NB>
int launch_nb(const uint8_t *W, const float *x, float *y, int n_out, int n_in, cudaStream_t s,
              const DeviceInfo &di) {
  const int grid = gemv_grid(di, n_out, kRows);
  const int max_rows = (n_out + grid - 1) / grid;
  const size_t smem = gemv_smem_bytes(
      di, size_t(NB) * (n_in >> 4) * kXStride * sizeof(float) + size_t(max_rows) * NB * sizeof(float));
  constexpr int P = NB <= 2 ? 8 : 4;  // loads in flight per lane
  auto kern = q8_0_gemv_kernel<NB, P>;
  if (smem > 48 * 1024) {
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const cudaError_t e = launch(kern, dim3(grid), dim3(kThreads), smem, s, W, x, y, n_out, n_in,
                               opt_l2_prefetch() == 1, make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace

int launch_q8_0_gemv(const void *Wv, const float *x, float *y, int n_out, int n_in, int batch,
                     cudaStream_t s) {
  if (gemv_xs_supported(n_in, batch, 0)) return launch_gemv_xs(0, 0, Wv, nullptr, x, nullptr, y, n_out, n_in, s);
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  const uint8_t *W = static_cast<const uint8_t *>(Wv);
  // batch groups: each group's activations must fit in shared memory
  const int budget = di.max_smem_optin < 200 * 1024 ? di.max_smem_optin : 200 * 1024;
  const int grid = gemv_grid(di, n_out, kRows);
  const int max_rows = (n_out + grid - 1) / grid;
  int per = budget / (((n_in >> 4) * kXStride + max_rows) * int(sizeof(float)));
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

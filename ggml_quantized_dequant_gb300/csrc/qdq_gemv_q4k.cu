// Q4_K dequant-GEMV family: plain GEMV, fused SwiGLU expansion, and GEMV plus
// residual (the down projection of the FFN block).
//
// "Module cuda_lane", Functions:
//   try_q4k_soa_gemv                -- on-device Q4_K dequant-GEMV;
//   try_q4k_soa_fused_swiglu        -- out[i] = silu(gate_row_i . x) * (up_row_i . x),
//                                      one kernel, one read of x for both weights;
//   try_q4k_soa_ffn_block_residual  -- out = residual + FFN(x), mid kept on device.
//
// Per 32-weight sub-block j of a superblock, weight = d*sc_j*q - dmin*m_j, so a
// row's dot product is  sum_j ( d*sc_j * S_j - dmin*m_j * X_j )  with
// S_j = sum_k q_k x_k over the sub-block and X_j = sum_k x_k.  X_j depends only
// on x and is computed once per CTA; S_j is the per-weight work.
//
// Design (HBM-bound, like the Q8_0 kernel): one CTA per SM over a contiguous
// row range, L2 bulk prefetch of that range before the programmatic-launch
// wait, x and X_j in shared memory, two rows per warp task.  Lane l handles
// sub-blocks l, l+32, ... of a row: 16 bytes of packed nibbles (weight e of
// the sub-block in nibble e&1 of byte e/2) with one 128-bit load, and the
// 16-byte header record of its superblock (d, dmin and the twelve-bit
// (sc_j, m_j) field of its own j = l mod 8).
//
// Nibble -> f32 exactly with one logic op: the nibble at bit p (p = 0, 4, 8,
// 12 of a 16-bit half) is masked in place and OR-ed into a float whose
// exponent makes bit p worth 1, giving 2^(23-p) + q; one packed subtraction
// of the constants recovers q for two weights at once.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

enum Mode { kPlain = 0, kSwiglu = 1, kResidual = 2 };

// Eight nibbles of `w` (weights 0..7 of a word) -> four exact float pairs.
__device__ __forceinline__ void u4x8_to_f2(uint32_t w, f2 q[4]) {
  const f2 bias01 = f2_make(-8388608.0f, -524288.0f);   // -2^23, -2^19
  const f2 bias23 = f2_make(-32768.0f, -2048.0f);       // -2^15, -2^11
  const uint32_t h = w >> 16;
  q[0] = f2_add(f2_from_u32((w & 0x000Fu) | 0x4B000000u, (w & 0x00F0u) | 0x49000000u), bias01);
  q[1] = f2_add(f2_from_u32((w & 0x0F00u) | 0x47000000u, (w & 0xF000u) | 0x45000000u), bias23);
  q[2] = f2_add(f2_from_u32((h & 0x000Fu) | 0x4B000000u, (h & 0x00F0u) | 0x49000000u), bias01);
  q[3] = f2_add(f2_from_u32((h & 0x0F00u) | 0x47000000u, (h & 0xF000u) | 0x45000000u), bias23);
}

// (D, M) = (d*sc_j, dmin*m_j) for this lane's sub-block j from a header record.
// `sel`/`sh` pick the 12-bit field j of the 96-bit field in words y, z, w.
__device__ __forceinline__ f2 q4k_scale_pair(const uint4 h, int sel, int sh) {
  const uint32_t lo = sel == 0 ? h.y : (sel == 1 ? h.z : h.w);
  const uint32_t hi = sel == 0 ? h.z : h.w;
  const uint32_t v = __funnelshift_r(lo, hi, sh);
  // sc in bits 0..5 -> 2^23 + sc;  m in bits 6..11 -> 2^17 + m
  const f2 scm = f2_add(f2_from_u32((v & 0x3Fu) | 0x4B000000u, (v & 0xFC0u) | 0x48000000u),
                        f2_make(-8388608.0f, -131072.0f));
  const __half2 dd = *reinterpret_cast<const __half2 *>(&h.x);
  const float2 df = __half22float2(dd);  // (d, dmin)
  return f2_mul(f2_make(df.x, df.y), scm);
}

template <int NB, int MODE>
__global__ void __launch_bounds__(kThreads) q4k_gemv_kernel(const uint8_t *__restrict__ W,
                                                            const uint8_t *__restrict__ W2,
                                                            const float *__restrict__ x,
                                                            const float *residual, float *y, int n_out,
                                                            int n_in, int l2_prefetch) {
  extern __shared__ float4 smem4[];
  constexpr int kRowsPerTask = MODE == kSwiglu ? 1 : 2;  // output rows per warp task
  const int nsb = n_in >> 5;                              // sub-blocks per row
  const int64_t q_bytes = int64_t(n_out) * (n_in >> 1);
  const int64_t q_row = n_in >> 1;
  const int64_t h_row = int64_t(n_in >> 8) * 16;
  const int r_begin = int(int64_t(blockIdx.x) * n_out / gridDim.x);
  const int r_end = int(int64_t(blockIdx.x + 1) * n_out / gridDim.x);

  if (l2_prefetch && threadIdx.x == 0) {
    prefetch_range_l2(W, q_bytes, r_begin * q_row, r_end * q_row);
    prefetch_range_l2(W + q_bytes, int64_t(n_out) * h_row, r_begin * h_row, r_end * h_row);
    if (MODE == kSwiglu) {
      prefetch_range_l2(W2, q_bytes, r_begin * q_row, r_end * q_row);
      prefetch_range_l2(W2 + q_bytes, int64_t(n_out) * h_row, r_begin * h_row, r_end * h_row);
    }
  }
  pdl_launch_dependents();
  pdl_wait();

  float4 *xs = smem4;                                                   // NB * nsb lines of 8 chunks
  float *xsum = reinterpret_cast<float *>(smem4 + size_t(NB) * nsb * 8);  // NB * nsb sums
  {
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const int n4 = NB * nsb * 8;
    for (int i = threadIdx.x; i < n4; i += kThreads) xs[swz_chunk(i >> 3, i & 7)] = x4[i];
  }
  __syncthreads();
  for (int l = threadIdx.x; l < NB * nsb; l += kThreads) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 v = xs[swz_chunk(l, c)];
      s += (v.x + v.y) + (v.z + v.w);
    }
    xsum[l] = s;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane & 7;  // sub-block index within the superblock, fixed per lane
  const int sel = (12 * j) >> 5, sh = (12 * j) & 31;
  const int ntask = (r_end - r_begin + kRowsPerTask - 1) / kRowsPerTask;

  for (int task = warp; task < ntask; task += kWarps) {
    const int r0 = r_begin + task * kRowsPerTask;
    const uint8_t *qrow[2];
    const uint8_t *hrow[2];
    if (MODE == kSwiglu) {
      qrow[0] = W + r0 * q_row;
      hrow[0] = W + q_bytes + r0 * h_row;
      qrow[1] = W2 + r0 * q_row;
      hrow[1] = W2 + q_bytes + r0 * h_row;
    } else {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = min(r0 + r, r_end - 1);  // a missing last row re-reads the previous one; result dropped
        qrow[r] = W + row * q_row;
        hrow[r] = W + q_bytes + row * h_row;
      }
    }
    f2 acc[2][NB];
    float accm[2][NB];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        acc[r][b] = f2_make(0.f, 0.f);
        accm[r][b] = 0.f;
      }

    int J = lane;
    uint4 qv[2], hv[2];
    if (J < nsb) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        qv[r] = ldg_stream(qrow[r] + int64_t(J) * 16);
        hv[r] = ldg_stream(hrow[r] + int64_t(J >> 3) * 16);
      }
    }
    while (J < nsb) {
      const int nx = J + 32;
      uint4 qn[2], hn[2];
      if (nx < nsb) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          qn[r] = ldg_stream(qrow[r] + int64_t(nx) * 16);
          hn[r] = ldg_stream(hrow[r] + int64_t(nx >> 3) * 16);
        }
      }
      f2 DM[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) DM[r] = q4k_scale_pair(hv[r], sel, sh);

      f2 S[2][NB];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) S[r][b] = f2_make(0.f, 0.f);
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        f2 q[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint32_t w = wd == 0 ? qv[r].x : wd == 1 ? qv[r].y : wd == 2 ? qv[r].z : qv[r].w;
          u4x8_to_f2(w, q[r]);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const int line = b * nsb + J;
          const float4 xa = xs[swz_chunk(line, 2 * wd)];
          const float4 xb = xs[swz_chunk(line, 2 * wd + 1)];
          const f2 x01 = f2_make(xa.x, xa.y), x23 = f2_make(xa.z, xa.w);
          const f2 x45 = f2_make(xb.x, xb.y), x67 = f2_make(xb.z, xb.w);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            S[r][b] = f2_fma(q[r][0], x01, S[r][b]);
            S[r][b] = f2_fma(q[r][1], x23, S[r][b]);
            S[r][b] = f2_fma(q[r][2], x45, S[r][b]);
            S[r][b] = f2_fma(q[r][3], x67, S[r][b]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float D, M;
        f2_split(DM[r], D, M);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          acc[r][b] = f2_fma(f2_make(D, D), S[r][b], acc[r][b]);
          accm[r][b] = fmaf(-M, xsum[b * nsb + J], accm[r][b]);
        }
      }
      if (nx < nsb) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          qv[r] = qn[r];
          hv[r] = hn[r];
        }
      }
      J = nx;
    }

    float v[2][NB];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float lo, hi;
        f2_split(acc[r][b], lo, hi);
        v[r][b] = warp_sum((lo + hi) + accm[r][b]);
      }
    if (lane == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (MODE == kSwiglu) {
          const float g = v[0][b], u = v[1][b];
          y[int64_t(b) * n_out + r0] = g / (1.0f + expf(-g)) * u;
        } else {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int row = r0 + r;
            if (row < r_end) {
              const int64_t o = int64_t(b) * n_out + row;
              y[o] = MODE == kResidual ? residual[o] + v[r][b] : v[r][b];
            }
          }
        }
      }
    }
  }
}

template <int NB, int MODE>
int launch_nb(const uint8_t *W, const uint8_t *W2, const float *x, const float *residual, float *y,
              int n_out, int n_in, cudaStream_t s, const DeviceInfo &di) {
  const int nsb = n_in >> 5;
  const size_t smem = gemv_smem_bytes(di, size_t(NB) * nsb * (8 * sizeof(float4) + sizeof(float)));
  auto kern = q4k_gemv_kernel<NB, MODE>;
  if (smem > 48 * 1024) {
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const int rows_per_task = MODE == kSwiglu ? 1 : 2;
  int grid = di.sm_count * opt_ctas_per_sm();
  const int max_grid = (n_out + rows_per_task - 1) / rows_per_task;
  if (grid > max_grid) grid = max_grid;
  const cudaError_t e = launch(kern, dim3(grid), dim3(kThreads), smem, s, W, W2, x, residual, y, n_out,
                               n_in, opt_l2_prefetch());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

template <int MODE>
int dispatch(int nb, const uint8_t *W, const uint8_t *W2, const float *x, const float *res, float *y,
             int n_out, int n_in, cudaStream_t s, const DeviceInfo &di) {
  switch (nb) {
    case 1: return launch_nb<1, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
    case 2: return launch_nb<2, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
    case 3: return launch_nb<3, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
    case 4: return launch_nb<4, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
    case 5: return launch_nb<5, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
    case 6: return launch_nb<6, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
    case 7: return launch_nb<7, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
    default: return launch_nb<8, MODE>(W, W2, x, res, y, n_out, n_in, s, di);
  }
}

}  // namespace

int launch_q4k_gemv(int mode, const void *Wv, const void *W2v, const float *x, const float *residual,
                    float *y, int n_out, int n_in, int batch, cudaStream_t s) {
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  const uint8_t *W = static_cast<const uint8_t *>(Wv);
  const uint8_t *W2 = static_cast<const uint8_t *>(W2v);
  const int budget = di.max_smem_optin < 200 * 1024 ? di.max_smem_optin : 200 * 1024;
  const int per_row = (n_in >> 5) * int(8 * sizeof(float4) + sizeof(float));
  int per = budget / per_row;
  if (per < 1) return QDQ_ERR_UNSUPPORTED;
  if (per > QDQ_MAX_GEMV_BATCH) per = QDQ_MAX_GEMV_BATCH;
  for (int b0 = 0; b0 < batch; b0 += per) {
    const int nb = (batch - b0) < per ? (batch - b0) : per;
    const float *xb = x + int64_t(b0) * n_in;
    const float *rb = residual ? residual + int64_t(b0) * n_out : nullptr;
    float *yb = y + int64_t(b0) * n_out;
    int rc;
    if (mode == kSwiglu) rc = dispatch<kSwiglu>(nb, W, W2, xb, rb, yb, n_out, n_in, s, di);
    else if (mode == kResidual) rc = dispatch<kResidual>(nb, W, W2, xb, rb, yb, n_out, n_in, s, di);
    else rc = dispatch<kPlain>(nb, W, W2, xb, rb, yb, n_out, n_in, s, di);
    if (rc != QDQ_OK) return rc;
  }
  return QDQ_OK;
}

}  // namespace qdq

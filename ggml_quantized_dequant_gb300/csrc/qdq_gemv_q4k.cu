// Q4_K dequant-GEMV family: plain GEMV, fused SwiGLU expansion, and GEMV plus
// residual (the down projection of the FFN block).
//
// "Module cuda_lane", Functions:
//   try_q4k_soa_gemv                -- on-device Q4_K dequant-GEMV;
//   try_q4k_soa_fused_swiglu        -- out[i] = silu(gate_row_i . x) * (up_row_i . x),
//                                      one kernel, one read of x for both weights;
//   try_q4k_soa_ffn_block_residual  -- out = residual + FFN(x), mid kept on device.
//
// Per 32-weight sub-block j of a superblock, weight = d*sc_j*q - dmin*m_j
// = d*sc_j*(q - mu_j) - R_j with an integer shift mu_j and R_j = dmin*m_j -
// d*sc_j*mu_j (q4k_mu), so a row's dot product is
// sum_j ( d*sc_j * S_j - R_j * X_j )  with S_j = sum_k (q_k - mu_j) x_k over the
// sub-block and X_j = sum_k x_k.  X_j depends only on x and is computed once per
// CTA; S_j is the per-weight work.  The shift keeps the rounding error a small
// multiple of sum |w||x| even where d*sc_j*q and dmin*m_j nearly cancel.
//
// Design (HBM-bound, like the Q8_0 kernel): one CTA per SM over a contiguous
// row range, L2 bulk prefetch of that range before the programmatic-launch
// wait, x and X_j in shared memory, two rows per warp task (gate and up row of
// the same output for SwiGLU), tasks x lane-iterations split evenly across the
// warps, P iterations of loads in flight per lane.  Lane l handles
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

// x staging: sub-block J (32 floats) of batch row b at float offset
// (b * nsb + J) * kXStride, followed by its sum X_J in the next float; the
// 144-byte stride puts the 16-byte reads of eight consecutive sub-blocks in
// eight different bank groups (9J mod 8 = J mod 8), with no index math.
constexpr int kXStride = 36;

// (D, M) = (d*sc_j, dmin*m_j) for this lane's sub-block j from a header record.
// Field j (sc in bits 0-5, m in bits 6-11) starts at bit 12j of words y,z,w:
// lanes j < 3 read it from (y, z), 3 <= j < 6 from (z, w), j >= 6 from w.
__device__ __forceinline__ float2 q4k_scale_pair(const uint4 h, bool g0, bool g1, int sh, const Magic &k) {
  const uint32_t lo = g0 ? h.y : (g1 ? h.z : h.w);
  const uint32_t hi = g0 ? h.z : h.w;
  const uint32_t v = __funnelshift_r(lo, hi, sh);
  // sc -> 2^23 + sc;  m (bits 6..11) -> 2^17 + m
  const float2 scm = q4k_field_to_f2(v, k);
  const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&h.x));  // (d, dmin)
  return __fmul2_rn(dd, scm);
}

template <int NB, int MODE, int P>
__global__ void __launch_bounds__(kThreads) q4k_gemv_kernel(const uint8_t *__restrict__ W,
                                                            const uint8_t *__restrict__ W2,
                                                            const float *__restrict__ x,
                                                            const float *residual, float *y, int n_out,
                                                            int n_in, int l2_prefetch, const Magic mg_param) {
  extern __shared__ float4 smem4[];
  const Magic mg = lane_magic(mg_param);
  constexpr int kRowsPerTask = MODE == kSwiglu ? 1 : 2;  // output rows per warp task
  constexpr int kOut = MODE == kSwiglu ? 2 : 1;          // sums per output row
  const int nsb = n_in >> 5;                              // sub-blocks per row
  const int64_t q_bytes = int64_t(n_out) * (n_in >> 1);
  const int64_t q_row = n_in >> 1;
  const int64_t h_row = int64_t(n_in >> 8) * 16;
  const int r_begin = int(int64_t(blockIdx.x) * n_out / gridDim.x);
  const int r_end = int(int64_t(blockIdx.x + 1) * n_out / gridDim.x);
  const int nrows = r_end - r_begin;

  if (l2_prefetch && threadIdx.x == 0) {
    prefetch_range_l2(W, q_bytes, r_begin * q_row, r_end * q_row);
    prefetch_range_l2(W + q_bytes, int64_t(n_out) * h_row, r_begin * h_row, r_end * h_row);
    if (MODE == kSwiglu) {
      prefetch_range_l2(W2, q_bytes, r_begin * q_row, r_end * q_row);
      prefetch_range_l2(W2 + q_bytes, int64_t(n_out) * h_row, r_begin * h_row, r_end * h_row);
    }
  }
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane & 7;  // sub-block index within the superblock, fixed per lane
  const bool g0 = j < 3, g1 = j < 6;
  const int sh = (12 * j) & 31;
  const int itpt = (nsb + 31) >> 5;  // lane iterations per task ("units")
  const int ntask = (nrows + kRowsPerTask - 1) / kRowsPerTask;
  const int total = ntask * itpt;
  // balanced contiguous unit ranges; never shorter than a task, so at most two
  // warps add into any output (two commuting shared-memory adds: deterministic)
  int per = (total + kWarps - 1) / kWarps;
  if (per < itpt) per = itpt;
  const int k0 = min(warp * per, total);
  const int k1 = min(k0 + per, total);

  // load cursor with per-task row pointers; the weight ring is filled before
  // waiting on the previous kernel, which only x depends on
  int lt = k0 / itpt, li = k0 - lt * itpt;
  const uint8_t *lq[2];
  const uint8_t *lh[2];
  auto set_rows = [&]() {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint8_t *base = (MODE == kSwiglu && r == 1) ? W2 : W;
      const int row = MODE == kSwiglu ? r_begin + lt : r_begin + min(2 * lt + r, nrows - 1);
      lq[r] = base + row * q_row + lane * 16;
      lh[r] = base + q_bytes + row * h_row + (lane >> 3) * 16;
    }
  };
  uint4 qb[P][2], hb[P][2];
  auto load = [&](int slot) {
    if (lane + 32 * li < nsb) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        qb[slot][r] = ldg_stream(lq[r] + li * 512);
        hb[slot][r] = ldg_stream(lh[r] + li * 64);
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
  float *ysm = xs + size_t(NB) * nsb * kXStride;  // [kOut][nrows][NB]
  {
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    for (int i = threadIdx.x; i < NB * nsb * 8; i += kThreads)
      *reinterpret_cast<float4 *>(xs + (i >> 3) * kXStride + (i & 7) * 4) = x4[i];
    for (int i = threadIdx.x; i < kOut * nrows * NB; i += kThreads) ysm[i] = 0.f;
  }
  __syncthreads();
  for (int l = threadIdx.x; l < NB * nsb; l += kThreads) {
    const float *xl = xs + l * kXStride;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 v = *reinterpret_cast<const float4 *>(xl + 4 * c);
      s += (v.x + v.y) + (v.z + v.w);
    }
    xs[l * kXStride + 32] = s;
  }
  __syncthreads();

  if (k0 < k1) {
    int ct = k0 / itpt, ci = k0 - ct * itpt;  // compute cursor
    float2 acc[2][NB];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = f2(0.f, 0.f);

    for (int kb = k0; kb < k1; kb += P) {
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const int k = kb + p;
        if (k < k1) {
          const int J = lane + 32 * ci;
          if (J < nsb) {
            // (d sc_j, R) with R = dmin m_j - d sc_j mu: the quants are summed as q - mu
            // (q4k_mu), which keeps near-cancelling weights' error proportional to sum |w||x|
            float2 DM[2], b01[2], b23[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              DM[r] = q4k_scale_pair(hb[p][r], g0, g1, sh, mg);
              const float mu = q4k_mu(DM[r]);
              DM[r].y = fmaf(-DM[r].x, mu, DM[r].y);
              b01[r] = __fadd2_rn(mg.b_u4_01, f2(-mu, -mu));
              b23[r] = __fadd2_rn(mg.b_u4_23, f2(-mu, -mu));
            }
            float2 S[2][NB], T[2][NB];  // two independent chains per row
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int b = 0; b < NB; ++b) S[r][b] = T[r][b] = f2(0.f, 0.f);
            const float *xj = xs + J * kXStride;
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
              float2 q[2][4];
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const uint32_t w = wd == 0 ? qb[p][r].x : wd == 1 ? qb[p][r].y : wd == 2 ? qb[p][r].z : qb[p][r].w;
                u4x8_to_f2_shifted(w, mg, b01[r], b23[r], q[r]);
              }
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                const float4 xa = *reinterpret_cast<const float4 *>(xj + b * nsb * kXStride + 8 * wd);
                const float4 xb = *reinterpret_cast<const float4 *>(xj + b * nsb * kXStride + 8 * wd + 4);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                  S[r][b] = __ffma2_rn(q[r][0], f2(xa.x, xa.y), S[r][b]);
                  T[r][b] = __ffma2_rn(q[r][1], f2(xa.z, xa.w), T[r][b]);
                  S[r][b] = __ffma2_rn(q[r][2], f2(xb.x, xb.y), S[r][b]);
                  T[r][b] = __ffma2_rn(q[r][3], f2(xb.z, xb.w), T[r][b]);
                }
              }
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const float xsum = xj[b * nsb * kXStride + 32];
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                // (acc.x, acc.y) += (D * S.x, D * S.y - R * X_J)
                const float2 t = __ffma2_rn(f2(DM[r].x, DM[r].x), __fadd2_rn(S[r][b], T[r][b]), acc[r][b]);
                acc[r][b] = f2(t.x, fmaf(-DM[r].y, xsum, t.y));
              }
            }
          }
          if (k + P < k1) load(p);
          if (++ci == itpt || k + 1 == k1) {  // this warp's share of task ct is complete
#pragma unroll
            for (int r = 0; r < 2; ++r) {
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                const float v = warp_sum(acc[r][b].x + acc[r][b].y);
                if (lane == 0) {
                  if (MODE == kSwiglu) {
                    atomicAdd(&ysm[(r * nrows + ct) * NB + b], v);
                  } else if (2 * ct + r < nrows) {
                    atomicAdd(&ysm[(2 * ct + r) * NB + b], v);
                  }
                }
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
    const int64_t o = int64_t(b) * n_out + r_begin + row;
    if (MODE == kSwiglu) {
      const float g = ysm[i], u = ysm[nrows * NB + i];
      y[o] = g / (1.0f + expf(-g)) * u;
    } else if (MODE == kResidual) {
      y[o] = residual[o] + ysm[i];
    } else {
      y[o] = ysm[i];
    }
  }
}

template <int NB, int MODE>
int launch_nb(const uint8_t *W, const uint8_t *W2, const float *x, const float *residual, float *y,
              int n_out, int n_in, cudaStream_t s, const DeviceInfo &di) {
  const int nsb = n_in >> 5;
  const int rows_per_task = MODE == kSwiglu ? 1 : 2;
  const int grid = gemv_grid(di, n_out, rows_per_task);
  const int max_rows = (n_out + grid - 1) / grid;
  const int outs = MODE == kSwiglu ? 2 : 1;
  const size_t smem = gemv_smem_bytes(
      di, size_t(NB) * nsb * kXStride * sizeof(float) + size_t(outs) * max_rows * NB * sizeof(float));
  constexpr int P = NB <= 2 ? 4 : 2;  // loads in flight per lane
  auto kern = q4k_gemv_kernel<NB, MODE, P>;
  if (smem > 48 * 1024) {
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const cudaError_t e = launch(kern, dim3(grid), dim3(kThreads), smem, s, W, W2, x, residual, y, n_out,
                               n_in, opt_l2_prefetch() == 1, make_magic());
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
  if (gemv_xs_supported(n_in, batch, 1)) return launch_gemv_xs(1, mode, Wv, W2v, x, residual, y, n_out, n_in, s);
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  const uint8_t *W = static_cast<const uint8_t *>(Wv);
  const uint8_t *W2 = static_cast<const uint8_t *>(W2v);
  const int budget = di.max_smem_optin < 200 * 1024 ? di.max_smem_optin : 200 * 1024;
  const int rows_per_task = mode == kSwiglu ? 1 : 2;
  const int grid = gemv_grid(di, n_out, rows_per_task);
  const int max_rows = (n_out + grid - 1) / grid;
  const int per_batch = (n_in >> 5) * kXStride * int(sizeof(float)) +
                        (mode == kSwiglu ? 2 : 1) * max_rows * int(sizeof(float));
  int per = budget / per_batch;
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

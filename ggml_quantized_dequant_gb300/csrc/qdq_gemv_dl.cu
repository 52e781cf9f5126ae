// Batch-1 dequant-GEMV with per-warp bulk-copy rings: every warp of the SM
// computes, and each streams its own weights into its own shared-memory slots.
//
// "Module cuda_lane", Functions: try_q8_0_cuda_gemv (Q8_0 GEMV), try_q4k_soa_gemv
// (Q4_K GEMV), try_q4k_soa_fused_swiglu (out[i] = silu(gate_i . x) * (up_i . x)),
// try_q4k_soa_ffn_block_residual (out = residual + W_down . mid), try_q4k_soa_qkv
// (Q, K, V from one activation); "QTensorEngine", dispatch_gemm_into (Q6_K).
//
// Layout of the work is the x-stationary one of the ring kernel: lane l of
// slice warp s owns the 32-weight column block 32 s + l for the whole kernel
// and keeps its 32 activations in registers; WPR = ceil(n_in / 1024) slice warps
// cover a row; G groups of slice warps take contiguous shares of the CTA's rows
// (one CTA per SM, about 16 warps).  A warp handles 4 (virtual) rows per stage:
// lane 0 copies the warp's slice of the 4 rows (quant bytes and scales, 1-D bulk
// copies completing on the slot's mbarrier) into one of its S slots, S - 1
// stages ahead; the lanes read their block from the slot, the slot is refilled at
// once, and a recursive-halving butterfly leaves row k's warp total in lane 8k;
// the slice totals of a row are added in fixed order at the end (deterministic).
//
// Against the co-resident ring kernel (a producer warp, a ring sized to half an
// SM so that the next kernel's CTA fits beside it, 6-9 computing warps): here
// every warp of the SM computes, each warp has S - 1 stages of copies in flight
// without holding registers for them, and the first S stages plus a bulk L2
// prefetch of the CTA's rows are issued before the wait for the previous kernel.
//
// Arithmetic: f32 (weights converted exactly, packed f32x2 FMAs; Q4_K with the
// sub-block shift q4k_mu), within 1e-5 sum |w||x| for every finite input.
// Every wait is bounded (2 s); a wait that runs out is counted
// (qdq_pipeline_timeouts) and the warp stops issuing and winds down.
#include "qdq_internal.cuh"

namespace qdq {

__device__ unsigned int g_dl_timeouts = 0;

namespace {

constexpr int kMaxWarps = 16;
enum Fmt { kQ8 = 0, kQ4 = 1, kQ6 = 2 };
enum Epi { kPlain = 0, kSwiglu = 1, kResidual = 2, kQkv = 3 };

struct DlArgs {
  const uint8_t *W, *W2, *W3;  // matrix (gate / W_q), up / W_k, W_v
  const float *x;
  const float *residual;
  float *y, *y2, *y3;          // output (q), k, v
  int seg1, seg2;              // QKV: rows [0, seg1) W_q, [seg1, seg2) W_k, [seg2, n_out) W_v
  int n_out, n_in, wpr, groups, slots, prefetch;
};

template <int FMT>
__device__ __forceinline__ int64_t q_row_bytes(int n_in) {
  return FMT == kQ8 ? int64_t(n_in) : FMT == kQ4 ? int64_t(n_in >> 1) : q6k_row_bytes(n_in);
}
template <int FMT>
__device__ __forceinline__ int64_t s_row_bytes(int n_in) {
  return FMT == kQ8 ? int64_t(n_in >> 4) : FMT == kQ4 ? int64_t(n_in >> 8) * 16 : 0;
}

// Matrix base, its row count and the local row of global (virtual) row R.
template <int EPI>
__device__ __forceinline__ const uint8_t *row_matrix(const DlArgs &a, int R, int up, int &lr, int &nm) {
  if (EPI == kQkv) {
    if (R < a.seg1) {
      lr = R;
      nm = a.seg1;
      return a.W;
    }
    if (R < a.seg2) {
      lr = R - a.seg1;
      nm = a.seg2 - a.seg1;
      return a.W2;
    }
    lr = R - a.seg2;
    nm = a.n_out - a.seg2;
    return a.W3;
  }
  lr = R;
  nm = a.n_out;
  return (EPI == kSwiglu && up) ? a.W2 : a.W;
}

// Bytes per row of one slice warp's copy (its up to 32 blocks of 32 weights): the
// quant part and the scale part.  Q6_K copies its low bits, high bits and scales
// as the quant part and the row's whole d region as the scale part.
struct SliceBytes {
  uint32_t q, s;       // per row in the slot (the 32-block maximum)
  uint32_t qc, sc;     // per row actually copied for this slice (nb blocks)
};
template <int FMT>
__device__ __forceinline__ SliceBytes slice_bytes(int n_in, int nb) {
  SliceBytes b;
  if (FMT == kQ8) {
    b.q = 1024, b.s = 64, b.qc = 32 * nb, b.sc = 2 * nb;
  } else if (FMT == kQ4) {
    b.q = 512, b.s = 64, b.qc = 16 * nb, b.sc = 2 * nb;  // 16-byte header per 8 blocks
  } else {
    const uint32_t d_off = uint32_t(n_in / 2 + n_in / 4 + n_in / 16);
    b.q = 832, b.s = uint32_t(q6k_row_bytes(n_in)) - d_off, b.qc = 26 * nb, b.sc = b.s;
  }
  return b;
}

// Slot layout: [4 rows x q part][4 rows x s part]; every part starts on 16 bytes.
template <int FMT, int EPI>
__device__ __forceinline__ void issue_stage(const DlArgs &a, uint8_t *slot, uint64_t *bar, int rr, int ge, int slice,
                                            int nb, const SliceBytes &sb) {
  constexpr int kV = EPI == kSwiglu ? 2 : 1;
  const int n_in = a.n_in;
  const int64_t qr = q_row_bytes<FMT>(n_in), sr = s_row_bytes<FMT>(n_in);
  mbar_arrive_expect_tx(bar, 4 * (sb.qc + sb.sc));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int up = kV == 2 ? (k & 1) : 0;
    int R = rr + (kV == 2 ? (k >> 1) : k);
    R = R < ge ? R : ge - 1;  // past the group's end: its last row again (dropped)
    int lr, nm;
    const uint8_t *base = row_matrix<EPI>(a, R, up, lr, nm);
    uint8_t *qd = slot + k * sb.q;
    uint8_t *sd = slot + 4 * sb.q + k * sb.s;
    if (FMT == kQ6) {
      const uint8_t *row = base + int64_t(lr) * qr;
      bulk_copy_g2s(qd, row + 512 * slice, 16 * nb, bar);                          // low bits
      bulk_copy_g2s(qd + 512, row + n_in / 2 + 256 * slice, 8 * nb, bar);          // high bits
      bulk_copy_g2s(qd + 768, row + n_in / 2 + n_in / 4 + 64 * slice, 2 * nb, bar);  // scales
      bulk_copy_g2s(sd, row + n_in / 2 + n_in / 4 + n_in / 16, sb.s, bar);         // the row's d values
    } else {
      bulk_copy_g2s(qd, base + int64_t(lr) * qr + int64_t(sb.q) * slice, sb.qc, bar);
      bulk_copy_g2s(sd, base + int64_t(nm) * qr + int64_t(lr) * sr + 64 * slice, sb.sc, bar);
    }
  }
}

template <int FMT, int EPI>
__global__ void __launch_bounds__(32 * kMaxWarps) gemv_dl_kernel(const DlArgs a, const Magic mg_param) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kV = EPI == kSwiglu ? 2 : 1;  // virtual rows per output row
  constexpr int kRowsPerStage = 4 / kV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int n_in = a.n_in, G = a.groups, S = a.slots;
  const int slice = warp % a.wpr, grp = warp / a.wpr;
  const int r0 = int(int64_t(blockIdx.x) * a.n_out / gridDim.x);
  const int r1 = int(int64_t(blockIdx.x + 1) * a.n_out / gridDim.x);
  const int nreal = r1 - r0;
  const int gb = r0 + grp * nreal / G, ge = r0 + (grp + 1) * nreal / G;  // this group's output rows
  const int nst = ((ge - gb) * kV + 3) / 4;                               // its stages of 4 virtual rows
  const int nblk = n_in >> 5;
  const int nb = min(32, nblk - 32 * slice);  // blocks of this slice
  const SliceBytes sb = slice_bytes<FMT>(n_in, nb);
  const uint32_t slot_bytes = 4 * (sb.q + sb.s);
  uint8_t *ring = smem + size_t(warp) * S * slot_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + size_t(nwarps) * S * slot_bytes) + warp * S;
  float *psum = reinterpret_cast<float *>(reinterpret_cast<uint64_t *>(smem + size_t(nwarps) * S * slot_bytes) +
                                          nwarps * S);  // [local virtual row][wpr]
  __shared__ int s_abort;

  if (lane == 0)
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
  if (threadIdx.x == 0) s_abort = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  // HBM starts streaming this CTA's rows at once: the weights do not depend on the previous kernel
  if (a.prefetch && threadIdx.x == 0) {
    const int64_t qr = q_row_bytes<FMT>(n_in), sr = s_row_bytes<FMT>(n_in);
    if (EPI == kQkv) {
      const uint8_t *Wm[3] = {a.W, a.W2, a.W3};
      const int off[4] = {0, a.seg1, a.seg2, a.n_out};
      for (int m = 0; m < 3; ++m) {
        const int lo = max(r0, off[m]) - off[m], hi = min(r1, off[m + 1]) - off[m], nm = off[m + 1] - off[m];
        if (lo >= hi) continue;
        prefetch_range_l2(Wm[m], int64_t(nm) * qr, lo * qr, hi * qr);
        if (sr) prefetch_range_l2(Wm[m] + int64_t(nm) * qr, int64_t(nm) * sr, lo * sr, hi * sr);
      }
    } else {
      for (int m = 0; m < kV; ++m) {
        const uint8_t *Wm = m ? a.W2 : a.W;
        prefetch_range_l2(Wm, int64_t(a.n_out) * qr, r0 * qr, r1 * qr);
        if (sr) prefetch_range_l2(Wm + int64_t(a.n_out) * qr, int64_t(a.n_out) * sr, r0 * sr, r1 * sr);
      }
    }
  }
  // this warp's first S stages, before the dependency wait
  int issued = 0;
  if (lane == 0)
    for (; issued < S && issued < nst; ++issued)
      issue_stage<FMT, EPI>(a, ring + issued * slot_bytes, &bars[issued], gb + issued * kRowsPerStage, ge, slice, nb,
                            sb);
  pdl_launch_dependents();

  const int blk = slice * 32 + lane;
  const bool valid = blk < nblk;
  const Magic mg = lane_magic(mg_param);
  pdl_wait();  // the activations come from the previous kernel
  float2 xr[16];
  float xsum = 0.f;
  {
    const float4 *xp = reinterpret_cast<const float4 *>(a.x + (valid ? blk : 0) * 32);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 v = valid ? ld_after_wait(xp + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      xr[2 * c] = f2(v.x, v.y);
      xr[2 * c + 1] = f2(v.z, v.w);
    }
    if constexpr (FMT == kQ4) {
      float2 t = f2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 16; ++c) t = __fadd2_rn(t, xr[c]);
      xsum = t.x + t.y;
    }
  }
  // Q4_K: this lane's 12-bit (sc, m) field lives at bit 12 j of header words 1..3
  const int j = lane & 7;
  const bool g0 = j < 3, g1 = j < 6;
  const int sh = (12 * j) & 31;
  const int bq = valid ? blk : 0;

  for (int t = 0; t < nst; ++t) {
    const int sl = t % S;
    if (!mbar_wait(&bars[sl], (t / S) & 1)) {
      s_abort = 1;
      break;
    }
    const uint8_t *slot = ring + sl * slot_bytes;
    // this lane's data of the 4 rows into registers, then the slot is refilled
    uint4 ra[4], rb[4];
    uint32_t rc[4], rd[4];
    uint2 rh[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint8_t *qd = slot + k * sb.q;
      const uint8_t *sd = slot + 4 * sb.q + k * sb.s;
      if constexpr (FMT == kQ8) {
        ra[k] = *reinterpret_cast<const uint4 *>(qd + 32 * lane);
        rb[k] = *reinterpret_cast<const uint4 *>(qd + 32 * lane + 16);
        rc[k] = *reinterpret_cast<const unsigned short *>(sd + 2 * lane);
      } else if constexpr (FMT == kQ4) {
        ra[k] = *reinterpret_cast<const uint4 *>(qd + 16 * lane);
        rb[k] = *reinterpret_cast<const uint4 *>(sd + 16 * (lane >> 3));
      } else {
        ra[k] = *reinterpret_cast<const uint4 *>(qd + 16 * lane);
        rh[k] = *reinterpret_cast<const uint2 *>(qd + 512 + 8 * lane);
        rc[k] = *reinterpret_cast<const unsigned short *>(qd + 768 + 2 * lane);
        rd[k] = *reinterpret_cast<const unsigned short *>(sd + 2 * (bq >> 3));
      }
    }
    __syncwarp();
    if (lane == 0 && t + S < nst && !*reinterpret_cast<volatile int *>(&s_abort)) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the reads above before the refill
      issue_stage<FMT, EPI>(a, ring + sl * slot_bytes, &bars[sl], gb + (t + S) * kRowsPerStage, ge, slice, nb, sb);
      issued = t + S + 1;
    }
    float part[4];
    if constexpr (FMT == kQ8) {
      float2 s0[4], s1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) s0[k] = s1[k] = f2(0.f, 0.f);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 &u = kk < 4 ? ra[k] : rb[k];
          const uint32_t w = (kk & 3) == 0 ? u.x : (kk & 3) == 1 ? u.y : (kk & 3) == 2 ? u.z : u.w;
          float2 q01, q23;
          s8x4_to_f2(w, mg, q01, q23);
          s0[k] = __ffma2_rn(q01, xr[2 * kk], s0[k]);
          s1[k] = __ffma2_rn(q23, xr[2 * kk + 1], s1[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 st = __fadd2_rn(s0[k], s1[k]);
        part[k] = __half2float(__ushort_as_half(uint16_t(rc[k]))) * (st.x + st.y);
      }
    } else if constexpr (FMT == kQ4) {
      float2 s0[4], s1[4], b01[4], b23[4];
      float D[4], R[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 h = rb[k];
        const uint32_t lo = g0 ? h.y : (g1 ? h.z : h.w);
        const uint32_t hi = g0 ? h.z : h.w;
        const float2 scm = q4k_field_to_f2(__funnelshift_r(lo, hi, sh), mg);  // (sc, m)
        const float2 DM = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&h.x)), scm);
        const float mu = q4k_mu(DM);
        D[k] = DM.x;
        R[k] = fmaf(-DM.x, mu, DM.y);
        b01[k] = __fadd2_rn(mg.b_u4_01, f2(-mu, -mu));
        b23[k] = __fadd2_rn(mg.b_u4_23, f2(-mu, -mu));
        s0[k] = s1[k] = f2(0.f, 0.f);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w = kk == 0 ? ra[k].x : kk == 1 ? ra[k].y : kk == 2 ? ra[k].z : ra[k].w;
          float2 qq[4];  // q - mu, exactly
          u4x8_to_f2_shifted(w, mg, b01[k], b23[k], qq);
          s0[k] = __ffma2_rn(qq[0], xr[4 * kk], s0[k]);
          s1[k] = __ffma2_rn(qq[1], xr[4 * kk + 1], s1[k]);
          s0[k] = __ffma2_rn(qq[2], xr[4 * kk + 2], s0[k]);
          s1[k] = __ffma2_rn(qq[3], xr[4 * kk + 3], s1[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 st = __fadd2_rn(s0[k], s1[k]);
        part[k] = fmaf(D[k], st.x + st.y, -R[k] * xsum);  // d sc sum((q - mu) x) - R sum(x)
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float d = __half2float(__ushort_as_half(uint16_t(rd[k])));
        const float ds0 = __fmul_rn(d, float(int8_t(rc[k] & 0xFFu)));
        const float ds1 = __fmul_rn(d, float(int8_t((rc[k] >> 8) & 0xFFu)));
        float2 v[16];
        q6k_block_to_f2(ra[k], rh[k], mg, v);
        float2 a0 = f2(0.f, 0.f), a1 = f2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 8; ++p) a0 = __ffma2_rn(v[p], xr[p], a0);
#pragma unroll
        for (int p = 8; p < 16; ++p) a1 = __ffma2_rn(v[p], xr[p], a1);
        part[k] = fmaf(ds1, a1.x + a1.y, ds0 * (a0.x + a0.y));
      }
    }
    // a lane past the slice's blocks read bytes no copy wrote: its partials are dropped
#pragma unroll
    for (int k = 0; k < 4; ++k) part[k] = valid ? part[k] : 0.f;
    butterfly4_rows(part, lane);
    if ((lane & 7) == 0) {
      const int k = lane >> 3;
      const int v = (gb - r0) * kV + 4 * t + k;  // local virtual row
      if (v < (ge - r0) * kV) psum[v * a.wpr + slice] = part[0];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) atomicAdd(&g_dl_timeouts, 1u);
  // epilogue: add the slice totals of each row in fixed order
  for (int r = threadIdx.x; r < nreal; r += blockDim.x) {
    if (EPI == kSwiglu) {
      const float *pg = psum + (2 * r) * a.wpr;
      const float *pu = psum + (2 * r + 1) * a.wpr;
      float g = 0.f, u = 0.f;
      for (int s = 0; s < a.wpr; ++s) {
        g += pg[s];
        u += pu[s];
      }
      a.y[r0 + r] = g / (1.0f + expf(-g)) * u;
    } else {
      float v = 0.f;
      const float *ps = psum + r * a.wpr;
      for (int s = 0; s < a.wpr; ++s) v += ps[s];
      const int R = r0 + r;
      if (EPI == kQkv) {
        if (R < a.seg1) a.y[R] = v;
        else if (R < a.seg2) a.y2[R - a.seg1] = v;
        else a.y3[R - a.seg2] = v;
      } else {
        a.y[R] = EPI == kResidual ? a.residual[R] + v : v;
      }
    }
  }
  // The last waits of the CTA: every copy this warp issued has landed before the CTA's
  // shared memory is released (the consumed stages have; this covers a stop on timeout).
  if (lane == 0) {
    bool drained = true;
    for (int t = issued - S < 0 ? 0 : issued - S; t < issued; ++t) drained = mbar_wait(&bars[t % S], (t / S) & 1) && drained;
    if (!drained) atomicAdd(&g_dl_timeouts, 1u);
  }
}

template <int FMT, int EPI>
int launch_dl(DlArgs a, cudaStream_t s) {
  DeviceInfo di;
  const cudaError_t e0 = device_info(&di);
  if (e0 != cudaSuccess) return fail_cuda(e0);
  constexpr int kV = EPI == kSwiglu ? 2 : 1;
  if ((a.n_in % 256) != 0) return QDQ_ERR_UNSUPPORTED;  // slice copies need whole 16-byte runs
  a.wpr = ((a.n_in >> 5) + 31) / 32;
  if (a.wpr > kMaxWarps) return QDQ_ERR_UNSUPPORTED;
  a.groups = opt_xs_groups() > 0 ? opt_xs_groups() : kMaxWarps / a.wpr;
  if (a.groups < 1) a.groups = 1;
  const int nwarps = a.wpr * a.groups;
  if (nwarps > kMaxWarps) return QDQ_ERR_UNSUPPORTED;
  int grid = di.sm_count * ctas_per_sm_or(1);
  if (grid > a.n_out) grid = a.n_out;
  const int max_rows = (a.n_out + grid - 1) / grid;
  const size_t psum_bytes = size_t(max_rows) * kV * a.wpr * sizeof(float);
  // slot bytes: 4 rows of the largest slice (as slice_bytes)
  const size_t d_off = size_t(a.n_in / 2 + a.n_in / 4 + a.n_in / 16);
  const size_t slot = FMT == kQ8 ? 4 * (1024 + 64) : FMT == kQ4 ? 4 * (512 + 64)
                                                                : 4 * (832 + (size_t(q6k_row_bytes(a.n_in)) - d_off));
  const long budget = long(di.max_smem_optin) - long(psum_bytes) - 1024;
  int S = int(budget / long(nwarps * (slot + 8)));
  if (S > 8) S = 8;
  if (S < 2) return QDQ_ERR_UNSUPPORTED;
  if (opt_xs_stages() > 0) S = opt_xs_stages();  // any S >= 1 is correct; 1 leaves no copy in flight
  a.slots = S;
  const size_t smem = size_t(nwarps) * S * slot + size_t(nwarps) * S * 8 + psum_bytes;
  if (smem > size_t(di.max_smem_optin)) return QDQ_ERR_UNSUPPORTED;
  // L2 prefetch of the CTA's rows: on by default when this call's weights fit in half the L2
  const int64_t w_bytes = int64_t(a.n_out) * (FMT == kQ8 ? int64_t(a.n_in) / 32 * 34
                                              : FMT == kQ4 ? int64_t(a.n_in) / 256 * 144
                                                           : q6k_row_bytes(a.n_in)) * kV;
  const int pf = opt_l2_prefetch();
  a.prefetch = pf == 3 ? 0 : pf == 1 ? 1 : (w_bytes <= int64_t(di.l2_bytes) / 2 ? 1 : 0);
  auto kern = gemv_dl_kernel<FMT, EPI>;
  const cudaError_t e1 = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
  if (e1 != cudaSuccess) return fail_cuda(e1);
  const cudaError_t e = launch(kern, dim3(grid), dim3(32 * nwarps), smem, s, a, make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace

int launch_gemv_dl(int fmt, int mode, const void *W, const void *W2, const float *x, const float *residual, float *y,
                   int n_out, int n_in, cudaStream_t s) {
  DlArgs a{};
  a.W = static_cast<const uint8_t *>(W);
  a.W2 = static_cast<const uint8_t *>(W2);
  a.x = x;
  a.residual = residual;
  a.y = y;
  a.n_out = n_out;
  a.n_in = n_in;
  if (fmt == 0) return launch_dl<kQ8, kPlain>(a, s);
  if (fmt == 2) return launch_dl<kQ6, kPlain>(a, s);
  if (mode == 1) return launch_dl<kQ4, kSwiglu>(a, s);
  if (mode == 2) return launch_dl<kQ4, kResidual>(a, s);
  return launch_dl<kQ4, kPlain>(a, s);
}

int read_dl_timeouts() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_dl_timeouts, sizeof(v)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_dl_timeouts, &zero, sizeof(zero)) != cudaSuccess) return -1;
  return int(v);
}

int launch_gemv_dl_qkv(const void *Wq, const void *Wk, const void *Wv, const float *x, float *q, float *k, float *v,
                       int n_q, int n_kv, int n_in, cudaStream_t s) {
  DlArgs a{};
  a.W = static_cast<const uint8_t *>(Wq);
  a.W2 = static_cast<const uint8_t *>(Wk);
  a.W3 = static_cast<const uint8_t *>(Wv);
  a.x = x;
  a.y = q;
  a.y2 = k;
  a.y3 = v;
  a.seg1 = n_q;
  a.seg2 = n_q + n_kv;
  a.n_out = n_q + 2 * n_kv;
  a.n_in = n_in;
  return launch_dl<kQ4, kQkv>(a, s);
}

}  // namespace qdq

// Batch-1 dequant-GEMV, direct-load form: the weights go from global memory
// straight into registers (no shared-memory staging, no producer warp).
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
// (one CTA per SM).  A warp handles 4 (virtual) rows per stage: each lane loads
// its block of the 4 rows with 128-bit loads into registers, multiplies, and a
// recursive-halving butterfly leaves row k's warp total in lane 8k; the slice
// totals of a row are added in fixed order at the end (deterministic results).
//
// Loads in flight: with DEPTH = 2 a warp holds two stages of registers and
// loads stage t + 2 as soon as it has used stage t, so a stage's loads are in
// flight during the previous stage's arithmetic (12 warps, about 160 registers
// a thread); DEPTH = 1 (rows of more than 12 slices) loads the next stage after
// the arithmetic of the current one.  The first stages are loaded before the
// wait for the previous kernel, and a bulk L2 prefetch of the CTA's rows is
// issued first when the call's weights fit in half the L2.
//
// Against the co-resident ring kernel (a producer warp streaming into a
// shared-memory ring sized to half an SM, so that the next kernel's CTA fits
// beside it, with 6-9 computing warps): here the whole SM computes and the
// registers of two stages keep the memory pipe busy.  A variant with per-warp
// bulk-copy rings in shared memory measured slower than this one (1 KB and
// 64-byte copies per row and warp).
//
// Arithmetic: f32 (weights converted exactly, packed f32x2 FMAs; Q4_K with the
// sub-block shift q4k_mu), within 1e-5 sum |w||x| for every finite input.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kMaxWarps = 16;
constexpr int kMaxWarpsDepth2 = 12;  // two stages of registers: about 160 a thread
enum Fmt { kQ8 = 0, kQ4 = 1, kQ6 = 2 };
enum Epi { kPlain = 0, kSwiglu = 1, kResidual = 2, kQkv = 3 };

struct DlArgs {
  const uint8_t *W, *W2, *W3;  // matrix (gate / W_q), up / W_k, W_v
  const float *x;
  const float *residual;
  float *y, *y2, *y3;          // output (q), k, v
  int seg1, seg2;              // QKV: rows [0, seg1) W_q, [seg1, seg2) W_k, [seg2, n_out) W_v
  int n_out, n_in, wpr, groups, prefetch;
  int psum_cap;  // floats of the row-total buffer in shared memory
};

// One lane's data of one row (its 32-weight block).
struct RowData {
  uint4 a, b;  // Q8_0: the 32 quants; Q4_K: a = 16 bytes of nibbles, b = the superblock header; Q6_K: a = low bits
  uint32_t c;  // Q8_0: d (fp16 bits); Q6_K: the two int8 scales
  uint2 h;     // Q6_K: high bits
  uint32_t d;  // Q6_K: d (fp16 bits)
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

template <int FMT, int EPI>
__device__ __forceinline__ RowData load_row(const DlArgs &a, int R, int up, int bq) {
  int lr, nm;
  const uint8_t *base = row_matrix<EPI>(a, R, up, lr, nm);
  const int n_in = a.n_in;
  const int64_t qr = q_row_bytes<FMT>(n_in), sr = s_row_bytes<FMT>(n_in);
  RowData d{};
  if (!QDQ_GUARD(lr >= 0 && lr < nm && bq >= 0 && bq < (n_in >> 5), QDQ_CHECK_ROW)) return d;
  if constexpr (FMT == kQ8) {
    const uint8_t *q = base + int64_t(lr) * qr + 32 * bq;
    d.a = ldg_stream(q);
    d.b = ldg_stream(q + 16);
    d.c = __ldg(reinterpret_cast<const unsigned short *>(base + int64_t(nm) * qr + int64_t(lr) * sr) + bq);
  } else if constexpr (FMT == kQ4) {
    d.a = ldg_stream(base + int64_t(lr) * qr + 16 * bq);
    d.b = __ldg(reinterpret_cast<const uint4 *>(base + int64_t(nm) * qr + int64_t(lr) * sr) + (bq >> 3));
  } else {
    const uint8_t *row = base + int64_t(lr) * qr;
    d.a = ldg_stream(row + 16 * bq);
    d.h = __ldg(reinterpret_cast<const uint2 *>(row + (n_in >> 1)) + bq);
    d.c = __ldg(reinterpret_cast<const unsigned short *>(row + (n_in >> 1) + (n_in >> 2)) + bq);
    d.d = __ldg(reinterpret_cast<const unsigned short *>(row + (n_in >> 1) + (n_in >> 2) + (n_in >> 4)) + (bq >> 3));
  }
  return d;
}

// The arithmetic of one stage (4 rows of this lane's block) -> part[k].
template <int FMT>
__device__ __forceinline__ void stage_math(const RowData (&rd)[4], const float2 (&xr)[16], float xsum, bool g0, bool g1,
                                           int sh, const Magic &mg, float (&part)[4]) {
    if constexpr (FMT == kQ8) {
      float2 s0[4], s1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) s0[k] = s1[k] = f2(0.f, 0.f);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 &u = kk < 4 ? rd[k].a : rd[k].b;
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
        part[k] = __half2float(__ushort_as_half(uint16_t(rd[k].c))) * (st.x + st.y);
      }
    } else if constexpr (FMT == kQ4) {
      float2 s0[4], s1[4], b01[4], b23[4];
      float D[4], R[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 h = rd[k].b;
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
          const uint4 &u = rd[k].a;
          const uint32_t w = kk == 0 ? u.x : kk == 1 ? u.y : kk == 2 ? u.z : u.w;
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
        const float d = __half2float(__ushort_as_half(uint16_t(rd[k].d)));
        const float ds0 = __fmul_rn(d, float(int8_t(rd[k].c & 0xFFu)));
        const float ds1 = __fmul_rn(d, float(int8_t((rd[k].c >> 8) & 0xFFu)));
        float2 v[16];
        q6k_block_to_f2(rd[k].a, rd[k].h, mg, v);
        float2 a0 = f2(0.f, 0.f), a1 = f2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 8; ++p) a0 = __ffma2_rn(v[p], xr[p], a0);
#pragma unroll
        for (int p = 8; p < 16; ++p) a1 = __ffma2_rn(v[p], xr[p], a1);
        part[k] = fmaf(ds1, a1.x + a1.y, ds0 * (a0.x + a0.y));
      }
    }
}

template <int FMT, int EPI, int DEPTH>
__global__ void __launch_bounds__(32 * (DEPTH == 2 ? kMaxWarpsDepth2 : kMaxWarps))
    gemv_dl_kernel(const DlArgs a, const Magic mg_param) {
  extern __shared__ float psum[];  // [local virtual row][wpr]
  constexpr int kV = EPI == kSwiglu ? 2 : 1;  // virtual rows per output row
  constexpr int kRowsPerStage = 4 / kV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_in = a.n_in, G = a.groups;
  const int slice = warp % a.wpr, grp = warp / a.wpr;
  const int r0 = int(int64_t(blockIdx.x) * a.n_out / gridDim.x);
  const int r1 = int(int64_t(blockIdx.x + 1) * a.n_out / gridDim.x);
  const int nreal = r1 - r0;
  const int gb = r0 + grp * nreal / G, ge = r0 + (grp + 1) * nreal / G;  // this group's output rows

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
  pdl_launch_dependents();

  const int nblk = n_in >> 5;
  const int blk = slice * 32 + lane;
  const bool valid = blk < nblk;
  const int bq = valid ? blk : 0;  // a lane past the end of the row reads block 0 against x = 0
  const Magic mg = lane_magic(mg_param);
  // virtual row k of the stage starting at output row rr; rows past the group's end
  // repeat its last row (in bounds) and are dropped
  auto vrow = [&](int rr, int k, int &up) {
    up = kV == 2 ? (k & 1) : 0;
    const int R = rr + (kV == 2 ? (k >> 1) : k);
    return R < ge ? R : ge - 1;
  };
  const int nst = ((ge - gb) * kV + 3) / 4;  // this group's stages of 4 virtual rows
  auto load_stage = [&](int t, RowData (&rd)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int up;
      const int R = vrow(gb + t * kRowsPerStage, k, up);
      rd[k] = load_row<FMT, EPI>(a, R, up, bq);
    }
  };
  RowData b0[4], b1[4];
  if (nst > 0) load_stage(0, b0);
  if (DEPTH == 2 && nst > 1) load_stage(1, b1);

  pdl_wait();  // the activations come from the previous kernel
  float2 xr[16];
  float xsum = 0.f;
  {
    const float4 *xp = reinterpret_cast<const float4 *>(a.x + bq * 32);
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

  // butterfly and store of stage t's row totals
  auto finish = [&](int t, float (&part)[4]) {
    butterfly4_rows(part, lane);
    if ((lane & 7) == 0) {
      const int v = (gb - r0) * kV + 4 * t + (lane >> 3);  // local virtual row
      if (v < (ge - r0) * kV && QDQ_GUARD(v * a.wpr + slice < a.psum_cap, QDQ_CHECK_SMEM))
        psum[v * a.wpr + slice] = part[0];
    }
  };
  if (DEPTH == 2) {
    for (int t = 0; t < nst; t += 2) {
      {
        float part[4];
        stage_math<FMT>(b0, xr, xsum, g0, g1, sh, mg, part);
        if (t + 2 < nst) load_stage(t + 2, b0);  // in flight during the next stage's arithmetic
        finish(t, part);
      }
      if (t + 1 < nst) {
        float part[4];
        stage_math<FMT>(b1, xr, xsum, g0, g1, sh, mg, part);
        if (t + 3 < nst) load_stage(t + 3, b1);
        finish(t + 1, part);
      }
    }
  } else {
    for (int t = 0; t < nst; ++t) {
      float part[4];
      stage_math<FMT>(b0, xr, xsum, g0, g1, sh, mg, part);
      if (t + 1 < nst) load_stage(t + 1, b0);  // the next stage's loads go out before this stage's reduction
      finish(t, part);
    }
  }
  __syncthreads();
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
}

template <int FMT, int EPI, int DEPTH>
int launch_dl_depth(DlArgs a, cudaStream_t s, const DeviceInfo &di) {
  constexpr int kV = EPI == kSwiglu ? 2 : 1;
  constexpr int kCap = DEPTH == 2 ? kMaxWarpsDepth2 : kMaxWarps;
  a.groups = opt_xs_groups() > 0 ? opt_xs_groups() : kCap / a.wpr;
  if (a.groups < 1) a.groups = 1;
  if (a.wpr * a.groups > kCap) return QDQ_ERR_UNSUPPORTED;
  int grid = di.sm_count * ctas_per_sm_or(1);
  if (grid > a.n_out) grid = a.n_out;
  const int max_rows = (a.n_out + grid - 1) / grid;
  const size_t smem = size_t(max_rows) * kV * a.wpr * sizeof(float);
  a.psum_cap = int(smem / sizeof(float));
  // L2 prefetch of the CTA's rows: on by default when this call's weights fit in half the L2
  const int64_t w_bytes = int64_t(a.n_out) * (FMT == kQ8 ? int64_t(a.n_in) / 32 * 34
                                              : FMT == kQ4 ? int64_t(a.n_in) / 256 * 144
                                                           : q6k_row_bytes(a.n_in)) * kV;
  const int pf = opt_l2_prefetch();
  a.prefetch = pf == 3 ? 0 : pf == 1 ? 1 : (w_bytes <= int64_t(di.l2_bytes) / 2 ? 1 : 0);
  auto kern = gemv_dl_kernel<FMT, EPI, DEPTH>;
  if (smem > 48 * 1024) {
    if (smem > size_t(di.max_smem_optin)) return QDQ_ERR_UNSUPPORTED;
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const cudaError_t e = launch(kern, dim3(grid), dim3(32 * a.wpr * a.groups), smem, s, a, make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

template <int FMT, int EPI>
int launch_dl(DlArgs a, cudaStream_t s) {
  DeviceInfo di;
  const cudaError_t e0 = device_info(&di);
  if (e0 != cudaSuccess) return fail_cuda(e0);
  a.wpr = ((a.n_in >> 5) + 31) / 32;
  if (a.wpr > kMaxWarps) return QDQ_ERR_UNSUPPORTED;
  // two stages of registers in flight unless a row needs more than 12 slice warps
  // (QDQ_OPT_XS_STAGES = 1 or 2 picks the depth)
  int depth = a.wpr <= kMaxWarpsDepth2 ? 2 : 1;
  if (opt_xs_stages() == 1 || opt_xs_stages() == 2) depth = opt_xs_stages();
  // more warps than two stages of registers allow (a wide row, or a forced group
  // count) run one stage deep
  const int warps = a.wpr * (opt_xs_groups() > 0 ? opt_xs_groups() : 1);
  if (warps > kMaxWarpsDepth2) depth = 1;
  return depth == 2 ? launch_dl_depth<FMT, EPI, 2>(a, s, di) : launch_dl_depth<FMT, EPI, 1>(a, s, di);
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

int read_dl_timeouts() { return 0; }  // the direct-load kernel has no waits
QDQ_CHECK_READER(read_checks_dl)

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

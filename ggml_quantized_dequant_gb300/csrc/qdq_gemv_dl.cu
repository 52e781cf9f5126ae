// Batch-1 dequant-GEMV, direct-load form: the weights go from global memory
// straight into registers (no shared-memory staging, no producer warp).
//
// "Module cuda_lane", Functions: try_q8_0_cuda_gemv (Q8_0 GEMV), try_q4k_soa_gemv
// (Q4_K GEMV), try_q4k_soa_fused_swiglu (out[i] = silu(gate_i . x) * (up_i . x)),
// try_q4k_soa_ffn_block_residual (out = residual + W_down . mid), try_q4k_soa_qkv
// (Q, K, V from one activation); "QTensorEngine", dispatch_gemm_into (Q6_K).
//
// Layout of the work is x-stationary: slice warp s owns the 1024 columns
// 1024 s .. 1024 s + 1023 for the whole kernel and each lane keeps its 32
// activations in registers.  Q4_K and Q6_K: lane l owns column block 32 s + l
// (its 16 bytes of low bits are contiguous with its neighbours').  Q8_0: lane l
// owns half l & 1 of blocks 32 s + (l >> 1) and 32 s + 16 + (l >> 1), so that
// each of its two 16-byte loads is one contiguous 512-byte span for the warp
// (a whole 32-byte block per lane would touch every sector twice).  WPR =
// ceil(n_in / 1024) slice warps cover a row.  Rows are dealt out in whole
// stages; by default a CTA is one group of slice warps, and as many CTAs as fit
// share an SM (QDQ_OPT_XS_GROUPS / QDQ_OPT_CTAS_PER_SM override both).  A warp
// handles 4 (virtual) rows per stage: each lane loads its part of the 4 rows
// with 128-bit loads into registers, multiplies, and a recursive-halving
// butterfly leaves row k's warp total in lane 8k; the slice totals of a row are
// added in fixed order at the end (deterministic results).
//
// Loads in flight: with DEPTH = 2 a warp holds two stages of registers and
// loads stage t + 2 as soon as it has used stage t, so a stage's loads are in
// flight during the previous stage's arithmetic (about 166 registers a thread:
// four 3-warp CTAs fill an SM); DEPTH = 1 (rows of more than 4 slices) loads the
// next stage after the arithmetic of the current one, at up to 128 registers, so
// that two 8-warp CTAs share an SM.  The first stages are loaded before the wait
// for the previous kernel.  Small CTAs are the point: the SM's CTAs finish at
// different times, and each one that finishes lets a CTA of the next kernel in
// the stream start its weight loads while the rest of this kernel completes
// (one SM-sized CTA per kernel measured 8.1 us per 3072 <-> 8192 Q8_0 matrix
// in the decode chain, the split shapes 6.9 us).
//
// A variant with per-warp bulk-copy rings in shared memory measured slower than
// registers (1 KB and 64-byte copies per row and warp), and so did a bulk L2
// prefetch of the CTA's rows at its start (QDQ_OPT_L2_PREFETCH = 1 still issues
// it).
//
// Arithmetic: f32 (weights converted exactly, packed f32x2 FMAs; Q4_K with the
// sub-block shift q4k_mu), within 1e-5 sum |w||x| for every finite input.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kMaxWarps = 16;
constexpr int kMaxWarpsDepth2 = 12;  // two stages of registers: about 160 a thread
enum Fmt { kQ8 = 0, kQ4 = 1, kQ6 = 2 };
enum Epi { kPlain = 0, kSwiglu = 1, kResidual = 2, kQkv = 3, kTopk = 4 };

struct DlArgs {
  const uint8_t *W, *W2, *W3;  // matrix (gate / W_q), up / W_k, W_v
  const float *x;
  const float *residual;
  float *y, *y2, *y3;          // output (q), k, v
  int seg1, seg2;              // QKV: rows [0, seg1) W_q, [seg1, seg2) W_k, [seg2, n_out) W_v
  int n_out, n_in, wpr, groups, prefetch;
  int psum_cap;  // floats of the row-total buffer in shared memory
  uint64_t *cand;  // kTopk: the k best keys of each CTA's rows, at cand[cta * k ...]
  int k;
  int key_off;     // kTopk: floats from the start of shared memory to the rows' keys (8-byte aligned)
  int fold_off;    // kTopk: ... to the warps' candidate lists (64 keys for each warp but the first)
};

// The columns one lane owns: Q4_K / Q6_K block `bq`; Q8_0 half `h` of blocks qa and qb.
struct LaneCols {
  int bq;            // Q4_K / Q6_K: the column block
  int qa, qb, h;     // Q8_0: the two blocks and the half (16 quants) of each
};

// One lane's data of one row.
struct RowData {
  uint4 a, b;  // Q8_0: the 16 quants of each half; Q4_K: a = 16 bytes of nibbles, b = the superblock header;
               // Q6_K: a = low bits
  uint32_t c;  // Q8_0: d of block qa (low half) and of block qb (high half), fp16 bits; Q6_K: the two int8 scales
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

// Per-lane pointers into one matrix, set once per kernel: the row-0 address of
// each piece of this lane's data, so that a row's address is one multiply-add
// (pointer + row * stride).  Q8_0: quants of half-blocks qa and qb, their two
// scales.  Q4_K: nibbles, superblock header.  Q6_K: low bits, high bits, scales, d.
struct LanePtrs {
  const uint8_t *p[4];
};

template <int FMT>
__device__ __forceinline__ LanePtrs lane_ptrs(const uint8_t *W, int nm, int n_in, const LaneCols &lc) {
  LanePtrs l;
  const int64_t qr = q_row_bytes<FMT>(n_in);
  if constexpr (FMT == kQ8) {
    const uint8_t *S = W + int64_t(nm) * qr;
    l.p[0] = W + 16 * lc.h + 32 * lc.qa;
    l.p[1] = W + 16 * lc.h + 32 * lc.qb;
    l.p[2] = S + 2 * lc.qa;
    l.p[3] = S + 2 * lc.qb;
  } else if constexpr (FMT == kQ4) {
    l.p[0] = W + 16 * lc.bq;
    l.p[1] = W + int64_t(nm) * qr + 16 * (lc.bq >> 3);
    l.p[2] = l.p[3] = nullptr;
  } else {
    l.p[0] = W + 16 * lc.bq;
    l.p[1] = W + (n_in >> 1) + 8 * lc.bq;
    l.p[2] = W + (n_in >> 1) + (n_in >> 2) + 2 * lc.bq;
    l.p[3] = W + (n_in >> 1) + (n_in >> 2) + (n_in >> 4) + 2 * (lc.bq >> 3);
  }
  return l;
}

// Loads this lane's data of local row lr of the matrix whose pointers are lp.
template <int FMT>
__device__ __forceinline__ RowData load_row(const LanePtrs &lp, int lr, int nm, int n_in) {
  const int64_t qr = q_row_bytes<FMT>(n_in), sr = s_row_bytes<FMT>(n_in);
  RowData d{};
  if (!QDQ_GUARD(lr >= 0 && lr < nm, QDQ_CHECK_ROW)) return d;
  if constexpr (FMT == kQ8) {
    d.a = ldg_stream(lp.p[0] + lr * qr);
    d.b = ldg_stream(lp.p[1] + lr * qr);
    d.c = uint32_t(__ldg(reinterpret_cast<const unsigned short *>(lp.p[2] + lr * sr))) |
          (uint32_t(__ldg(reinterpret_cast<const unsigned short *>(lp.p[3] + lr * sr))) << 16);
  } else if constexpr (FMT == kQ4) {
    d.a = ldg_stream(lp.p[0] + lr * qr);
    d.b = __ldg(reinterpret_cast<const uint4 *>(lp.p[1] + lr * sr));
  } else {
    d.a = ldg_stream(lp.p[0] + lr * qr);
    d.h = __ldg(reinterpret_cast<const uint2 *>(lp.p[1] + lr * qr));
    d.c = __ldg(reinterpret_cast<const unsigned short *>(lp.p[2] + lr * qr));
    d.d = __ldg(reinterpret_cast<const unsigned short *>(lp.p[3] + lr * qr));
  }
  return d;
}

// The arithmetic of one stage (4 rows of this lane's block) -> part[k].
template <int FMT>
__device__ __forceinline__ void stage_math(const RowData (&rd)[4], const float2 (&xr)[16], float xsum, bool g0, bool g1,
                                           int sh, const Magic &mg, float (&part)[4]) {
    if constexpr (FMT == kQ8) {
      float2 sa[4], sb[4];  // the two half blocks: xr[0..7] and xr[8..15]
#pragma unroll
      for (int k = 0; k < 4; ++k) sa[k] = sb[k] = f2(0.f, 0.f);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 &u = rd[k].a, &v = rd[k].b;
          const uint32_t wa = kk == 0 ? u.x : kk == 1 ? u.y : kk == 2 ? u.z : u.w;
          const uint32_t wb = kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
          float2 q01, q23;
          s8x4_to_f2(wa, mg, q01, q23);
          sa[k] = __ffma2_rn(q01, xr[2 * kk], sa[k]);
          sa[k] = __ffma2_rn(q23, xr[2 * kk + 1], sa[k]);
          s8x4_to_f2(wb, mg, q01, q23);
          sb[k] = __ffma2_rn(q01, xr[8 + 2 * kk], sb[k]);
          sb[k] = __ffma2_rn(q23, xr[8 + 2 * kk + 1], sb[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float da = __half2float(__ushort_as_half(uint16_t(rd[k].c & 0xFFFFu)));
        const float db = __half2float(__ushort_as_half(uint16_t(rd[k].c >> 16)));
        part[k] = fmaf(db, sb[k].x + sb[k].y, da * (sa[k].x + sa[k].y));
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
  // rows are dealt out in units of one stage (kRowsPerStage output rows), so that
  // only the matrix's last stage can be partial: units [u0, u1) to this CTA, and
  // a contiguous share of them to each group
  const int units = (a.n_out + kRowsPerStage - 1) / kRowsPerStage;
  const int u0 = int(int64_t(blockIdx.x) * units / gridDim.x), u1 = int(int64_t(blockIdx.x + 1) * units / gridDim.x);
  const int r0 = u0 * kRowsPerStage, r1 = min(u1 * kRowsPerStage, a.n_out);
  const int nreal = r1 - r0;
  const int gu0 = u0 + grp * (u1 - u0) / G, gu1 = u0 + (grp + 1) * (u1 - u0) / G;
  const int gb = gu0 * kRowsPerStage, ge = min(gu1 * kRowsPerStage, a.n_out);  // this group's output rows

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
  // this lane's columns; a block past the end of the row reads block 0 against x = 0
  LaneCols lc;
  int xo0, xo1;        // the lane's two runs of 16 activations
  bool valid0, valid1;
  if (FMT == kQ8) {
    const int qa = 32 * slice + (lane >> 1), qb = qa + 16;
    valid0 = qa < nblk;
    valid1 = qb < nblk;
    lc.h = lane & 1;
    lc.qa = valid0 ? qa : 0;
    lc.qb = valid1 ? qb : 0;
    lc.bq = 0;
    xo0 = 32 * lc.qa + 16 * lc.h;
    xo1 = 32 * lc.qb + 16 * lc.h;
  } else {
    const int blk = slice * 32 + lane;
    valid0 = valid1 = blk < nblk;
    lc.bq = valid0 ? blk : 0;
    lc.qa = lc.qb = lc.h = 0;
    xo0 = 32 * lc.bq;
    xo1 = xo0 + 16;
  }
  const Magic mg = lane_magic(mg_param);
  // the lane's pointers into each matrix (QKV: W_q, W_k, W_v; SwiGLU: gate, up)
  constexpr int kM = EPI == kQkv ? 3 : kV;
  LanePtrs lp[kM];
  int nmat[kM];
  if (EPI == kQkv) {
    nmat[0] = a.seg1;
    nmat[1 % kM] = a.seg2 - a.seg1;
    nmat[2 % kM] = a.n_out - a.seg2;
    lp[0] = lane_ptrs<FMT>(a.W, nmat[0], n_in, lc);
    lp[1 % kM] = lane_ptrs<FMT>(a.W2, nmat[1 % kM], n_in, lc);
    lp[2 % kM] = lane_ptrs<FMT>(a.W3, nmat[2 % kM], n_in, lc);
  } else {
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      nmat[m] = a.n_out;
      lp[m] = lane_ptrs<FMT>(m ? a.W2 : a.W, a.n_out, n_in, lc);
    }
  }
  const int nst = gu1 - gu0;  // this group's stages
  // stage t: output rows gb + kRowsPerStage t + i; a row past the group's end (only
  // in the matrix's last stage) repeats the group's last row and is dropped
  auto load_stage = [&](int t, RowData (&rd)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int up = kV == 2 ? (k & 1) : 0;
      int R = gb + t * kRowsPerStage + (kV == 2 ? (k >> 1) : k);
      R = R < ge ? R : ge - 1;
      if (EPI == kQkv) {
        const bool m0 = R < a.seg1, m1 = !m0 && R < a.seg2;
        const int lr = m0 ? R : m1 ? R - a.seg1 : R - a.seg2;
        const int nm = m0 ? nmat[0] : m1 ? nmat[1 % kM] : nmat[2 % kM];
        LanePtrs l;
#pragma unroll
        for (int i = 0; i < 4; ++i) l.p[i] = m0 ? lp[0].p[i] : m1 ? lp[1 % kM].p[i] : lp[2 % kM].p[i];
        rd[k] = load_row<FMT>(l, lr, nm, n_in);
      } else {
        rd[k] = load_row<FMT>(lp[up], R, nmat[up], n_in);
      }
    }
  };
  RowData b0[4], b1[4];
  if (nst > 0) load_stage(0, b0);
  if (DEPTH == 2 && nst > 1) load_stage(1, b1);

  pdl_wait();  // the activations come from the previous kernel
  float2 xr[16];
  float xsum = 0.f;
  {
    const float4 *xp0 = reinterpret_cast<const float4 *>(a.x + xo0);
    const float4 *xp1 = reinterpret_cast<const float4 *>(a.x + xo1);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const bool ok = c < 4 ? valid0 : valid1;
      const float4 v = ok ? ld_after_wait(c < 4 ? xp0 + c : xp1 + (c - 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
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
      if (EPI == kTopk) reinterpret_cast<uint64_t *>(psum + a.key_off)[r] = topk_key(v, uint32_t(R));
    }
  }
  if constexpr (EPI == kTopk) {
    // the k best keys of this CTA's rows: warp w keeps a running top 64 over chunks w,
    // w + warps, ... of 64 keys; warp 0 then merges the other warps' lists
    __syncthreads();
    const int nw = int(blockDim.x >> 5);
    const uint64_t *keys = reinterpret_cast<const uint64_t *>(psum + a.key_off);
    uint64_t *fold = reinterpret_cast<uint64_t *>(psum + a.fold_off);
    uint64_t ta = 0, tb = 0;
    for (int c0 = 64 * warp; c0 < nreal; c0 += 64 * nw) {
      uint64_t ka = c0 + lane < nreal ? keys[c0 + lane] : 0ull;
      uint64_t kb = c0 + 32 + lane < nreal ? keys[c0 + 32 + lane] : 0ull;
      warp_sort64_desc(ka, kb, lane);
      warp_top64_merge(ta, tb, ka, kb, lane);
    }
    if (warp > 0) {
      fold[(warp - 1) * 64 + lane] = ta;
      fold[(warp - 1) * 64 + lane + 32] = tb;
    }
    __syncthreads();
    if (warp == 0) {
      for (int w = 1; w < nw && 64 * w < nreal; ++w)
        warp_top64_merge(ta, tb, fold[(w - 1) * 64 + lane], fold[(w - 1) * 64 + lane + 32], lane);
      uint64_t *o = a.cand + int64_t(blockIdx.x) * a.k;
      if (lane < a.k) o[lane] = ta;
      if (lane + 32 < a.k) o[lane + 32] = tb;
    }
  }
}

template <int FMT, int EPI, int DEPTH>
int launch_dl_depth(DlArgs a, cudaStream_t s, const DeviceInfo &di, int *grid_out) {
  constexpr int kV = EPI == kSwiglu ? 2 : 1;
  constexpr int kCap = DEPTH == 2 ? kMaxWarpsDepth2 : kMaxWarps;
  // default: one group of slice warps per CTA, and as many CTAs per SM as fit, so
  // that a CTA that finishes early frees room for the next kernel's CTA (its
  // weight loads then overlap this kernel's tail)
  a.groups = opt_xs_groups() > 0 ? opt_xs_groups() : 1;
  if (a.wpr * a.groups > kCap) return QDQ_ERR_UNSUPPORTED;
  const int threads = 32 * a.wpr * a.groups;
  constexpr int kRowsPerStage = 4 / kV;
  const int units = (a.n_out + kRowsPerStage - 1) / kRowsPerStage;
  auto kern = gemv_dl_kernel<FMT, EPI, DEPTH>;
  auto psum_bytes = [&](int grid) { return size_t((units + grid - 1) / grid * kRowsPerStage) * kV * a.wpr * 4; };
  // kTopk: the rows' keys after the row totals (8-byte aligned), then the warps' lists
  auto smem_bytes = [&](int grid) {
    const size_t p = psum_bytes(grid);
    return EPI == kTopk ? (p + 7) / 8 * 8 + size_t((units + grid - 1) / grid * kRowsPerStage) * 8 +
                              size_t(threads / 32 - 1) * 64 * 8
                        : p;
  };
  int per_sm = ctas_per_sm_or(0);
  if (per_sm == 0) {
    // shared memory of the largest CTA share at one CTA per SM bounds every other shape's
    const size_t smem0 = smem_bytes(units < di.sm_count ? units : di.sm_count);
    if (smem0 > 48 * 1024) {
      if (smem0 > size_t(di.max_smem_optin)) return QDQ_ERR_UNSUPPORTED;
      const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem0));
      if (e != cudaSuccess) return fail_cuda(e);
    }
    int nb = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, threads, smem0);
    if (e != cudaSuccess) return fail_cuda(e);
    per_sm = nb < 1 ? 1 : nb > 16 ? 16 : nb;
  }
  int grid = di.sm_count * per_sm;
  if (grid > units) grid = units;
  const size_t smem = smem_bytes(grid);
  a.psum_cap = int(psum_bytes(grid) / sizeof(float));
  a.key_off = int((psum_bytes(grid) + 7) / 8 * 2);
  a.fold_off = a.key_off + (units + grid - 1) / grid * kRowsPerStage * 2;
  if (grid_out) *grid_out = grid;
  // L2 prefetch of the CTA's rows: off unless QDQ_OPT_L2_PREFETCH = 1 (measured no faster here)
  a.prefetch = opt_l2_prefetch() == 1 ? 1 : 0;
  if (smem > 48 * 1024) {
    if (smem > size_t(di.max_smem_optin)) return QDQ_ERR_UNSUPPORTED;
    const cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const cudaError_t e = launch(kern, dim3(grid), dim3(threads), smem, s, a, make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

template <int FMT, int EPI>
int launch_dl(DlArgs a, cudaStream_t s, int *grid_out = nullptr) {
  DeviceInfo di;
  const cudaError_t e0 = device_info(&di);
  if (e0 != cudaSuccess) return fail_cuda(e0);
  a.wpr = ((a.n_in >> 5) + 31) / 32;
  if (a.wpr > kMaxWarps) return QDQ_ERR_UNSUPPORTED;
  // two stages of registers in flight for rows of up to 4 slice warps (several
  // such CTAs share an SM); wider rows run one stage deep, which lets two of
  // their CTAs share an SM (QDQ_OPT_XS_STAGES = 1 or 2 picks the depth)
  int depth = a.wpr <= 4 ? 2 : 1;
  if (opt_xs_stages() == 1 || opt_xs_stages() == 2) depth = opt_xs_stages();
  // more warps than two stages of registers allow (a forced group count) run one stage deep
  const int warps = a.wpr * (opt_xs_groups() > 0 ? opt_xs_groups() : 1);
  if (warps > kMaxWarpsDepth2) depth = 1;
  return depth == 2 ? launch_dl_depth<FMT, EPI, 2>(a, s, di, grid_out)
                    : launch_dl_depth<FMT, EPI, 1>(a, s, di, grid_out);
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

int launch_gemv_dl_topk(const void *W, const float *x, float *y, int n_out, int n_in, uint64_t *cand, int k,
                        int *n_cand, cudaStream_t s) {
  DlArgs a{};
  a.W = static_cast<const uint8_t *>(W);
  a.x = x;
  a.y = y;
  a.n_out = n_out;
  a.n_in = n_in;
  a.cand = cand;
  a.k = k;
  int grid = 0;
  const int rc = launch_dl<kQ8, kTopk>(a, s, &grid);
  *n_cand = grid * k;
  return rc;
}

int gemv_dl_max_ctas() {
  DeviceInfo di;
  return device_info(&di) == cudaSuccess ? di.sm_count * 16 : 0;
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

// Batch-1 dequant-GEMV fast path: "x-stationary" consumers fed by a bulk-copy
// weight pipeline in shared memory.
//
// "Module cuda_lane", Functions: try_q8_0_cuda_gemv / q8_0_gemv_oracle_into
// (Q8_0 GEMV), try_q4k_soa_gemv (Q4_K GEMV), try_q4k_soa_fused_swiglu
// (out[i] = silu(gate_i . x) * (up_i . x)), try_q4k_soa_ffn_block_residual
// (out = residual + W_down . mid).  Token decode multiplies one activation
// vector by every weight matrix, so this is the path the decode loop takes.
//
// Layout of the work:
//  * a row of n_in weights is cut into nblk = n_in / 32 column blocks (one Q8_0
//    block, or one Q4_K sub-block); lane l of "slice" warp s owns block
//    32 s + l for the whole kernel and keeps its 32 activations in registers,
//    so WPR = ceil(nblk / 32) slice warps cover a row and x never goes through
//    shared memory;
//  * a CTA owns a contiguous range of output rows (one CTA per SM).  A
//    producer warp streams them in stages of 4 rows -- quant bytes and scale
//    (Q8_0 d) or header (Q4_K) bytes, each a contiguous range of its plane --
//    with 1-D bulk async copies into a ring of stages in shared memory.  The
//    weights do not depend on the previous kernel, so the ring is filled
//    before the previous kernel has finished (programmatic dependent launch);
//  * the slice warps form G groups; group g owns a contiguous share of the
//    CTA's rows and consumes its stages, in order, from its own ring slots.
//    For each stage a lane reads its block of the 4 rows, and a
//    recursive-halving butterfly reduces the 4 per-lane partial sums across the
//    warp (lane 8k ends with row k's warp total).  The WPR slice totals of a
//    row are added in fixed order at the end, so results are deterministic.
// SwiGLU streams gate and up rows as pairs (a stage = 2 output rows, each
// with its gate row and its up row) and combines them in the epilogue.
// The fused QKV projection ("Module cuda_lane", try_q4k_soa_qkv) runs the rows
// of W_q, then W_k, then W_v as one row range against the one x; a stage that
// crosses from one matrix into the next is copied in pieces, and the epilogue
// writes each row to q, k or v.
//
// Arithmetic (QDQ_OPT_XS_FLOAT_X).  By default the weights are converted
// exactly to f32 (magic-number LOP3s, one packed subtraction per pair) and
// multiplied with packed f32x2 FMAs against the f32 activations: every
// product's error is relative to |w_j x_j| itself, so a row is within
// 1e-5 sum |w||x| for every finite input.  Q4_K sums its quants shifted by the
// sub-block's integer offset mu (q4k_mu) and applies d sc and the remainder R
// once per sub-block: d sc sum (q - mu) x - R sum x.
// The opt-in fixed-point arithmetic keeps the weights integers instead: a lane
// turns its 32 activations once into 24-bit block fixed point
// X_j = rint(x_j 2^e) (e from the block's largest |x|, |X_j| <= 2^22), split
// into three int8 limbs, and a row's block dot product sum_j q_j X_j is three
// exact dp4a byte dot products per 4 weights, scaled in f32 ((d / 2^e) sum q X,
// and for Q4_K (d sc sum (q - mu) X - R sum X) / 2^e, the shift applied to the
// exact integer sums).  Its approximation beyond f32 rounding is
// |x_j - X_j 2^-e| <= 2^-22 max_block |x|, so
//   |y - exact| <= 2^-22 sum_b max_{j in b} |x_j| sum_{j in b} |w_j| + f32 rounding,
// which is within 1e-5 sum |w||x| unless a row's weights concentrate on the
// small activations of blocks whose largest activation they skip: a bound
// relative to each block's largest activation, not to each product, so it is
// not the default.  A block holding an inf or a NaN gives NaN rows on the
// fixed path (the f32 path propagates them by IEEE rules).
// Every pipeline wait is bounded; a wait that runs out is counted
// (qdq_pipeline_timeouts) and the CTA winds down instead of hanging.
#include <mutex>
#include <vector>

#include "qdq_internal.cuh"

namespace qdq {

__device__ unsigned int g_xs_timeouts = 0;

namespace {

constexpr int kStageRows = 4;    // virtual rows per stage = butterfly width
constexpr int kMaxThreads = 544;  // up to 16 consumer warps + the producer

enum Fmt { kQ8 = 0, kQ4 = 1, kQ6 = 2 };
enum Epi { kPlain = 0, kSwiglu = 1, kResidual = 2, kQkv = 3 };
enum Arith { kFixedX = 0, kFloatX = 1 };

// Four-way byte dot products: c + sum_i a.byte[i] * b.byte[i], the bytes of a
// and b read as signed (s) or unsigned (u).
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One lane's 32 activations in block fixed point (see Arithmetic above):
// X_j = rint(x_j 2^e), e = 148 - (biased exponent of max_j |x_j|), so
// 2^21 <= max|X| <= 2^22 for a normal maximum.  X_j = L2 2^16 + L1 2^8 + L0
// with L0, L1 the unsigned bytes 0, 1 of X_j and L2 = X_j >> 16 in [-64, 64].
// p[l][w] packs limb l of the four activations that weight word w multiplies:
// Q8_0 word w holds weights 4w..4w+3; Q4_K word c holds nibbles 8c..8c+7 and is
// split into its even nibbles (packed word 2c) and odd nibbles (word 2c + 1).
struct FixedX {
  uint32_t p[3][8];
  float inv_s;  // 2^-e (NaN when the block holds an inf or a NaN)
  float xsum;   // sum_j X_j (Q4_K)
  int s01;      // sum_j (L1_j 2^8 + L0_j) = sum_j (X_j & 0xFFFF) (Q4_K)
  int s2;       // sum_j L2_j (Q4_K)
};

template <int FMT>
__device__ __forceinline__ void to_fixed(const float (&xv)[32], FixedX &f) {
  // max |x| as the largest bit pattern with the sign cleared (inf and NaN patterns
  // are the largest of all), reduced as a tree
  uint32_t mb[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    mb[j] = max(__float_as_uint(xv[2 * j]) & 0x7fffffffu, __float_as_uint(xv[2 * j + 1]) & 0x7fffffffu);
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) mb[j] = max(mb[j], mb[j + w]);
  const int E = int(mb[0] >> 23);
  if (E >= 255) {
#pragma unroll
    for (int l = 0; l < 3; ++l)
#pragma unroll
      for (int w = 0; w < 8; ++w) f.p[l][w] = 0u;
    f.inv_s = __int_as_float(0x7fffffff);
    f.xsum = 0.f;
    f.s01 = f.s2 = 0;
    return;
  }
  const int e = 148 - (E > 1 ? E : 1);  // -106 .. 147; a zero or subnormal maximum takes E = 1
  // 2^e as two normal factors; x * 2^(e>>1) is exact wherever the product can round to X != 0
  const float s1 = __int_as_float(((e >> 1) + 127) << 23);
  const float s2 = __int_as_float((e - (e >> 1) + 127) << 23);
  f.inv_s = e <= 126 ? __int_as_float((127 - e) << 23) : __int_as_float(1 << (149 - e));
  int X[32];
#pragma unroll
  for (int j = 0; j < 32; ++j)  // |x 2^e| < 2^22: adding 1.5 * 2^23 rounds it to an integer in the low mantissa bits
    X[j] = __float_as_int(__fmaf_rn(__fmul_rn(xv[j], s1), s2, 12582912.0f)) - 0x4B400000;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    int i[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) i[b] = FMT == kQ8 ? 4 * w + b : 8 * (w >> 1) + 2 * b + (w & 1);
    const uint32_t t0 = __byte_perm(X[i[0]], X[i[1]], 0x5140);  // b0 b0' b1 b1' of elements 0, 1
    const uint32_t t1 = __byte_perm(X[i[2]], X[i[3]], 0x5140);
    f.p[0][w] = __byte_perm(t0, t1, 0x5410);
    f.p[1][w] = __byte_perm(t0, t1, 0x7632);
    const uint32_t u0 = __byte_perm(X[i[0]], X[i[1]], 0x0062);  // b2 b2' of elements 0, 1
    const uint32_t u1 = __byte_perm(X[i[2]], X[i[3]], 0x0062);
    f.p[2][w] = __byte_perm(u0, u1, 0x5410);
  }
  if constexpr (FMT == kQ4) {
    int t[16], lo[16], hi[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      t[j] = X[2 * j] + X[2 * j + 1];
      lo[j] = (X[2 * j] & 0xFFFF) + (X[2 * j + 1] & 0xFFFF);
      hi[j] = (X[2 * j] >> 16) + (X[2 * j + 1] >> 16);
    }
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
      for (int j = 0; j < w; ++j) {
        t[j] += t[j + w];
        lo[j] += lo[j + w];
        hi[j] += hi[j + w];
      }
    f.xsum = __int2float_rn(t[0]);
    f.s01 = lo[0];
    f.s2 = hi[0];
  } else {
    f.xsum = 0.f;
    f.s01 = f.s2 = 0;
  }
}

// Reduce v[0..3] (one partial per row per lane) over the warp; afterwards lane
// 8k holds the warp total of row k.
__device__ __forceinline__ void butterfly4(float v[kStageRows], int lane) {
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = up ? v[i] : v[i + 2];
      const float keep = up ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool up = lane & 8;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 4);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
}

struct XsArgs {
  const uint8_t *W;   // packed matrix (gate for SwiGLU, W_q for QKV)
  const uint8_t *W2;  // up matrix (SwiGLU), W_k (QKV)
  const uint8_t *W3;  // W_v (QKV)
  const float *x;
  const float *residual;
  float *y;           // output (q for QKV)
  float *y2, *y3;     // k, v (QKV)
  int seg1, seg2;     // QKV: rows [0, seg1) are W_q's, [seg1, seg2) W_k's, [seg2, n_out) W_v's
  int n_out;        // output rows
  int n_in;
  int wpr;          // slice warps per row
  int groups;       // consumer groups per CTA
  int sg;           // ring slots per consumer group (the ring holds groups * sg stages)
  int stage_bytes;  // bytes per ring stage (multiple of 128)
  int l2_prefetch;
  int psum_cap;     // floats of the row-total buffer in shared memory
};

template <int FMT, int EPI, int AR>
__global__ void __launch_bounds__(kMaxThreads) gemv_xs_kernel(const XsArgs a, const Magic mg_param) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kV = EPI == kSwiglu ? 2 : 1;  // virtual rows per output row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncw = a.wpr * a.groups;  // consumer warps; warp ncw is the producer
  const int n_in = a.n_in;
  const int G = a.groups, SG = a.sg, S = G * SG;  // slots: group g owns g*SG .. g*SG+SG-1

  const int r0 = int(int64_t(blockIdx.x) * a.n_out / gridDim.x);
  const int r1 = int(int64_t(blockIdx.x + 1) * a.n_out / gridDim.x);
  const int nreal = r1 - r0;
  // Group g owns the output rows [gbeg(g), gbeg(g + 1)) of this CTA, so the groups
  // finish together (a partial last stage per group, not a whole stage of imbalance).
  auto gbeg = [&](int g) { return r0 + g * nreal / G; };
  auto gstages = [&](int g) { return ((gbeg(g + 1) - gbeg(g)) * kV + kStageRows - 1) / kStageRows; };
  constexpr int kRowsPerStage = kStageRows / kV;

  // quant bytes and scale/header bytes per row (Q6_K: the whole padded row, one plane)
  const int64_t q_row = FMT == kQ8 ? int64_t(n_in) : FMT == kQ4 ? int64_t(n_in >> 1) : q6k_row_bytes(n_in);
  const int64_t s_row = FMT == kQ8 ? int64_t(n_in >> 4) : FMT == kQ4 ? int64_t(n_in >> 8) * 16 : 0;
  const int64_t q_bytes = int64_t(a.n_out) * q_row;

  uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(S) * a.stage_bytes);
  uint64_t *empty = full + S;
  float *psum = reinterpret_cast<float *>(empty + S);  // [virtual rows][wpr]
  __shared__ int s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], a.wpr);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();

  // producer bookkeeping for the final drain: stages issued so far
  int rounds = 0, stop_i = 0, stop_g = 0;
  if (warp == ncw) {
    // ---------------- producer: weights only, so no wait on the previous kernel ----------------
    // Round i issues stage i of every group that has one.  Group g consumes its
    // stages in order from its own slots g*SG + i % SG; a slot is refilled only
    // after that group released it, so no wait can ever see a phase that is two
    // fills old.
    if (lane == 0) {
      if (EPI != kQkv && a.l2_prefetch == 1) {
        prefetch_range_l2(a.W, q_bytes, r0 * q_row, r1 * q_row);
        prefetch_range_l2(a.W + q_bytes, int64_t(a.n_out) * s_row, r0 * s_row, r1 * s_row);
        if (EPI == kSwiglu) {
          prefetch_range_l2(a.W2, q_bytes, r0 * q_row, r1 * q_row);
          prefetch_range_l2(a.W2 + q_bytes, int64_t(a.n_out) * s_row, r0 * s_row, r1 * s_row);
        }
      }
      for (int g = 0; g < G; ++g) rounds = max(rounds, gstages(g));
      stop_i = rounds;  // first stage not issued (stop_i, stop_g), if the loop stopped early
      for (int i = 0; i < rounds && stop_i == rounds; ++i) {
        if (EPI != kQkv && i == SG && a.l2_prefetch == 2) {
          // after the first fill of every slot: pull the rows that did not fit the ring
          // into L2, so that their refills do not wait on HBM
          for (int g = 0; g < G; ++g) {
            const int lo = min(gbeg(g) + SG * kRowsPerStage, gbeg(g + 1)), hi = gbeg(g + 1);
            if (lo >= hi) continue;
            prefetch_range_l2(a.W, q_bytes, lo * q_row, hi * q_row);
            prefetch_range_l2(a.W + q_bytes, int64_t(a.n_out) * s_row, lo * s_row, hi * s_row);
            if (EPI == kSwiglu) {
              prefetch_range_l2(a.W2, q_bytes, lo * q_row, hi * q_row);
              prefetch_range_l2(a.W2 + q_bytes, int64_t(a.n_out) * s_row, lo * s_row, hi * s_row);
            }
          }
        }
        for (int g = 0; g < G; ++g) {
          if (i >= gstages(g)) continue;
          const int s = g * SG + i % SG;
          // after any timed-out wait in this CTA, issue nothing more
          if (*reinterpret_cast<volatile int *>(&s_abort) ||
              (i >= SG && !mbar_wait(&empty[s], ((i / SG) + 1) & 1))) {
            s_abort = 1;
            stop_i = i;
            stop_g = g;
            break;
          }
          uint8_t *stq = smem + size_t(s) * a.stage_bytes;
          uint8_t *sts = stq + kStageRows * q_row;
          const int rr = gbeg(g) + i * kRowsPerStage;           // first output row of the stage
          const int nr = min(kRowsPerStage, gbeg(g + 1) - rr);  // output rows in the stage
          mbar_arrive_expect_tx(&full[s], uint32_t(kV * nr * (q_row + s_row)));
          if constexpr (EPI == kQkv) {
            // rows [rr, rr + nr) of W_q | W_k | W_v, one piece per matrix they touch
            const uint8_t *Wm[3] = {a.W, a.W2, a.W3};
            const int off[4] = {0, a.seg1, a.seg2, a.n_out};
#pragma unroll
            for (int m = 0; m < 3; ++m) {
              const int lo = max(rr, off[m]), hi = min(rr + nr, off[m + 1]);
              if (lo >= hi) continue;
              const int64_t qb = int64_t(off[m + 1] - off[m]) * q_row;  // this matrix's quant plane
              bulk_copy_g2s(stq + (lo - rr) * q_row, Wm[m] + (lo - off[m]) * q_row, uint32_t((hi - lo) * q_row),
                            &full[s]);
              bulk_copy_g2s(sts + (lo - rr) * s_row, Wm[m] + qb + (lo - off[m]) * s_row,
                            uint32_t((hi - lo) * s_row), &full[s]);
            }
          } else {
            bulk_copy_g2s(stq, a.W + rr * q_row, uint32_t(nr * q_row), &full[s]);
            if (FMT != kQ6) bulk_copy_g2s(sts, a.W + q_bytes + rr * s_row, uint32_t(nr * s_row), &full[s]);
          }
          if (EPI == kSwiglu) {  // up rows go to slots 2, 3
            bulk_copy_g2s(stq + 2 * q_row, a.W2 + rr * q_row, uint32_t(nr * q_row), &full[s]);
            bulk_copy_g2s(sts + 2 * s_row, a.W2 + q_bytes + rr * s_row, uint32_t(nr * s_row), &full[s]);
          }
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    const int slice = warp % a.wpr, grp = warp / a.wpr;
    const int blk = slice * 32 + lane;
    const bool valid = blk < (n_in >> 5);
    const Magic mg = lane_magic(mg_param);
    // Activations come from the previous kernel.  One warp waits for it; the
    // others sleep on a named barrier instead of polling beside the CTA that
    // is still computing on this SM.  The second wait returns at once and
    // gives every consumer thread the dependency's memory visibility.
    if (warp == 0) pdl_wait();
    named_bar_sync(1, 32 * ncw);
    pdl_wait();
    float2 xr[16];  // f32 path: activation pairs, aligned register pairs for the packed FMAs
    float xsum = 0.f;
    FixedX fx;      // fixed path
    {
      float xv[32];
      if (valid) {
        const float4 *xp = reinterpret_cast<const float4 *>(a.x + blk * 32);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v = ld_after_wait(xp + c);  // x comes from the previous kernel
          xv[4 * c] = v.x;
          xv[4 * c + 1] = v.y;
          xv[4 * c + 2] = v.z;
          xv[4 * c + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) xv[k] = 0.f;
      }
      if constexpr (AR == kFixedX) {
        to_fixed<FMT>(xv, fx);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) xr[c] = f2(xv[2 * c], xv[2 * c + 1]);
        if constexpr (FMT == kQ4) {
          float2 t = f2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 16; ++c) t = __fadd2_rn(t, xr[c]);
          xsum = t.x + t.y;
        }
      }
    }
    // Q4_K: this lane's 12-bit (sc, m) field lives at bit 12 j of header words 1..3
    const int j = lane & 7;
    const bool g0 = j < 3, g1 = j < 6;
    const int sh = (12 * j) & 31;
    // a lane past the end of the row reads block 0 (finite data) against x = 0
    const int bq = valid ? blk : 0;
    const int qoff = FMT == kQ8 ? bq * 32 : bq * 16;
    const int soff = FMT == kQ8 ? bq * 2 : FMT == kQ4 ? (bq >> 3) * 16 : 0;
    // Q6_K: this lane's high-bit, scale and d bytes within the packed row
    const int q6_hi = (n_in >> 1) + 8 * bq, q6_sc = (n_in >> 1) + (n_in >> 2) + 2 * bq;
    const int q6_d = (n_in >> 1) + (n_in >> 2) + (n_in >> 4) + 2 * (bq >> 3);
    // byte offsets of this lane's data for the 4 rows of a stage (the same in every stage);
    // SwiGLU: virtual rows gate r, up r, gate r+1, up r+1 sit in slots 0, 2, 1, 3
    int qofs[kStageRows], sofs[kStageRows];
#pragma unroll
    for (int k = 0; k < kStageRows; ++k) {
      const int slot = EPI == kSwiglu ? ((k & 1) << 1) | (k >> 1) : k;
      qofs[k] = int(slot * q_row) + qoff;
      sofs[k] = int(kStageRows * q_row + slot * s_row) + soff;
    }

    const int rbeg = gbeg(grp) - r0;                 // this group's first local output row
    const int vend = (gbeg(grp + 1) - r0) * kV;      // end of its virtual rows
    const int nst = gstages(grp);
    int s = grp * SG;      // this group's current slot and the parity of its fill:
    uint32_t parity = 0;   // tracked incrementally (no division in the loop)
    for (int t = 0; t < nst; ++t) {
      if (!mbar_wait(&full[s], parity)) {
        s_abort = 1;
        break;
      }
      const uint8_t *stq = smem + size_t(s) * a.stage_bytes;
      // Q4_K GEMV / down projection: the slot is released as soon as the stage's bytes
      // are in registers (the arrive is a release, so the reads are ordered before the
      // refill) and the producer refills it while this warp computes.  Measured on
      // 3072 <-> 8192 chains, that helps there but slows the SwiGLU and the Q8_0 GEMV,
      // which release after their arithmetic.
      constexpr bool kEarlyRelease = (FMT == kQ4 || FMT == kQ6) && EPI != kSwiglu;
      auto release = [&](int slot) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      };
      float part[kStageRows];
      // All four rows' loads first, then their arithmetic interleaved word by word:
      // eight independent accumulation chains per lane.  Rows past the end of the
      // last stage compute from stale shared memory and are dropped; the butterfly
      // never mixes rows, so they cannot touch the kept sums.
      if constexpr (FMT == kQ8) {
        uint4 qa[kStageRows], qb[kStageRows];
        float dv[kStageRows];
#pragma unroll
        for (int k = 0; k < kStageRows; ++k) {
          qa[k] = *reinterpret_cast<const uint4 *>(stq + qofs[k]);
          qb[k] = *reinterpret_cast<const uint4 *>(stq + qofs[k] + 16);
          dv[k] = __half2float(*reinterpret_cast<const __half *>(stq + sofs[k]));
        }
        if (kEarlyRelease) release(s);
        if constexpr (AR == kFixedX) {
          int c0[kStageRows], c1[kStageRows], c2[kStageRows];  // sum_j q_j L_l(X_j), one per limb
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) c0[k] = c1[k] = c2[k] = 0;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int k = 0; k < kStageRows; ++k) {
              const uint32_t w = kk == 0 ? qa[k].x : kk == 1 ? qa[k].y : kk == 2 ? qa[k].z : kk == 3 ? qa[k].w
                               : kk == 4 ? qb[k].x : kk == 5 ? qb[k].y : kk == 6 ? qb[k].z : qb[k].w;
              c0[k] = dp4a_su(w, fx.p[0][kk], c0[k]);
              c1[k] = dp4a_su(w, fx.p[1][kk], c1[k]);
              c2[k] = dp4a_ss(w, fx.p[2][kk], c2[k]);
            }
          }
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) {
            // sum q X = c2 2^16 + (c1 2^8 + c0); the bracket is exact in int32 (|.| < 2^30)
            const float qx = fmaf(__int2float_rn(c2[k]), 65536.0f, __int2float_rn(c0[k] + c1[k] * 256));
            part[k] = (dv[k] * qx) * fx.inv_s;
          }
        } else {
          float2 s0[kStageRows], s1[kStageRows];
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) s0[k] = s1[k] = f2(0.f, 0.f);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int k = 0; k < kStageRows; ++k) {
              const uint32_t w = kk == 0 ? qa[k].x : kk == 1 ? qa[k].y : kk == 2 ? qa[k].z : kk == 3 ? qa[k].w
                               : kk == 4 ? qb[k].x : kk == 5 ? qb[k].y : kk == 6 ? qb[k].z : qb[k].w;
              float2 q01, q23;
              s8x4_to_f2(w, mg, q01, q23);
              s0[k] = __ffma2_rn(q01, xr[2 * kk], s0[k]);
              s1[k] = __ffma2_rn(q23, xr[2 * kk + 1], s1[k]);
            }
          }
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) {
            const float2 st = __fadd2_rn(s0[k], s1[k]);
            part[k] = dv[k] * (st.x + st.y);
          }
        }
      } else if constexpr (FMT == kQ6) {
        // f32 only: each block is two 16-weight sub-blocks, scaled once each by the
        // exact d * scale (no offset term, so the error is relative to sum |w||x|)
        uint4 ql[kStageRows];
        uint2 qh[kStageRows];
        float ds0[kStageRows], ds1[kStageRows];
#pragma unroll
        for (int k = 0; k < kStageRows; ++k) {
          const uint8_t *rw = stq + qofs[k] - qoff;  // the row's first byte in the stage
          ql[k] = *reinterpret_cast<const uint4 *>(rw + qoff);
          qh[k] = *reinterpret_cast<const uint2 *>(rw + q6_hi);
          const uint32_t sc2 = *reinterpret_cast<const uint16_t *>(rw + q6_sc);
          const float d = __half2float(*reinterpret_cast<const __half *>(rw + q6_d));
          ds0[k] = __fmul_rn(d, float(int8_t(sc2 & 0xFFu)));
          ds1[k] = __fmul_rn(d, float(int8_t(sc2 >> 8)));
        }
        if (kEarlyRelease) release(s);
        float2 a0[kStageRows], a1[kStageRows];
#pragma unroll
        for (int k = 0; k < kStageRows; ++k) a0[k] = a1[k] = f2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kStageRows; ++k) {
          float2 v[16];
          q6k_block_to_f2(ql[k], qh[k], mg, v);
#pragma unroll
          for (int p = 0; p < 8; ++p) a0[k] = __ffma2_rn(v[p], xr[p], a0[k]);
#pragma unroll
          for (int p = 8; p < 16; ++p) a1[k] = __ffma2_rn(v[p], xr[p], a1[k]);
        }
#pragma unroll
        for (int k = 0; k < kStageRows; ++k) part[k] = fmaf(ds1[k], a1[k].x + a1[k].y, ds0[k] * (a0[k].x + a0[k].y));
      } else {
        uint4 q[kStageRows], h[kStageRows];
#pragma unroll
        for (int k = 0; k < kStageRows; ++k) {
          q[k] = *reinterpret_cast<const uint4 *>(stq + qofs[k]);
          h[k] = *reinterpret_cast<const uint4 *>(stq + sofs[k]);
        }
        if (kEarlyRelease) release(s);
        float2 DM[kStageRows];
        float mu[kStageRows], R[kStageRows];
#pragma unroll
        for (int k = 0; k < kStageRows; ++k) {
          const uint32_t lo = g0 ? h[k].y : (g1 ? h[k].z : h[k].w);
          const uint32_t hi = g0 ? h[k].z : h[k].w;
          const uint32_t f = __funnelshift_r(lo, hi, sh);
          const float2 scm = q4k_field_to_f2(f, mg);  // (sc, m)
          DM[k] = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&h[k].x)), scm);  // (d sc, dmin m)
          // each weight is d sc (q - mu) - R with the shift mu of q4k_mu: the quants are
          // shifted before they are summed, so near-cancelling weights keep the error
          // proportional to sum |w||x|
          mu[k] = q4k_mu(DM[k]);
          R[k] = fmaf(-DM[k].x, mu[k], DM[k].y);
        }
        if constexpr (AR == kFixedX) {
          int c0[kStageRows], c1[kStageRows], c2[kStageRows];
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) c0[k] = c1[k] = c2[k] = 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int k = 0; k < kStageRows; ++k) {
              const uint32_t w = kk == 0 ? q[k].x : kk == 1 ? q[k].y : kk == 2 ? q[k].z : q[k].w;
              const uint32_t ev = w & 0x0F0F0F0Fu, od = (w >> 4) & 0x0F0F0F0Fu;  // even / odd nibbles as bytes
              c0[k] = dp4a_uu(od, fx.p[0][2 * kk + 1], dp4a_uu(ev, fx.p[0][2 * kk], c0[k]));
              c1[k] = dp4a_uu(od, fx.p[1][2 * kk + 1], dp4a_uu(ev, fx.p[1][2 * kk], c1[k]));
              c2[k] = dp4a_us(od, fx.p[2][2 * kk + 1], dp4a_us(ev, fx.p[2][2 * kk], c2[k]));
            }
          }
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) {
            // sum (q - mu) X = hi 2^16 + lo, both exact in int32 (|hi| < 2^17, |lo| < 2^26)
            const int m = int(mu[k]);
            const int hi = c2[k] - m * fx.s2;
            const int lo = c0[k] + c1[k] * 256 - m * fx.s01;
            const float qx = fmaf(__int2float_rn(hi), 65536.0f, __int2float_rn(lo));
            part[k] = fmaf(DM[k].x, qx, -R[k] * fx.xsum) * fx.inv_s;  // (d sc sum (q - mu) X - R sum X) / 2^e
          }
        } else {
          float2 s0[kStageRows], s1[kStageRows], b01[kStageRows], b23[kStageRows];
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) {
            s0[k] = s1[k] = f2(0.f, 0.f);
            b01[k] = __fadd2_rn(mg.b_u4_01, f2(-mu[k], -mu[k]));  // -(2^23 + mu), -(2^19 + mu): exact
            b23[k] = __fadd2_rn(mg.b_u4_23, f2(-mu[k], -mu[k]));
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int k = 0; k < kStageRows; ++k) {
              const uint32_t w = kk == 0 ? q[k].x : kk == 1 ? q[k].y : kk == 2 ? q[k].z : q[k].w;
              float2 qq[4];  // q - mu, exactly
              u4x8_to_f2_shifted(w, mg, b01[k], b23[k], qq);
              s0[k] = __ffma2_rn(qq[0], xr[4 * kk], s0[k]);
              s1[k] = __ffma2_rn(qq[1], xr[4 * kk + 1], s1[k]);
              s0[k] = __ffma2_rn(qq[2], xr[4 * kk + 2], s0[k]);
              s1[k] = __ffma2_rn(qq[3], xr[4 * kk + 3], s1[k]);
            }
          }
#pragma unroll
          for (int k = 0; k < kStageRows; ++k) {
            const float2 st = __fadd2_rn(s0[k], s1[k]);
            part[k] = fmaf(DM[k].x, st.x + st.y, -R[k] * xsum);  // d sc_j sum((q - mu) x) - R sum(x)
          }
        }
      }
      if (!kEarlyRelease) release(s);
      if (++s == (grp + 1) * SG) {
        s = grp * SG;
        parity ^= 1u;
      }
      butterfly4(part, lane);
      if ((lane & 7) == 0) {
        const int v = rbeg * kV + t * kStageRows + (lane >> 3);  // local virtual row
        if (v < vend && QDQ_GUARD(v * a.wpr + slice < a.psum_cap, QDQ_CHECK_SMEM)) psum[v * a.wpr + slice] = part[0];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) atomicAdd(&g_xs_timeouts, 1u);
  // epilogue: add the slice totals of each row in fixed order
  for (int r = threadIdx.x; r < nreal; r += blockDim.x) {
    if (EPI == kSwiglu) {
      // local output row r is virtual row 2r (gate) and 2r + 1 (up)
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
  // The last thing the CTA waits for: the completion of every copy the producer
  // issued (the last fill of each slot), so that no bulk copy can still be writing
  // into this CTA's shared memory when it exits, also after a timed-out wait.
  if (warp == ncw && lane == 0) {
    bool drained = true;
    for (int g = 0; g < G; ++g) {
      const int issued = stop_i == rounds ? gstages(g) : min(gstages(g), stop_i + (g < stop_g ? 1 : 0));
      for (int i = issued - SG < 0 ? 0 : issued - SG; i < issued; ++i)
        drained = mbar_wait(&full[g * SG + i % SG], (i / SG) & 1) && drained;
    }
    if (!drained) atomicAdd(&g_xs_timeouts, 1u);
  }
}

// Registers per thread of a kernel (queried once per kernel).
cudaError_t kernel_regs(const void *func, int *regs) {
  static std::mutex mu;
  static std::vector<std::pair<const void *, int>> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto &c : cache)
    if (c.first == func) {
      *regs = c.second;
      return cudaSuccess;
    }
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, func);
  if (e != cudaSuccess) return e;
  cache.emplace_back(func, fa.numRegs);
  *regs = fa.numRegs;
  return cudaSuccess;
}

// `a` arrives with the pointers, n_out and n_in set; this fills in the launch shape.
template <int FMT, int EPI, int AR>
int launch_xs_ar(XsArgs a, cudaStream_t s, const DeviceInfo &di) {
  const int n_out = a.n_out, n_in = a.n_in;
  a.wpr = ((n_in >> 5) + 31) / 32;
  auto kern = gemv_xs_kernel<FMT, EPI, AR>;
  // About 6 consumer warps (9 for the f32 Q4_K arithmetic and the SwiGLU, which
  // carry twice the weights per byte, or two matrices): measured best on
  // 3072 <-> 8192 decode chains.  More warps add contention without adding throughput.  The groups must also fit in half an SM's
  // registers together with the producer warp, so that the next kernel's CTA
  // fits beside this one and its weights stream in while this one computes.
  int regs = 0;
  const cudaError_t er = kernel_regs(reinterpret_cast<const void *>(kern), &regs);
  if (er != cudaSuccess) return fail_cuda(er);
  const int warps_half_sm = di.regs_per_sm / 2 / (((regs + 7) / 8) * 8 * 32);
  a.groups = (FMT == kQ8 || (AR == kFixedX && EPI != kSwiglu) ? 6 : 9) / a.wpr;
  if (a.groups > (warps_half_sm - 1) / a.wpr) a.groups = (warps_half_sm - 1) / a.wpr;
  if (a.groups > (kMaxThreads / 32 - 1) / a.wpr) a.groups = (kMaxThreads / 32 - 1) / a.wpr;
  if (a.groups < 1) a.groups = 1;
  if (opt_xs_groups() > 0) a.groups = opt_xs_groups();
  if (32 * (a.wpr * a.groups + 1) > kMaxThreads) return QDQ_ERR_UNSUPPORTED;
  const int pf = opt_l2_prefetch();
  a.l2_prefetch = EPI == kQkv ? 0 : pf == 3 ? 0 : pf;
  const int64_t q_row = FMT == kQ8 ? n_in : FMT == kQ4 ? n_in / 2 : q6k_row_bytes(n_in);
  const int64_t s_row = FMT == kQ8 ? n_in / 16 : FMT == kQ4 ? (n_in / 256) * 16 : 0;
  a.stage_bytes = int((kStageRows * (q_row + s_row) + 127) / 128 * 128);
  // The FFN kernels (SwiGLU, down + residual) run two CTAs per SM with two ring slots
  // per group: both CTAs compute at once instead of one computing beside the next
  // kernel's prefill, which measured ~7 % faster for the block.  The GEMVs keep one.
  constexpr bool kFfn = EPI == kSwiglu || EPI == kResidual;
  int grid = di.sm_count * ctas_per_sm_or(kFfn ? 2 : 1);
  if (grid > n_out) grid = n_out;
  const int max_rows = (n_out + grid - 1) / grid;
  const size_t psum_bytes = size_t(max_rows) * (EPI == kSwiglu ? 2 : 1) * a.wpr * sizeof(float);
  // ring: about half an SM's shared memory, so the next kernel's CTA fits beside
  // this one; at least two slots per group, so drop groups that would not fit
  const long budget = long(di.smem_per_sm) / 2 - di.reserved_smem_per_block - long(psum_bytes) - 1024;
  if (opt_xs_groups() == 0) {
    const int g_smem = int(budget / (2L * a.stage_bytes));
    if (a.groups > g_smem) a.groups = g_smem < 1 ? 1 : g_smem;
  }
  int sg = kFfn ? 2 : int(budget / (long(a.stage_bytes) * a.groups));
  if (sg > 8) sg = 8;
  if (sg < 2) sg = 2;
  if (opt_xs_stages() > 0) sg = opt_xs_stages();
  a.sg = sg;
  const int stages = a.groups * sg;
  // Automatic L2 prefetch (option 0) of the rows the first ring fill leaves out:
  // measured faster for the Q8_0 GEMV chains (the 8192-wide down projection most),
  // slower for the FFN.  Only when those rows fit in half the L2: on a matrix
  // several times larger than L2 (a vocabulary projection) the prefetched lines
  // evict one another before they are read, and the prefetch costs time.
  if (pf == 0 && FMT == kQ8 && EPI != kQkv) {
    const int64_t rest = int64_t(n_out) * (q_row + s_row) - int64_t(grid) * stages * kStageRows * (q_row + s_row);
    a.l2_prefetch = rest <= int64_t(di.l2_bytes) / 2 ? 2 : 0;
  }
  const size_t smem = size_t(stages) * a.stage_bytes + 2 * stages * sizeof(uint64_t) + psum_bytes;
  a.psum_cap = int(psum_bytes / sizeof(float));
  if (smem > size_t(di.max_smem_optin)) return QDQ_ERR_UNSUPPORTED;
  const cudaError_t e0 = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(smem));
  if (e0 != cudaSuccess) return fail_cuda(e0);
  const cudaError_t e = launch(kern, dim3(grid), dim3(32 * (a.wpr * a.groups + 1)), smem, s, a, make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

template <int FMT, int EPI>
int launch_xs(const XsArgs &a, cudaStream_t s, const DeviceInfo &di) {
  if constexpr (FMT == kQ6) return launch_xs_ar<FMT, EPI, kFloatX>(a, s, di);  // Q6_K: f32 arithmetic only
  else
    return opt_xs_float_x() ? launch_xs_ar<FMT, EPI, kFloatX>(a, s, di) : launch_xs_ar<FMT, EPI, kFixedX>(a, s, di);
}

}  // namespace

bool gemv_xs_supported(int n_in, int batch, int fmt) {
  // one 32-weight block per lane and at most 16 slice warps per row; stage copies of
  // the Q8_0 scale plane start on 16-byte boundaries only when n_in % 256 == 0
  return batch == 1 && (n_in >> 5) <= 32 * 16 && (fmt != 0 || n_in % 256 == 0);
}

int launch_gemv_xs(int fmt, int mode, const void *W, const void *W2, const float *x, const float *residual,
                   float *y, int n_out, int n_in, cudaStream_t s) {
  // the f32 arithmetic runs in the direct-load kernel unless the ring kernel is selected
  if (opt_batch1_kernel() == 0 && (opt_xs_float_x() || fmt == 2))
    return launch_gemv_dl(fmt, mode, W, W2, x, residual, y, n_out, n_in, s);
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  XsArgs a{};
  a.W = static_cast<const uint8_t *>(W);
  a.W2 = static_cast<const uint8_t *>(W2);
  a.x = x;
  a.residual = residual;
  a.y = y;
  a.n_out = n_out;
  a.n_in = n_in;
  if (fmt == 0) return launch_xs<kQ8, kPlain>(a, s, di);
  if (fmt == 2) return launch_xs<kQ6, kPlain>(a, s, di);
  if (mode == 1) return launch_xs<kQ4, kSwiglu>(a, s, di);
  if (mode == 2) return launch_xs<kQ4, kResidual>(a, s, di);
  return launch_xs<kQ4, kPlain>(a, s, di);
}

int launch_gemv_xs_qkv(const void *Wq, const void *Wk, const void *Wv, const float *x, float *q, float *k, float *v,
                       int n_q, int n_kv, int n_in, cudaStream_t s) {
  if (opt_batch1_kernel() == 0 && opt_xs_float_x())
    return launch_gemv_dl_qkv(Wq, Wk, Wv, x, q, k, v, n_q, n_kv, n_in, s);
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  XsArgs a{};
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
  return launch_xs<kQ4, kQkv>(a, s, di);
}

QDQ_CHECK_READER(read_checks_xs)

int read_xs_timeouts() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_xs_timeouts, sizeof(v)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_xs_timeouts, &zero, sizeof(zero)) != cudaSuccess) return -1;
  return int(v);
}

}  // namespace qdq

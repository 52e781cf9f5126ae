// Batch-prefill GEMMs on the 5th-generation tensor cores (tcgen05, TMEM, TMA):
// Q8_0 and Q4_K weights, and the Q4_K SwiGLU expansion for M > 1 tokens.
//
// "Module cuda_lane", Goal: prefer tensor-core dense matmul for batch
// prefill-shaped GEMMs; "weight_cache.rs", try_cuda_batch_gemv: hidden is
// packed batch x n_in, weight is row-major n_out x n_in (GGML rows), out is
// batch x n_out.  The reference densifies the weights on the host, pads every
// dimension to 16 and transposes for a WMMA kernel; here the quantised weights
// stay on the device and are dequantised tile by tile in shared memory, and
// ragged token counts are masked instead of padded.  The Q4_K form serves the
// prefill-shaped batches of the Q4_K runners ("Module cuda_lane",
// try_q4k_soa_gemv / try_q4k_soa_fused_swiglu): for the SwiGLU the gate and up
// rows of a tile share the activation tile and accumulate side by side in TMEM,
// and the epilogue writes silu(g) * u.
//
// Computation (per output element):  Y[m, r] = sum_k bf16(X[m, k]) * bf16(w[r, k])
// with f32 accumulation, w the exact f32 dequantised weight (Q8_0: d*q;
// Q4_K: RN(d*sc*q - dmin*m), one FMA) rounded once to bf16; X is rounded once to
// bf16 by a small conversion kernel that runs first.
//
// Tiling ("swap AB"): the MMA's M dimension is 128 weight rows (n_out), its N
// dimension is the token tile (16..256), K steps by 64 per pipeline stage.
// One CTA = one (128-row, token-tile, K-range) tile; K is split across CTAs
// when the tile count alone cannot fill the SMs.  Split partial tiles go to a
// workspace; the CTA that finishes a tile last (an atomic ticket per tile, no
// waiting) adds the partials in split order and writes Y, so results do not
// depend on which CTA ran first.
//
// Warp roles (576 threads):
//   warps 0-15 dequantise the weight tile(s) into bf16 A tiles in the
//              128-byte-swizzled K-major layout the tensor core reads (Q8_0:
//              four threads per row, 16 quants each, from a 64-byte-swizzled
//              int8 TMA tile; Q4_K: a warp per 8 rows, four threads per row,
//              16 nibbles each, from a dense 32-byte-row TMA tile, with the
//              row's superblock header fetched once per superblock); after the
//              last stage the same warps read the accumulators out of TMEM and
//              store Y (warp w reads TMEM lanes 32*(w%4).. and every fourth
//              16-column chunk);
//   warp 16    TMA producer: weight tile(s) and the bf16 activation tile
//              (N x 64, 128-byte swizzle) per stage;
//   warp 17    allocates TMEM, and one lane issues tcgen05.mma (K = 16 each)
//              and tcgen05.commit to release each stage.
// Every mbarrier wait is bounded by a wall-clock limit; a wait that runs out
// counts a pipeline timeout (qdq_pipeline_timeouts) and the CTA winds down
// instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "qdq_internal.cuh"

namespace qdq {

__device__ unsigned int g_pipeline_timeouts = 0;

namespace {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K per stage (128 bytes of bf16: one swizzle span)
constexpr int kDequantWarps = 16;  // 4 per SM sub-partition: hides ALU latency
constexpr int kThreads = 32 * (kDequantWarps + 2);
constexpr uint32_t kATileBytes = BM * BK * 2;  // bf16 weight tile
enum WFmt { kWQ8 = 0, kWQ4 = 1 };

// ---- TMA ----------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// L2 prefetch of one TMA tile (no shared memory, no completion): issued well ahead
// of the tile's load, so that many more weight rows are in flight from HBM than
// the shared-memory ring alone could hold.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *tm, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y)
               : "memory");
}
constexpr int kPrefetchStages = 16;  // how far ahead of the loads the weight tiles are prefetched into L2

// ---- tcgen05 --------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile in the canonical
// 128-byte-swizzle layout: rows of 128 bytes (64 bf16 along K), groups of 8
// rows 1024 bytes apart, 16-byte chunk c of row r stored at chunk c ^ (r % 8).
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29,
// unused for this layout), stride byte offset >> 4 (32-45), descriptor
// version 1 (46-47), swizzle mode 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// Instruction descriptor, kind::f16: f32 accumulator (bits 4-5 = 1), A and B
// bf16 (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

constexpr uint32_t round1k(uint32_t v) { return (v + 1023u) & ~1023u; }

// Two rings in shared memory, every tile on a 1024-byte boundary (the 128-byte
// swizzle atom):
//   load ring, kSL slots, filled by TMA:  [ NA weight tiles as stored | X tile ]
//     (X tile: the f32 activations, N x 64, when kXF; else the bf16 B tile);
//   A ring, kSA slots, filled by the dequantising warps:  [ NA bf16 A tiles |
//     the bf16 B tile when kXF ].
// The load ring is as deep as shared memory allows (up to 16 slots), so that
// many weight tiles are in flight per SM; the A ring only needs to keep the
// tensor core fed.  kXF (token tiles of 64 or fewer): X arrives as f32 and is
// rounded to bf16 in the kernel, so no conversion kernel runs before it.
template <int FMT, int N, int NA>
struct GemmCfg {
  static constexpr bool kXF = N <= 64;
  static constexpr uint32_t kQTileBytes = FMT == kWQ8 ? BM * BK : BM * BK / 2;
  static constexpr uint32_t kBTileBytes = uint32_t(N) * 128;
  static constexpr uint32_t kXTileBytes = kXF ? uint32_t(N) * BK * 4 : kBTileBytes;
  static constexpr uint32_t kLoadSlot = round1k(NA * kQTileBytes + kXTileBytes);
  static constexpr uint32_t kASlot = round1k(NA * kATileBytes + (kXF ? kBTileBytes : 0u));
  static constexpr int kSA = (NA == 1 && N <= 32) ? 3 : 2;
  static constexpr int kFit = int((227u * 1024u - 2048u - uint32_t(kSA) * kASlot) / kLoadSlot);
  static constexpr int kSL = kFit > 16 ? 16 : kFit;
  static constexpr uint32_t kCols = uint32_t(NA * N);
  static constexpr uint32_t kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static constexpr size_t kSmemBytes = 1024 + size_t(kSL) * kLoadSlot + size_t(kSA) * kASlot + 512;
  static_assert(kSL >= 2, "the load ring needs two slots");
  static_assert(kSmemBytes <= 227u * 1024u, "shared memory");
};

struct GemmArgs {
  const uint8_t *W[2];  // packed weights (gate and up for the SwiGLU)
  float *Y;
  float *partials;      // [split][NA][M][n_out] when split > 1
  int *tickets;         // one per (row tile, token tile), zero on entry
  int n_out, n_in, M;
  int kb_per_split, split;
};

// One Q4_K sub-block's (d*sc_j, dmin*m_j) from a 16-byte header record.
__device__ __forceinline__ float2 q4k_header_scale(const uint4 h, int j) {
  const uint64_t lo = uint64_t(h.y) | (uint64_t(h.z) << 32);
  const int bit = 12 * j;
  uint32_t f;
  if (bit + 12 <= 64) f = uint32_t(lo >> bit) & 0xFFFu;
  else if (bit >= 64) f = (h.w >> (bit - 64)) & 0xFFFu;
  else f = (uint32_t(lo >> bit) | (h.w << (64 - bit))) & 0xFFFu;
  const float d = __half2float(__ushort_as_half(uint16_t(h.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(uint16_t(h.x >> 16)));
  return f2(__fmul_rn(d, float(f & 63u)), __fmul_rn(dmin, float(f >> 6)));  // both exact
}

__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) {
  const __nv_bfloat162 p = __float22bfloat162_rn(v);
  return *reinterpret_cast<const uint32_t *>(&p);
}

template <int FMT, int N, int NA>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
                   const __grid_constant__ CUtensorMap tm_x, const GemmArgs g, const Magic mg_param) {
  using C = GemmCfg<FMT, N, NA>;
  const Magic mg = lane_magic(mg_param);
  constexpr int SL = C::kSL, SA = C::kSA;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *aring = smem + SL * C::kLoadSlot;
  uint64_t *lfull = reinterpret_cast<uint64_t *>(aring + SA * C::kASlot);
  uint64_t *lempty = lfull + SL;
  uint64_t *aready = lempty + SL;
  uint64_t *aempty = aready + SA;
  uint64_t *accum = aempty + SA;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
  __shared__ int s_abort, s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int issued = 0;  // TMA stages the producer issued (drained before the CTA exits)
  const int tile_n = blockIdx.x, tile_m = blockIdx.y;
  const int n_in = g.n_in, n_out = g.n_out, M = g.M;
  const int nkb = n_in / BK;
  const int kb0 = blockIdx.z * g.kb_per_split;
  const int kb1 = min(kb0 + g.kb_per_split, nkb);
  const int nk = kb1 - kb0;
  auto qtile = [&](int s, int a) { return smem + s * C::kLoadSlot + a * C::kQTileBytes; };
  auto xtile = [&](int s) { return smem + s * C::kLoadSlot + NA * C::kQTileBytes; };
  auto atile = [&](int j, int a) { return aring + j * C::kASlot + a * kATileBytes; };
  // the MMA's B operand of stage i: in the A slot (converted here) or the load slot (TMA)
  auto btile = [&](int i) { return C::kXF ? aring + (i % SA) * C::kASlot + NA * kATileBytes : xtile(i % SL); };
  constexpr int kQBox = FMT == kWQ8 ? BK : BK / 2;  // inner TMA coordinate step of a weight tile per stage

  if (threadIdx.x == 0) {
    for (int i = 0; i < SL; ++i) {
      mbar_init(&lfull[i], 1);
      mbar_init(&lempty[i], 1);
    }
    for (int j = 0; j < SA; ++j) {
      mbar_init(&aready[j], kDequantWarps * 32);
      mbar_init(&aempty[j], 1);
    }
    mbar_init(accum, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kDequantWarps + 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_launch_dependents();

  if (warp == kDequantWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q0)) : "memory");
      if (NA == 2) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q1)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      constexpr uint32_t kTx = NA * C::kQTileBytes + C::kXTileBytes;
      const int npre = nk < SL ? nk : SL;
      // weights do not depend on the previous kernel: start them before the wait
      for (int i = npre; i < nk && i < npre + kPrefetchStages; ++i) {
        tma_prefetch_2d(&tm_q0, (kb0 + i) * kQBox, tile_n * BM);
        if (NA == 2) tma_prefetch_2d(&tm_q1, (kb0 + i) * kQBox, tile_n * BM);
      }
      for (int i = 0; i < npre; ++i) {
        mbar_arrive_expect_tx(&lfull[i], kTx);
        tma_load_2d(qtile(i, 0), &tm_q0, (kb0 + i) * kQBox, tile_n * BM, &lfull[i]);
        if (NA == 2) tma_load_2d(qtile(i, 1), &tm_q1, (kb0 + i) * kQBox, tile_n * BM, &lfull[i]);
      }
      pdl_wait();
      for (int i = 0; i < npre; ++i) tma_load_2d(xtile(i), &tm_x, (kb0 + i) * BK, tile_m * N, &lfull[i]);
      issued = npre;
      for (int i = npre; i < nk; ++i) {
        const int s = i % SL;
        // after any timed-out wait in this CTA, issue nothing more
        if (*reinterpret_cast<volatile int *>(&s_abort) || !mbar_wait(&lempty[s], ((i / SL) + 1) & 1)) {
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&lfull[s], kTx);
        tma_load_2d(qtile(s, 0), &tm_q0, (kb0 + i) * kQBox, tile_n * BM, &lfull[s]);
        if (NA == 2) tma_load_2d(qtile(s, 1), &tm_q1, (kb0 + i) * kQBox, tile_n * BM, &lfull[s]);
        tma_load_2d(xtile(s), &tm_x, (kb0 + i) * BK, tile_m * N, &lfull[s]);
        issued = i + 1;
        if (i + kPrefetchStages < nk) {
          tma_prefetch_2d(&tm_q0, (kb0 + i + kPrefetchStages) * kQBox, tile_n * BM);
          if (NA == 2) tma_prefetch_2d(&tm_q1, (kb0 + i + kPrefetchStages) * kQBox, tile_n * BM);
        }
      }
    } else {
      pdl_wait();
    }
  } else if (warp == kDequantWarps + 1) {
    // ---------------- MMA issuer ----------------
    pdl_wait();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, N);
      for (int i = 0; i < nk; ++i) {
        const int s = i % SL, j = i % SA;
        if (!mbar_wait(&aready[j], (i / SA) & 1) || !mbar_wait(&lfull[s], (i / SL) & 1)) {
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t b_base = smem_u32(btile(i));
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          const uint32_t a_base = smem_u32(atile(j, a));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(tmem + uint32_t(a * N), desc_kmajor_sw128(a_base + 32 * k), desc_kmajor_sw128(b_base + 32 * k),
                      idesc, (i | k) != 0);
        }
        umma_commit(&aempty[j]);  // the A slot (and the B tile in it) is free once these MMAs are done
        umma_commit(&lempty[s]);  // so is the load slot
      }
      umma_commit(accum);
    }
  } else {
    // ---------------- dequantise, then epilogue ----------------
    // The weights do not depend on the previous kernel, so dequantisation starts
    // at once; only the epilogue (which writes Y) waits for it.
    bool ok = true;
    // stage i may overwrite A slot i % SA once the MMAs of stage i - SA are done
    auto wait_slots = [&](int i) {
      if (!mbar_wait(&lfull[i % SL], (i / SL) & 1)) return false;
      return i < SA || mbar_wait(&aempty[i % SA], ((i / SA) - 1) & 1);
    };
    // kXF: X rows of the stage (f32, 256 bytes each) -> the bf16 B tile in the
    // 128-byte-swizzled K-major layout; one 16-byte chunk (8 values) per thread
    auto convert_x = [&](int i) {
      if constexpr (C::kXF) {
        const float *xs = reinterpret_cast<const float *>(xtile(i % SL));
        uint8_t *bt = btile(i);
        for (int t = threadIdx.x; t < N * 8; t += kDequantWarps * 32) {
          const int r = t >> 3, c = t & 7;
          const float4 v0 = *reinterpret_cast<const float4 *>(xs + r * BK + 8 * c);
          const float4 v1 = *reinterpret_cast<const float4 *>(xs + r * BK + 8 * c + 4);
          *reinterpret_cast<uint4 *>(bt + r * 128 + ((c ^ (r & 7)) << 4)) =
              make_uint4(pack_bf16x2(f2(v0.x, v0.y)), pack_bf16x2(f2(v0.z, v0.w)), pack_bf16x2(f2(v1.x, v1.y)),
                         pack_bf16x2(f2(v1.z, v1.w)));
        }
      }
    };
    if constexpr (FMT == kWQ8) {
      const int row = threadIdx.x & (BM - 1);  // weight row within the tile
      const int part = threadIdx.x >> 7;       // which 16 of the row's 64 quants
      const int grow = tile_n * BM + row;
      const uint32_t *d32[NA];
#pragma unroll
      for (int a = 0; a < NA; ++a)
        d32[a] = reinterpret_cast<const uint32_t *>(g.W[a] + int64_t(n_out) * n_in) + int64_t(grow) * (n_in / BK);
      const int qsw = (row >> 1) & 3;  // 64-byte swizzle of the TMA-written int8 tile
      // the row's two block scales per stage (an fp16 pair), fetched four stages ahead
      uint32_t dqa[4][NA];
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int a = 0; a < NA; ++a) dqa[t][a] = t < nk ? __ldg(d32[a] + kb0 + t) : 0u;
      for (int i = 0; i < nk; ++i) {
        const int s = i % SL, j = i % SA;
        uint32_t dq[NA];
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          dq[a] = dqa[0][a];
          dqa[0][a] = dqa[1][a];
          dqa[1][a] = dqa[2][a];
          dqa[2][a] = dqa[3][a];
          dqa[3][a] = i + 4 < nk ? __ldg(d32[a] + kb0 + i + 4) : 0u;
        }
        if (!wait_slots(i)) {
          s_abort = 1;
          ok = false;
          break;
        }
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          const uint8_t *qt = qtile(s, a);
          uint8_t *at = atile(j, a);
          const __half2 dh = *reinterpret_cast<const __half2 *>(&dq[a]);
          const float dsc = part < 2 ? __low2float(dh) : __high2float(dh);  // block scale of K 32*(part/2)..
          const float2 dpair = f2(dsc, dsc);
          const uint4 qv = *reinterpret_cast<const uint4 *>(qt + row * 64 + ((part ^ qsw) << 4));
          const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
          uint32_t packed[8];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            float2 q01, q23;
            s8x4_to_f2(words[w], mg, q01, q23);
            packed[2 * w] = pack_bf16x2(__fmul2_rn(q01, dpair));  // d*q exact in f32, rounded once
            packed[2 * w + 1] = pack_bf16x2(__fmul2_rn(q23, dpair));
          }
          // 16 quants -> two 16-byte bf16 chunks (K 16p..16p+7 and 16p+8..16p+15)
          *reinterpret_cast<uint4 *>(at + row * 128 + (((2 * part) ^ (row & 7)) << 4)) =
              make_uint4(packed[0], packed[1], packed[2], packed[3]);
          *reinterpret_cast<uint4 *>(at + row * 128 + (((2 * part + 1) ^ (row & 7)) << 4)) =
              make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
        convert_x(i);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&aready[j]);
      }
    } else {
      // Q4_K: warp w takes rows 8w..8w+7, four threads per row, 16 nibbles (8 bytes) each:
      // a warp reads 256 contiguous bytes of the dense tile
      const int row = warp * 8 + (lane >> 2);
      const int part = lane & 3;
      const int grow = tile_n * BM + row;
      const uint4 *hdr[NA];  // the row's superblock headers
#pragma unroll
      for (int a = 0; a < NA; ++a)
        hdr[a] = reinterpret_cast<const uint4 *>(g.W[a] + int64_t(n_out) * (n_in / 2)) + int64_t(grow) * (n_in / 256);
      // the header of the current superblock, and of the next one fetched ahead
      const int nsb = n_in / 256;
      uint4 hcur[NA], hnext[NA];
      int cur_sb = kb0 >> 2;
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        hcur[a] = __ldg(hdr[a] + cur_sb);
        hnext[a] = cur_sb + 1 < nsb ? __ldg(hdr[a] + cur_sb + 1) : hcur[a];
      }
      for (int i = 0; i < nk; ++i) {
        const int s = i % SL, jj = i % SA;
        const int kb = kb0 + i;
        if ((kb >> 2) != cur_sb) {  // entering the next superblock
          ++cur_sb;
#pragma unroll
          for (int a = 0; a < NA; ++a) {
            hcur[a] = hnext[a];
            hnext[a] = cur_sb + 1 < nsb ? __ldg(hdr[a] + cur_sb + 1) : hcur[a];
          }
        }
        const int j = 2 * (kb & 3) + (part >> 1);  // sub-block of these 16 weights in the superblock
        float2 dm[NA];                             // (d*sc_j, dmin*m_j)
#pragma unroll
        for (int a = 0; a < NA; ++a) dm[a] = q4k_header_scale(hcur[a], j);
        if (!wait_slots(i)) {
          s_abort = 1;
          ok = false;
          break;
        }
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          const uint2 qv = *reinterpret_cast<const uint2 *>(qtile(s, a) + row * 32 + part * 8);
          uint8_t *at = atile(jj, a);
          const float2 D = f2(dm[a].x, dm[a].x), Dm = f2(-dm[a].y, -dm[a].y);
          uint32_t packed[8];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            float2 q[4];
            u4x8_to_f2(w == 0 ? qv.x : qv.y, mg, q);
#pragma unroll
            for (int p = 0; p < 4; ++p) packed[4 * w + p] = pack_bf16x2(__ffma2_rn(D, q[p], Dm));  // RN(D q - Dm)
          }
          *reinterpret_cast<uint4 *>(at + row * 128 + (((2 * part) ^ (row & 7)) << 4)) =
              make_uint4(packed[0], packed[1], packed[2], packed[3]);
          *reinterpret_cast<uint4 *>(at + row * 128 + (((2 * part + 1) ^ (row & 7)) << 4)) =
              make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
        convert_x(i);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&aready[jj]);
      }
    }
    pdl_wait();
    if (ok && mbar_wait(accum, 0)) {
      tc_fence_after();
      const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
      const int m0 = tile_m * N;
      const int erow = tile_n * BM + (warp & 3) * 32 + lane;  // this thread's output row (TMEM lane)
      const int tile_id = tile_m * gridDim.x + tile_n;
      if (g.split == 1) {
#pragma unroll 1
        for (int c0 = (warp >> 2) * 16; c0 < N; c0 += 16 * (kDequantWarps / 4)) {
          uint32_t r[NA][16];
#pragma unroll
          for (int a = 0; a < NA; ++a) tmem_ld16(tmem + lane_base + uint32_t(a * N + c0), r[a]);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int m = m0 + c0 + jj;
            if (m < M) {
              float v = __uint_as_float(r[0][jj]);
              if (NA == 2) {
                const float u = __uint_as_float(r[NA - 1][jj]);
                v = v / (1.0f + expf(-v)) * u;
              }
              if (QDQ_GUARD(erow < n_out, QDQ_CHECK_OUT)) g.Y[int64_t(m) * n_out + erow] = v;
            }
          }
        }
      } else {
        // split-K: store this split's partial tile, take a ticket; the last of the
        // tile's splits adds all partials in split order and writes Y
        const int z = blockIdx.z;
#pragma unroll 1
        for (int c0 = (warp >> 2) * 16; c0 < N; c0 += 16 * (kDequantWarps / 4)) {
          uint32_t r[NA][16];
#pragma unroll
          for (int a = 0; a < NA; ++a) tmem_ld16(tmem + lane_base + uint32_t(a * N + c0), r[a]);
#pragma unroll
          for (int a = 0; a < NA; ++a)
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int m = m0 + c0 + jj;
              if (m < M && QDQ_GUARD(erow < n_out, QDQ_CHECK_OUT))
                g.partials[((int64_t(z) * NA + a) * M + m) * n_out + erow] = __uint_as_float(r[a][jj]);
            }
        }
        __threadfence();
        named_bar_sync(1, 32 * kDequantWarps);
        if (threadIdx.x == 0) s_last = atomicAdd(&g.tickets[tile_id], 1) == g.split - 1;
        named_bar_sync(1, 32 * kDequantWarps);
        if (s_last) {
          __threadfence();
          // the tile's partials, added in split order: every load of a 16-column chunk is
          // issued before any is used, so the reads overlap instead of queueing
#pragma unroll 1
          for (int c0 = (warp >> 2) * 16; c0 < N; c0 += 16 * (kDequantWarps / 4)) {
#pragma unroll 1
            for (int h = 0; h < 16; h += 8) {  // 8 columns at a time
              float acc[NA][8];
#pragma unroll
              for (int a = 0; a < NA; ++a)
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) acc[a][jj] = 0.f;
              for (int zz = 0; zz < g.split; ++zz) {
#pragma unroll
                for (int a = 0; a < NA; ++a)
#pragma unroll
                  for (int jj = 0; jj < 8; ++jj) {
                    const int m = m0 + c0 + h + jj;
                    if (m < M) acc[a][jj] += __ldcg(&g.partials[((int64_t(zz) * NA + a) * M + m) * n_out + erow]);
                  }
              }
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int m = m0 + c0 + h + jj;
                if (m < M) {
                  float v = acc[0][jj];
                  if (NA == 2) v = v / (1.0f + expf(-v)) * acc[NA - 1][jj];
                  g.Y[int64_t(m) * n_out + erow] = v;
                }
              }
            }
          }
          if (threadIdx.x == 0) g.tickets[tile_id] = 0;  // ready for the next call
        }
      }
    } else {
      s_abort = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  // The last waits of the CTA: every MMA the issuer started has completed (the
  // accumulator commit is issued after the MMA loop even when it stopped early)
  // before the TMEM is freed, and every TMA load the producer issued has landed
  // before the CTA's shared memory is released.
  bool drained = true;
  if (warp == kDequantWarps + 1 && lane == 0) drained = mbar_wait(accum, 0);
  if (warp == kDequantWarps && lane == 0)
    for (int i = issued - SL < 0 ? 0 : issued - SL; i < issued; ++i)
      drained = mbar_wait(&lfull[i % SL], (i / SL) & 1) && drained;
  if (!drained) atomicAdd(&g_pipeline_timeouts, 1u);
  if (threadIdx.x == 0 && s_abort) atomicAdd(&g_pipeline_timeouts, 1u);
  if (warp == kDequantWarps + 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// X (f32, M x n_in) -> bf16 workspace; zero the split-K tickets.
__global__ void __launch_bounds__(256) x_to_bf16_kernel(const float4 *__restrict__ X, uint2 *__restrict__ xb,
                                                        int64_t n4, int *tickets, int n_tickets) {
  pdl_launch_dependents();
  pdl_wait();  // the workspace may still be in use by the previous kernel
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += stride) {
    const float4 v = X[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    xb[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
  }
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_tickets; i += stride) tickets[i] = 0;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, []() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

bool encode_2d(CUtensorMap *tm, CUtensorMapDataType dt, void *base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(tm, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The token tile for M tokens.
int token_tile(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256; }

// Launch shape and workspace layout of one GEMM call.  The workspace starts
// with kTicketBytes of split-K tile counters (zero between calls: the last CTA
// of a tile resets its counter), then the bf16 copy of X (token tiles above
// 64 only), then the split-K partial tiles.
constexpr size_t kTicketBytes = 65536;
constexpr int kMaxTiles = int(kTicketBytes / sizeof(int));
struct GemmPlan {
  int N, ntile_n, ntile_m, nkb, split, kb_per;
  size_t xb_bytes, part_bytes;
};
GemmPlan plan_gemm(int M, int n_out, int n_in, int na, int sm_count) {
  GemmPlan p;
  p.N = token_tile(M);
  p.ntile_n = n_out / BM;
  p.ntile_m = (M + p.N - 1) / p.N;
  p.nkb = n_in / BK;
  const int tiles = p.ntile_n * p.ntile_m;
  int split = sm_count / tiles;
  if (split < 1) split = 1;
  if (split > p.nkb) split = p.nkb;
  p.kb_per = (p.nkb + split - 1) / split;
  p.split = (p.nkb + p.kb_per - 1) / p.kb_per;  // every split gets at least one K block
  p.xb_bytes = p.N <= 64 ? 0 : (size_t(M) * n_in * 2 + 255) / 256 * 256;
  p.part_bytes = p.split > 1 ? size_t(p.split) * na * M * n_out * 4 : 0;
  return p;
}

template <int FMT, int N, int NA>
int launch_tile(const uint8_t *const W[2], const float *X, float *Y, void *ws, int n_out, int n_in, int M,
                const GemmPlan &p, cudaStream_t s, const DeviceInfo &di) {
  using C = GemmCfg<FMT, N, NA>;
  CUtensorMap tm_q[2], tm_x;
  for (int a = 0; a < 2; ++a) {
    const uint8_t *w = W[a < NA ? a : 0];
    const bool okq = FMT == kWQ8
                         ? encode_2d(&tm_q[a], CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t *>(w), uint64_t(n_in),
                                     uint64_t(n_out), uint64_t(n_in), BK, BM, CU_TENSOR_MAP_SWIZZLE_64B)
                         : encode_2d(&tm_q[a], CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t *>(w),
                                     uint64_t(n_in / 2), uint64_t(n_out), uint64_t(n_in / 2), BK / 2, BM,
                                     CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!okq) return QDQ_ERR_UNSUPPORTED;
  }

  uint8_t *wsb = static_cast<uint8_t *>(ws);
  GemmArgs g{};
  g.W[0] = W[0];
  g.W[1] = W[NA - 1];
  g.Y = Y;
  g.tickets = reinterpret_cast<int *>(wsb);
  g.partials = reinterpret_cast<float *>(wsb + kTicketBytes + p.xb_bytes);
  g.n_out = n_out;
  g.n_in = n_in;
  g.M = M;
  g.kb_per_split = p.kb_per;
  g.split = p.split;
  if (p.split > 1 && p.ntile_n * p.ntile_m > kMaxTiles) return QDQ_ERR_UNSUPPORTED;

  cudaError_t e;
  if (C::kXF) {
    // X is read as f32 and rounded to bf16 inside the GEMM
    if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float *>(X), uint64_t(n_in), uint64_t(M),
                   uint64_t(n_in) * 4, BK, N, CU_TENSOR_MAP_SWIZZLE_NONE))
      return QDQ_ERR_UNSUPPORTED;
  } else {
    // conversion of X into the workspace, and zeroing of the split-K tickets
    uint8_t *xb = wsb + kTicketBytes;
    if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, uint64_t(n_in), uint64_t(M), uint64_t(n_in) * 2, BK,
                   N, CU_TENSOR_MAP_SWIZZLE_128B))
      return QDQ_ERR_UNSUPPORTED;
    const int64_t n4 = int64_t(M) * n_in / 4;
    int cgrid = int((n4 + 255) / 256);
    if (cgrid > di.sm_count * 8) cgrid = di.sm_count * 8;
    if (cgrid < 1) cgrid = 1;
    e = launch(x_to_bf16_kernel, dim3(cgrid), dim3(256), 0, s, reinterpret_cast<const float4 *>(X),
               reinterpret_cast<uint2 *>(xb), n4, g.tickets, p.split > 1 ? p.ntile_n * p.ntile_m : 0);
    if (e != cudaSuccess) return fail_cuda(e);
  }

  auto kern = gemm_tc_kernel<FMT, N, NA>;
  e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(C::kSmemBytes));  // once per kernel
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch(kern, dim3(p.ntile_n, p.ntile_m, p.split), dim3(kThreads), C::kSmemBytes, s, tm_q[0], tm_q[1], tm_x, g,
             make_magic());
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

template <int FMT, int NA>
int launch_gemm(const uint8_t *const W[2], const float *X, float *Y, void *ws, int n_out, int n_in, int M,
                cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return fail_cuda(e);
  e = get_encoder();
  if (e != cudaSuccess) return fail_cuda(e);
  const GemmPlan p = plan_gemm(M, n_out, n_in, NA, di.sm_count);
  switch (p.N) {
    case 16: return launch_tile<FMT, 16, NA>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 32: return launch_tile<FMT, 32, NA>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 64: return launch_tile<FMT, 64, NA>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 128: return launch_tile<FMT, 128, NA>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    default: return launch_tile<FMT, 256, NA>(W, X, Y, ws, n_out, n_in, M, p, s, di);
  }
}

}  // namespace

size_t gemm_workspace_bytes(int M, int n_out, int n_in, int na) {
  DeviceInfo di;
  if (device_info(&di) != cudaSuccess) return 0;
  const GemmPlan p = plan_gemm(M, n_out, n_in, na, di.sm_count);
  return kTicketBytes + p.xb_bytes + p.part_bytes;
}

int launch_q8_0_gemm_batch(const void *W, const float *X, float *Y, void *ws, int n_out, int n_in, int M,
                           cudaStream_t s) {
  const uint8_t *w[2] = {static_cast<const uint8_t *>(W), nullptr};
  return launch_gemm<kWQ8, 1>(w, X, Y, ws, n_out, n_in, M, s);
}

int launch_q4k_gemm_batch(const void *W, const float *X, float *Y, void *ws, int n_out, int n_in, int M,
                          cudaStream_t s) {
  const uint8_t *w[2] = {static_cast<const uint8_t *>(W), nullptr};
  return launch_gemm<kWQ4, 1>(w, X, Y, ws, n_out, n_in, M, s);
}

int launch_q4k_swiglu_batch(const void *Wg, const void *Wu, const float *X, float *mid, void *ws, int n_ff,
                            int n_embd, int M, cudaStream_t s) {
  const uint8_t *w[2] = {static_cast<const uint8_t *>(Wg), static_cast<const uint8_t *>(Wu)};
  return launch_gemm<kWQ4, 2>(w, X, mid, ws, n_ff, n_embd, M, s);
}

QDQ_CHECK_READER(read_checks_gemm)

int read_gemm_timeouts() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_pipeline_timeouts, sizeof(v)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_pipeline_timeouts, &zero, sizeof(zero)) != cudaSuccess) return -1;
  return int(v);
}

}  // namespace qdq

extern "C" int qdq_pipeline_timeouts(void) {
  const int a = qdq::read_gemm_timeouts(), b = qdq::read_xs_timeouts(), c = qdq::read_dl_timeouts();
  return (a < 0 || b < 0 || c < 0) ? -1 : a + b + c;
}

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
// bf16 (inside the GEMM for token tiles of 16, and of 32 with one weight matrix,
// else by a small conversion kernel that runs first).
//
// Tiling ("swap AB"): the MMA's M dimension is 128 weight rows (n_out), its N
// dimension is the token tile (16..256), K steps by 64 or 128 per pipeline
// stage.  One CTA = one (128-row, token-tile, K-range) tile; K is split across
// the CTAs of a (1, 1, split) thread-block cluster when the tile count alone
// cannot fill the SMs: each split leaves its partial tile in its own shared
// memory, and after a cluster barrier split z adds the partials of its share of
// the tile's tokens in split order through distributed shared memory and
// writes Y, so results do not depend on which CTA ran first.
//
// Warp roles (576 threads):
//   warps 0-15 dequantise the weight tile(s) into bf16 A tiles in the
//              128-byte-swizzled K-major layout the tensor core reads, as two
//              groups of 8 warps taking alternate K stages (Q8_0: two threads
//              per row, 32 quants and one block scale each, from a
//              64-byte-swizzled int8 TMA tile; Q4_K: two threads per row, one
//              32-weight sub-block each, from a dense 32-byte-row TMA tile, with
//              the row's superblock header fetched once per superblock); Q8_0
//              with token tiles of 32 and of 64 and above writes the A tiles into
//              TMEM instead (tcgen05.st; the MMA reads A from there); for the
//              tiles that round X in the kernel the same warps round the stage's
//              f32 X tile to the bf16 B tile.  After the last stage the 16 warps
//              read the accumulators out of TMEM and store Y (warp w reads TMEM
//              lanes 32*(w%4).. and every fourth 16-column chunk);
//   warp 16    TMA producer: weight tile(s) and the activation tile (f32, or
//              bf16 with the 128-byte swizzle for larger token tiles) per stage,
//              into a load ring as deep as shared memory allows;
//   warp 17    allocates TMEM and issues tcgen05.mma (K = 16 each) and
//              tcgen05.commit to release each stage's A slot and load slot.
// Warps 16 and 17 run their loops warp-wide, one elected lane issuing the copies,
// MMAs and commits (the same loops run by lane 0 alone were 10-15 % slower).
// A per-CTA timeline (%globaltimer stamps per stage) showed why the groups: with
// one group of 16 warps every stage cost ~0.5 us of dequantisation latency (the
// tiles were already in shared memory, the tensor core idle), at M = 16 and at
// M = 512 alike.
// Every mbarrier wait is bounded by a wall-clock limit; a wait that runs out
// counts a pipeline timeout (qdq_pipeline_timeouts) and the CTA winds down
// instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "qdq_internal.cuh"

namespace qdq {

__device__ unsigned int g_pipeline_timeouts = 0;

namespace {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K per sub-block (128 bytes of bf16: one swizzle span); a stage holds KB sub-blocks
constexpr int kDequantWarps = 16;  // two groups of 8, taking alternate stages
constexpr int kGroupThreads = 32 * kDequantWarps / 2;
constexpr int kThreads = 32 * (kDequantWarps + 2);
constexpr uint32_t kATileBytes = BM * BK * 2;  // bf16 weight tile of one sub-block
enum WFmt { kWQ8 = 0, kWQ4 = 1 };

// ---- TMA ----------------------------------------------------------------------
// The TMA load / expect-tx arrival issued by the lane whose `leader` is non-zero (the
// whole warp runs the producer loop, as the MMA warp does).
__device__ __forceinline__ void tma_load_2d_if(uint32_t leader, void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_if(uint32_t leader, uint64_t *bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)), "r"(bytes), "r"(leader)
               : "memory");
}

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
// 16 consecutive TMEM columns of this thread's lane (a warp writes its 32 lanes).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// elect.sync over the full warp: 1 in exactly one lane
__device__ __forceinline__ uint32_t elect_lane() {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(r));
  return r;
}
// tcgen05.mma (kind::f16, bf16 operands, f32 accumulator in TMEM; `accumulate` = 0
// overwrites D) and tcgen05.commit, issued by the lane whose `leader` is non-zero while
// every lane of the warp runs the same instruction stream: in warp-uniform code the
// operands stay warp-uniform values, and a 64-K stage's MMAs issued this way measured
// 10-15 % faster per GEMM than the same loop run by lane 0 alone.
__device__ __forceinline__ void umma_bf16_if(uint32_t leader, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
// ... with the A operand in TMEM (a_tmem: its first column, lane 0)
__device__ __forceinline__ void umma_bf16_ta_if(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void umma_commit_if(uint32_t leader, uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar)),
      "r"(leader)
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
//     (X tile: the f32 activations, N x 64 KB, when kXF; else the bf16 B tile);
//   A ring, kSA slots, filled by the dequantising warps:  [ NA bf16 A tiles |
//     the bf16 B tile when kXF ]  (each A / B tile is KB sub-tiles of 64 K).
// The load ring is as deep as shared memory allows (up to 16 slots); the A ring
// only needs to keep the tensor core fed.  kXF (token tiles of 16, and of 32 for one
// weight matrix): X arrives as f32 and is rounded to bf16 in the kernel, so no
// conversion kernel runs before it; the other tiles load the bf16 X a conversion
// kernel wrote (at 64 tokens, and 32 for the SwiGLU, the dequantising warps' extra
// rounding work cost more than that kernel: 6-8 % on those calls).  KB = 2 (the kXF
// tiles, n_in % 128 == 0): 128 K per stage, which halves the per-stage barrier and
// MMA-issue overhead that bounds the small-token pipeline.
// Whether a token tile of N rounds X to bf16 in the kernel (else it loads the bf16 X
// that x_to_bf16_kernel wrote into the workspace).
__host__ __device__ constexpr bool x_in_kernel(int N, int NA) { return N == 16 || (N == 32 && NA == 1); }

template <int FMT, int N, int NA, int KB>
struct GemmCfg {
  static constexpr bool kXF = x_in_kernel(N, NA);
  static_assert(KB == 1 || kXF, "two sub-blocks per stage only with the in-kernel X conversion");
  static constexpr uint32_t kQRowBytes = uint32_t(FMT == kWQ8 ? BK : BK / 2) * KB;  // a weight row's bytes per stage
  static constexpr uint32_t kQTileBytes = BM * kQRowBytes;
  static constexpr uint32_t kBSub = uint32_t(N) * 128;  // bf16 B tile of one sub-block
  static constexpr uint32_t kBTileBytes = KB * kBSub;
  static constexpr uint32_t kXTileBytes = kXF ? uint32_t(N) * BK * 4 * KB : kBTileBytes;
  static constexpr uint32_t kATile = KB * kATileBytes;
  static constexpr uint32_t kLoadSlot = round1k(NA * kQTileBytes + kXTileBytes);
  // Q8_0, one weight matrix, token tiles of 32 and of 64 and above: the bf16 A tiles live
  // in TMEM, written by the dequantising warps with tcgen05.st, which leaves shared memory
  // to the load ring (one more slot at 256-token tiles, twice the slots at 32) and takes
  // the A tiles' traffic off shared memory.  (The same for Q4_K measured no faster: its
  // rows then need one header load per thread; at 16 tokens it measured no faster either.)
  static constexpr bool kTA = FMT == kWQ8 && NA == 1 && (KB == 1 ? !kXF || N == 64 : N == 32);
  static constexpr uint32_t kASlot = kTA ? (kXF ? round1k(kBTileBytes) : 0u) : round1k(NA * kATile + (kXF ? kBTileBytes : 0u));
  // the two dequantising groups and the tensor core each hold a slot (two when they are large)
  static constexpr int kSA = kTA ? 3 : (kASlot > 40u * 1024u ? 2 : 3);
  static constexpr int kFit = int((227u * 1024u - 2048u - uint32_t(kSA) * kASlot) / kLoadSlot);
  static constexpr int kSL = kFit > 16 ? 16 : kFit;
  static constexpr uint32_t kACol = uint32_t(NA * N);  // kTA: A slot j at columns kACol + 32 KB j
  static constexpr uint32_t kCols = kACol + (kTA ? uint32_t(kSA) * 32u * KB : 0u);
  static constexpr uint32_t kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static constexpr size_t kRingBytes = size_t(kSL) * kLoadSlot + size_t(kSA) * kASlot;
  static constexpr size_t kPBytes = size_t(NA) * N * BM * 4;  // a split's partial tile (f32)
  static constexpr size_t kSmemBytes = 1024 + kRingBytes + 512;
  static_assert(kSL >= 2, "the load ring needs two slots");
  static_assert(kSmemBytes <= 227u * 1024u, "shared memory");
};

struct GemmArgs {
  const uint8_t *W[2];  // packed weights (gate and up for the SwiGLU)
  float *Y;
  int n_out, n_in, M;
  int st_per_split, split;  // K stages per split, splits (= the cluster size along z)
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

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

template <int FMT, int N, int NA, int KB>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
                   const __grid_constant__ CUtensorMap tm_x, const GemmArgs g, const Magic mg_param) {
  using C = GemmCfg<FMT, N, NA, KB>;
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
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int issued = 0;  // TMA stages the producer issued (drained before the CTA exits)
  const int tile_n = blockIdx.x, tile_m = blockIdx.y;
  const int n_in = g.n_in, n_out = g.n_out, M = g.M;
  const int nst = n_in / (BK * KB);  // K stages of the whole row
  const int kb0 = blockIdx.z * g.st_per_split;  // this split's first stage
  const int kb1 = min(kb0 + g.st_per_split, nst);
  const int nk = kb1 - kb0;
  auto qtile = [&](int s, int a) { return smem + s * C::kLoadSlot + a * C::kQTileBytes; };
  auto xtile = [&](int s) { return smem + s * C::kLoadSlot + NA * C::kQTileBytes; };
  auto atile = [&](int j, int a) { return aring + j * C::kASlot + a * C::kATile; };
  // the MMA's B operand of stage i: in the A slot (converted here) or the load slot (TMA)
  auto btile = [&](int i) {
    return C::kXF ? aring + (i % SA) * C::kASlot + (C::kTA ? 0u : NA * C::kATile) : xtile(i % SL);
  };
  constexpr int kQBox = int(C::kQRowBytes);  // inner TMA coordinate step of a weight tile per stage

  if (threadIdx.x == 0) {
    for (int i = 0; i < SL; ++i) {
      mbar_init(&lfull[i], 1);
      // kXF: only the dequantising group reads a load slot (one arrival per warp);
      // else the tensor core reads its B tile (one commit)
      mbar_init(&lempty[i], C::kXF ? kDequantWarps / 2 : 1);
    }
    for (int j = 0; j < SA; ++j) {
      mbar_init(&aready[j], kDequantWarps / 2);  // one arrival per warp of the stage's group
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
    {  // the whole warp runs the loop; one elected lane issues
      const uint32_t leader = elect_lane();
      if (leader) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q0)) : "memory");
        if (NA == 2) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q1)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      }
      __syncwarp();
      constexpr uint32_t kTx = NA * C::kQTileBytes + C::kXTileBytes;
      const int npre = nk < SL ? nk : SL;
      for (int i = 0; i < npre; ++i) {
        mbar_expect_tx_if(leader, &lfull[i], kTx);
        tma_load_2d_if(leader, qtile(i, 0), &tm_q0, (kb0 + i) * kQBox, tile_n * BM, &lfull[i]);
        if (NA == 2) tma_load_2d_if(leader, qtile(i, 1), &tm_q1, (kb0 + i) * kQBox, tile_n * BM, &lfull[i]);
      }
      pdl_wait();
      for (int i = 0; i < npre; ++i) tma_load_2d_if(leader, xtile(i), &tm_x, (kb0 + i) * BK * KB, tile_m * N, &lfull[i]);
      issued = npre;
      for (int i = npre; i < nk; ++i) {
        const int s = i % SL;
        if (!__all_sync(0xffffffffu, !*reinterpret_cast<volatile int *>(&s_abort) &&
                                         mbar_wait(&lempty[s], ((i / SL) + 1) & 1))) {
          s_abort = 1;
          break;
        }
        mbar_expect_tx_if(leader, &lfull[s], kTx);
        tma_load_2d_if(leader, qtile(s, 0), &tm_q0, (kb0 + i) * kQBox, tile_n * BM, &lfull[s]);
        if (NA == 2) tma_load_2d_if(leader, qtile(s, 1), &tm_q1, (kb0 + i) * kQBox, tile_n * BM, &lfull[s]);
        tma_load_2d_if(leader, xtile(s), &tm_x, (kb0 + i) * BK * KB, tile_m * N, &lfull[s]);
        issued = i + 1;
      }
    }
  } else if (warp == kDequantWarps + 1) {
    // ---------------- MMA issuer ----------------
    pdl_wait();
    {  // the whole warp runs the loop; one elected lane issues the MMAs and commits
      const uint32_t leader = elect_lane();
      constexpr uint32_t idesc = idesc_bf16_f32(BM, N);
      for (int i = 0; i < nk; ++i) {
        const int s = i % SL, j = i % SA;
        // kXF: A and B are both written by the dequantising group (aready covers them).
        // Else B is the load slot's X tile: it lands on the same barrier as the weight tiles,
        // which the group waited for before its arrival, so aready covers it too (one wait
        // less per stage in this thread, whose loop paces the larger token tiles)
        if (!__all_sync(0xffffffffu, mbar_wait(&aready[j], (i / SA) & 1))) {
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t b_base = smem_u32(btile(i));
        if constexpr (C::kTA) {
#pragma unroll
          for (int kb = 0; kb < KB; ++kb)
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)  // K 16 k .. 16 k + 15 of sub-block kb: 8 columns of the A slot
              umma_bf16_ta_if(leader, tmem, tmem + C::kACol + uint32_t(32 * KB * j + 32 * kb + 8 * k),
                              desc_kmajor_sw128(b_base + kb * C::kBSub + 32 * k), idesc, (i | kb | k) != 0);
        } else {
#pragma unroll
          for (int a = 0; a < NA; ++a) {
            const uint32_t a_base = smem_u32(atile(j, a));
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                umma_bf16_if(leader, tmem + uint32_t(a * N), desc_kmajor_sw128(a_base + kb * kATileBytes + 32 * k),
                             desc_kmajor_sw128(b_base + kb * C::kBSub + 32 * k), idesc, (i | kb | k) != 0);
          }
        }
        umma_commit_if(leader, &aempty[j]);  // the A slot (and the B tile in it) is free once these MMAs are done
        if (!C::kXF) umma_commit_if(leader, &lempty[s]);  // so is the load slot (its B tile)
      }
      umma_commit_if(leader, accum);
    }
  } else {
    // ---------------- dequantise, then epilogue ----------------
    // Two groups of 8 warps take alternate stages (group g: stages g, g + 2, ...), so
    // that one group's dequantisation overlaps the other's: a stage's work is a short
    // dependent chain (shared-memory load, conversion, store, proxy fence), and one
    // group alone leaves most issue slots empty.  The weights do not depend on the
    // previous kernel, so dequantisation starts at once; only the epilogue (which
    // writes Y) waits for it.
    bool ok = true;
    const int grp = warp >> 3;                        // dequantising group
    const int gt = threadIdx.x & (kGroupThreads - 1);  // thread within the group
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
        for (int t = gt; t < N * 8 * KB; t += kGroupThreads) {
          const int kb = t / (N * 8), r = (t >> 3) % N, c = t & 7;
          uint8_t *bt = btile(i) + kb * C::kBSub;
          const float4 v0 = *reinterpret_cast<const float4 *>(xs + r * BK * KB + kb * BK + 8 * c);
          const float4 v1 = *reinterpret_cast<const float4 *>(xs + r * BK * KB + kb * BK + 8 * c + 4);
          *reinterpret_cast<uint4 *>(bt + r * 128 + ((c ^ (r & 7)) << 4)) =
              make_uint4(pack_bf16x2(f2(v0.x, v0.y)), pack_bf16x2(f2(v0.z, v0.w)), pack_bf16x2(f2(v1.x, v1.y)),
                         pack_bf16x2(f2(v1.z, v1.w)));
        }
      }
    };
    // the end of a stage: every write of the warp fenced for the tensor core, then one arrival
    auto finish_stage = [&](int i) {
      convert_x(i);
      if constexpr (C::kTA) {
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");  // this thread's A writes are done
        tc_fence_before();
      }
      if constexpr (!C::kTA || C::kXF)  // the B tile written here (kXF) or the A tile, for the tensor core
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&aready[i % SA]);
        if (C::kXF) mbar_arrive(&lempty[i % SL]);  // the warp has read its part of the load slot
      }
    };
    if constexpr (FMT == kWQ8) {
      // thread: weight row gt % 128, block half = gt / 128 of each 64-K sub-block (32 quants,
      // one block scale)
      const int row = gt & (BM - 1);
      const int half = gt >> 7;
      const int grow = tile_n * BM + row;
      const unsigned short *d16[NA];
#pragma unroll
      for (int a = 0; a < NA; ++a)
        d16[a] = reinterpret_cast<const unsigned short *>(g.W[a] + int64_t(n_out) * n_in) + int64_t(grow) * (n_in / 32) +
                 half;
      // 16-byte chunk c of the row as the TMA swizzle stored it (64-byte rows: 64-byte
      // swizzle; 128-byte rows: 128-byte swizzle)
      auto qchunk = [&](int c) { return KB == 1 ? c ^ ((row >> 1) & 3) : c ^ (row & 7); };
      // block scales fetched four of this group's stages ahead into slot u, which the
      // stage four later reads (unrolled by 4: no register copy waits for a load);
      // sub-block kb of stage i is 64-K block (kb0 + i) * KB + kb, blocks 2 x + half
      auto scale_at = [&](int a, int i, int kb) { return __ldg(d16[a] + 2 * ((kb0 + i) * KB + kb)); };
      unsigned short dqa[4][NA][KB];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) dqa[u][a][kb] = grp + 2 * u < nk ? scale_at(a, grp + 2 * u, kb) : 0;
      for (int i0 = grp; i0 < nk && ok; i0 += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + 2 * u;
          if (i >= nk) break;
          const int s = i % SL, j = i % SA;
          float dsc[NA][KB];
#pragma unroll
          for (int a = 0; a < NA; ++a)
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
              dsc[a][kb] = __half2float(__ushort_as_half(dqa[u][a][kb]));
              dqa[u][a][kb] = i + 8 < nk ? scale_at(a, i + 8, kb) : 0;
            }
          // warp-uniform: the warp's lanes arrive together (one arrival per warp)
          if (!__all_sync(0xffffffffu, wait_slots(i))) {
            s_abort = 1;
            ok = false;
            break;
          }
          if constexpr (C::kTA) tc_fence_after();
#pragma unroll
          for (int a = 0; a < NA; ++a)
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
              const uint8_t *qt = qtile(s, a);
              uint8_t *at = C::kTA ? nullptr : atile(j, a) + kb * kATileBytes;
              const float2 dpair = f2(dsc[a][kb], dsc[a][kb]);
              uint32_t tw[16];  // kTA: the half's 32 bf16 weights, K order, two per column
#pragma unroll
              for (int pp = 0; pp < 2; ++pp) {
                const int part = 2 * half + pp;  // 16 quants: K 16 part .. 16 part + 15 of the sub-block
                const uint4 qv =
                    *reinterpret_cast<const uint4 *>(qt + row * C::kQRowBytes + (qchunk(4 * kb + part) << 4));
                const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
                uint32_t packed[8];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  float2 q01, q23;
                  s8x4_to_f2_sel(words[w], mg, q01, q23);
                  packed[2 * w] = pack_bf16x2(__fmul2_rn(q01, dpair));  // d*q exact in f32, rounded once
                  packed[2 * w + 1] = pack_bf16x2(__fmul2_rn(q23, dpair));
                }
                if constexpr (C::kTA) {
#pragma unroll
                  for (int w = 0; w < 8; ++w) tw[8 * pp + w] = packed[w];
                } else {
                  // two 16-byte bf16 chunks (K 16p..16p+7 and 16p+8..16p+15)
                  *reinterpret_cast<uint4 *>(at + row * 128 + (((2 * part) ^ (row & 7)) << 4)) =
                      make_uint4(packed[0], packed[1], packed[2], packed[3]);
                  *reinterpret_cast<uint4 *>(at + row * 128 + (((2 * part + 1) ^ (row & 7)) << 4)) =
                      make_uint4(packed[4], packed[5], packed[6], packed[7]);
                }
              }
              // kTA: row = TMEM lane 32 (warp % 4) + lane; K 32 half .. at column 16 half of the slot
              if constexpr (C::kTA)
                tmem_st16(tmem + (uint32_t((warp & 3) * 32) << 16) + C::kACol + uint32_t(32 * KB * j + 32 * kb + 16 * half),
                          tw);
            }
          finish_stage(i);
        }
    } else {
      // Q4_K: warp w of the group takes rows 16w..16w+15, two threads per row, one
      // 32-weight sub-block (16 bytes) of each 64-K block: a warp reads 512 bytes of
      // the tile per 64-K block
      const int row = (warp & 7) * 16 + (lane >> 1);
      const int part = lane & 1;
      const int grow = tile_n * BM + row;
      // 16-byte chunk c of the row as stored (32-byte rows: no swizzle; 64-byte rows:
      // 64-byte swizzle)
      auto qchunk = [&](int c) { return KB == 1 ? c : c ^ ((row >> 1) & 3); };
      const uint4 *hdr[NA];  // the row's superblock headers
#pragma unroll
      for (int a = 0; a < NA; ++a)
        hdr[a] = reinterpret_cast<const uint4 *>(g.W[a] + int64_t(n_out) * (n_in / 2)) + int64_t(grow) * (n_in / 256);
      // the header of the current superblock, and of the next one fetched ahead
      const int nsb = n_in / 256;
      uint4 hcur[NA], hnext[NA];
      int cur_sb = ((kb0 + grp) * KB) >> 2;
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        hcur[a] = __ldg(hdr[a] + cur_sb);
        hnext[a] = cur_sb + 1 < nsb ? __ldg(hdr[a] + cur_sb + 1) : hcur[a];
      }
      for (int i = grp; i < nk; i += 2) {
        const int s = i % SL, jj = i % SA;
        const int k64 = (kb0 + i) * KB;  // the stage's first 64-K block (a stage stays in one superblock)
        if ((k64 >> 2) != cur_sb) {      // entering the next superblock
          ++cur_sb;
#pragma unroll
          for (int a = 0; a < NA; ++a) {
            hcur[a] = hnext[a];
            hnext[a] = cur_sb + 1 < nsb ? __ldg(hdr[a] + cur_sb + 1) : hcur[a];
          }
        }
        float2 dm[NA][KB];  // (d*sc_j, dmin*m_j) of sub-block j = 2 (64-K block % 4) + part
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) dm[a][kb] = q4k_header_scale(hcur[a], 2 * ((k64 + kb) & 3) + part);
        if (!__all_sync(0xffffffffu, wait_slots(i))) {
          s_abort = 1;
          ok = false;
          break;
        }
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            const uint4 qv =
                *reinterpret_cast<const uint4 *>(qtile(s, a) + row * C::kQRowBytes + (qchunk(2 * kb + part) << 4));
            uint8_t *at = atile(jj, a) + kb * kATileBytes;
            const float2 D = f2(dm[a][kb].x, dm[a][kb].x), Dm = f2(-dm[a][kb].y, -dm[a][kb].y);
            const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // 16 weights -> two 16-byte chunks of the A row
              uint32_t packed[8];
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                float2 q[4];
                u4x8_to_f2(words[2 * h + w], mg, q);
#pragma unroll
                for (int p = 0; p < 4; ++p) packed[4 * w + p] = pack_bf16x2(__ffma2_rn(D, q[p], Dm));  // RN(D q - Dm)
              }
              const int c = 4 * part + 2 * h;  // 16-byte chunk of K 8c .. 8c + 15
              *reinterpret_cast<uint4 *>(at + row * 128 + ((c ^ (row & 7)) << 4)) =
                  make_uint4(packed[0], packed[1], packed[2], packed[3]);
              *reinterpret_cast<uint4 *>(at + row * 128 + (((c + 1) ^ (row & 7)) << 4)) =
                  make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
          }
        finish_stage(i);
      }
    }
    pdl_wait();
    if (ok && mbar_wait(accum, 0)) {
      tc_fence_after();
      const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
      const int m0 = tile_m * N;
      const int erow = tile_n * BM + (warp & 3) * 32 + lane;  // this thread's output row (TMEM lane)
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
        // split-K: this split's partial tile goes to its own shared memory (the rings
        // are idle now: every stage was consumed and every MMA completed), [a][token][row]
        if constexpr (C::kPBytes <= C::kRingBytes) {  // else the host never splits K
          float *P = reinterpret_cast<float *>(smem);
          const int prow = (warp & 3) * 32 + lane;
#pragma unroll 1
          for (int c0 = (warp >> 2) * 16; c0 < N; c0 += 16 * (kDequantWarps / 4)) {
            uint32_t r[NA][16];
#pragma unroll
            for (int a = 0; a < NA; ++a) tmem_ld16(tmem + lane_base + uint32_t(a * N + c0), r[a]);
#pragma unroll
            for (int a = 0; a < NA; ++a)
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) P[(a * N + c0 + jj) * BM + prow] = __uint_as_float(r[a][jj]);
          }
        }
      }
    } else {
      s_abort = 1;
    }
  }

  if (g.split > 1) {
    // The K splits of a tile form one thread-block cluster: after a cluster barrier every
    // split's partial tile is readable through distributed shared memory, and split z
    // writes its share of the tile's tokens, adding the partials in split order (so the
    // result does not depend on which CTA finished first).  Every thread of every CTA
    // takes both barriers, also after an abort; then no Y is written for the tile.
    cluster_sync_all();
    if (warp < kDequantWarps) {
      const int split = g.split, z = blockIdx.z;
      bool all_ok = true;
      for (int r = 0; r < split; ++r) all_ok = all_ok && ld_cluster_s32(cluster_addr(&s_abort, uint32_t(r))) == 0;
      if (all_ok && C::kPBytes <= C::kRingBytes) {
        const float *P = reinterpret_cast<const float *>(smem);
        const int c_lo = N * z / split, c_hi = N * (z + 1) / split;  // this split's tokens of the tile
        // warp w takes tokens c_lo + w, c_lo + w + 16, ...; lane l rows 4 l .. 4 l + 3 of the
        // tile (16-byte loads from every split, all in flight before the sums)
        const int erow = tile_n * BM + 4 * lane;
        const int m0 = tile_m * N;
        uint32_t base[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) base[r] = cluster_addr(P, uint32_t(r < split ? r : 0));
#pragma unroll 1
        for (int c = c_lo + warp; c < c_hi; c += kDequantWarps) {
          float4 acc[NA];
#pragma unroll
          for (int a = 0; a < NA; ++a) {
            float4 v[8];
            const uint32_t off = uint32_t(((a * N + c) * BM + 4 * lane) * 4);
#pragma unroll
            for (int r = 0; r < 8; ++r) v[r] = r < split ? ld_cluster_f32x4(base[r] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
            acc[a] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if (r < split) {
                acc[a].x += v[r].x;
                acc[a].y += v[r].y;
                acc[a].z += v[r].z;
                acc[a].w += v[r].w;
              }
          }
          const int m = m0 + c;
          if (m < M && QDQ_GUARD(erow + 4 <= n_out, QDQ_CHECK_OUT)) {
            float4 y = acc[0];
            if (NA == 2) {
              y.x = y.x / (1.0f + expf(-y.x)) * acc[NA - 1].x;
              y.y = y.y / (1.0f + expf(-y.y)) * acc[NA - 1].y;
              y.z = y.z / (1.0f + expf(-y.z)) * acc[NA - 1].z;
              y.w = y.w / (1.0f + expf(-y.w)) * acc[NA - 1].w;
            }
            *reinterpret_cast<float4 *>(g.Y + int64_t(m) * n_out + erow) = y;  // n_out % 128 == 0, Y 16-byte aligned
          }
        }
      } else if (threadIdx.x == 0) {
        s_abort = 1;
      }
    }
    cluster_sync_all();  // no CTA leaves while another may still read its shared memory
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

// X (f32, M x n_in) -> bf16 workspace.
__global__ void __launch_bounds__(256) x_to_bf16_kernel(const float4 *__restrict__ X, uint2 *__restrict__ xb,
                                                        int64_t n4) {
  pdl_launch_dependents();
  pdl_wait();  // the workspace may still be in use by the previous kernel
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += stride) {
    const float4 v = X[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    xb[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
  }
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

// The token tile for up to 128 tokens; more tokens choose among 128, 192 and 256 (plan_gemm).
int token_tile(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

// Clusters of cz CTAs (one CTA per SM, as every GEMM instantiation takes) that can be
// resident at once on the current device, measured once per size; 0 if unknown.
int resident_clusters(int cz) {
  static std::atomic<int> cache[9];  // per cluster size (0: not yet measured, -1: unknown)
  if (cz < 2 || cz > 8) return 0;
  int mc = cache[cz].load(std::memory_order_relaxed);
  if (mc == 0) {
    using C = GemmCfg<kWQ8, 256, 1, 1>;
    auto kern = gemm_tc_kernel<kWQ8, 256, 1, 1>;
    if (allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(C::kSmemBytes)) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, unsigned(cz));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = unsigned(cz);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&mc, kern, &cfg) != cudaSuccess || mc < 1) {
      (void)cudaGetLastError();
      mc = -1;
    }
    cache[cz].store(mc, std::memory_order_relaxed);
  }
  return mc > 0 ? mc : 0;
}

// Whether the split-K partial tile fits the CTA's rings (else K is never split).
template <int FMT, int NA>
bool splittable(int N) {
  switch (N) {
    case 16: return GemmCfg<FMT, 16, NA, 2>::kPBytes <= GemmCfg<FMT, 16, NA, 2>::kRingBytes;
    case 32: {
      using C32 = GemmCfg<FMT, 32, NA, x_in_kernel(32, NA) ? 2 : 1>;
      return C32::kPBytes <= C32::kRingBytes;
    }
    case 64: return GemmCfg<FMT, 64, NA, 1>::kPBytes <= GemmCfg<FMT, 64, NA, 1>::kRingBytes;
    case 128: return GemmCfg<FMT, 128, NA, 1>::kPBytes <= GemmCfg<FMT, 128, NA, 1>::kRingBytes;
    case 192: return GemmCfg<FMT, 192, NA, 1>::kPBytes <= GemmCfg<FMT, 192, NA, 1>::kRingBytes;
    default: return GemmCfg<FMT, 256, NA, 1>::kPBytes <= GemmCfg<FMT, 256, NA, 1>::kRingBytes;
  }
}

// Launch shape and workspace of one GEMM call (the workspace holds only the bf16
// copy of X, for the token tiles that do not round X in the kernel).
struct GemmPlan {
  int N, KB, ntile_n, ntile_m, nst;
  int split, st_per;  // K splits (the cluster size along z) and K stages per split
  size_t xb_bytes;
};
// The shape for token tile N: K is split when the tiles alone cannot fill the SMs, at
// most 8 ways (a portable cluster) and only as far as every tile's cluster stays
// resident at once (one wave).
template <int FMT, int NA>
GemmPlan plan_for(int N, int M, int n_out, int n_in, int sm_count) {
  GemmPlan p;
  p.N = N;
  // 64-K sub-blocks per stage: two for token tiles up to 32 (at 64 the larger stage
  // leaves too few load slots and measured slower)
  p.KB = x_in_kernel(p.N, NA) && n_in % (2 * BK) == 0 ? 2 : 1;
  p.ntile_n = n_out / BM;
  p.ntile_m = (M + p.N - 1) / p.N;
  p.nst = n_in / (BK * p.KB);
  const int tiles = p.ntile_n * p.ntile_m;
  int split = sm_count / tiles;
  if (split > 8) split = 8;
  if (split > p.nst) split = p.nst;
  if (split < 1 || !splittable<FMT, NA>(p.N)) split = 1;
  while (split > 1 && resident_clusters(split) < tiles) --split;
  p.st_per = (p.nst + split - 1) / split;
  p.split = (p.nst + p.st_per - 1) / p.st_per;  // every split gets at least one stage
  p.xb_bytes = x_in_kernel(p.N, NA) ? 0 : (size_t(M) * n_in * 2 + 255) / 256 * 256;
  return p;
}
// Above 128 tokens the token tile is the one of 128, 192 and 256 with the least
// estimated time: waves of CTAs x K stages per CTA x a stage's time, which the
// measurements put at about 0.35 us + 1.2 ns per token of the tile.  (8192 -> 3072
// at 512 tokens: 24 row tiles, so 256-token tiles leave 96 CTAs and 192-token tiles
// 144; 3072 -> 8192 at 512 tokens: 64 row tiles, where 192-token tiles would take
// two waves.)
template <int FMT, int NA>
GemmPlan plan_gemm(int M, int n_out, int n_in, int sm_count) {
  if (M <= 128) return plan_for<FMT, NA>(token_tile(M), M, n_out, n_in, sm_count);
  GemmPlan best{};
  double best_cost = 0.0;
  for (const int N : {256, 192, 128}) {
    const GemmPlan p = plan_for<FMT, NA>(N, M, n_out, n_in, sm_count);
    const int ctas = p.ntile_n * p.ntile_m * p.split;
    const int waves = (ctas + sm_count - 1) / sm_count;
    const double cost = double(waves) * p.st_per * (0.35 + 0.0012 * N);
    if (best.N == 0 || cost < best_cost * (1.0 - 1e-9)) {
      best = p;
      best_cost = cost;
    }
  }
  return best;
}

// Launch with programmatic dependent launch and a (1, 1, cz) thread-block cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_z(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cz,
                             Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = opt_pdl() ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = unsigned(cz);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int FMT, int N, int NA, int KB>
int launch_tile(const uint8_t *const W[2], const float *X, float *Y, void *ws, int n_out, int n_in, int M,
                const GemmPlan &p, cudaStream_t s, const DeviceInfo &di) {
  using C = GemmCfg<FMT, N, NA, KB>;
  auto kern = gemm_tc_kernel<FMT, N, NA, KB>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), int(C::kSmemBytes));
  if (e != cudaSuccess) return fail_cuda(e);

  const int split = p.split, st_per = p.st_per;

  CUtensorMap tm_q[2], tm_x;
  for (int a = 0; a < 2; ++a) {
    const uint8_t *w = W[a < NA ? a : 0];
    // weight tile rows of kQRowBytes (Q8_0: 64 or 128; Q4_K: 32 or 64), swizzled to match
    const uint64_t row_bytes = FMT == kWQ8 ? uint64_t(n_in) : uint64_t(n_in / 2);
    const CUtensorMapSwizzle sw = C::kQRowBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : C::kQRowBytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    const bool okq = encode_2d(&tm_q[a], CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t *>(w), row_bytes,
                               uint64_t(n_out), row_bytes, C::kQRowBytes, BM, sw);
    if (!okq) return QDQ_ERR_UNSUPPORTED;
  }

  GemmArgs g{};
  g.W[0] = W[0];
  g.W[1] = W[NA - 1];
  g.Y = Y;
  g.n_out = n_out;
  g.n_in = n_in;
  g.M = M;
  g.st_per_split = st_per;
  g.split = split;

  if (C::kXF) {
    // X is read as f32 and rounded to bf16 inside the GEMM
    if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float *>(X), uint64_t(n_in), uint64_t(M),
                   uint64_t(n_in) * 4, BK * KB, N, CU_TENSOR_MAP_SWIZZLE_NONE))
      return QDQ_ERR_UNSUPPORTED;
  } else {
    // conversion of X into the workspace
    uint8_t *xb = static_cast<uint8_t *>(ws);
    if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, uint64_t(n_in), uint64_t(M), uint64_t(n_in) * 2, BK,
                   N, CU_TENSOR_MAP_SWIZZLE_128B))
      return QDQ_ERR_UNSUPPORTED;
    const int64_t n4 = int64_t(M) * n_in / 4;
    int cgrid = int((n4 + 255) / 256);
    if (cgrid > di.sm_count * 8) cgrid = di.sm_count * 8;
    if (cgrid < 1) cgrid = 1;
    e = launch(x_to_bf16_kernel, dim3(cgrid), dim3(256), 0, s, reinterpret_cast<const float4 *>(X),
               reinterpret_cast<uint2 *>(xb), n4);
    if (e != cudaSuccess) return fail_cuda(e);
  }

  const dim3 grid(p.ntile_n, p.ntile_m, split);
  e = split > 1 ? launch_cluster_z(kern, grid, dim3(kThreads), C::kSmemBytes, s, split, tm_q[0], tm_q[1], tm_x, g,
                                   make_magic())
                : launch(kern, grid, dim3(kThreads), C::kSmemBytes, s, tm_q[0], tm_q[1], tm_x, g, make_magic());
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
  const GemmPlan p = plan_gemm<FMT, NA>(M, n_out, n_in, di.sm_count);
  switch (p.N * 2 + p.KB - 1) {
    case 32: return launch_tile<FMT, 16, NA, 1>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 33: return launch_tile<FMT, 16, NA, 2>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 64: return launch_tile<FMT, 32, NA, 1>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 65:
      if constexpr (x_in_kernel(32, NA)) return launch_tile<FMT, 32, NA, 2>(W, X, Y, ws, n_out, n_in, M, p, s, di);
      return QDQ_ERR_UNSUPPORTED;  // not planned
    case 128: return launch_tile<FMT, 64, NA, 1>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 256: return launch_tile<FMT, 128, NA, 1>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    case 384: return launch_tile<FMT, 192, NA, 1>(W, X, Y, ws, n_out, n_in, M, p, s, di);
    default: return launch_tile<FMT, 256, NA, 1>(W, X, Y, ws, n_out, n_in, M, p, s, di);
  }
}

}  // namespace

size_t gemm_workspace_bytes(int M, int n_out, int n_in, int na) {
  // the bf16 copy of X (every token tile but those that round X in the kernel: token_tile(M)
  // is 16 up to 16 tokens and 32 up to 32), else 256 bytes reserved
  (void)n_out;
  const bool conv = !x_in_kernel(token_tile(M), na);
  const size_t xb = conv ? (size_t(M) * n_in * 2 + 255) / 256 * 256 : 0;
  return xb > 256 ? xb : 256;
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

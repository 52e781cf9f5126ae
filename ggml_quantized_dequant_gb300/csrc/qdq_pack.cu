// One-time repack of GGML blocks into the device plane layout, and the
// dequantisation kernels used to verify it bit for bit.
//
// "Module cuda_lane", Functions: preload_q4k_soa_weights -- the pages upload
// and lay out quantised weights once at plan build so that decode never
// reformats them; here the same step rewrites the 34-byte Q8_0 blocks and the
// 144-byte Q4_K superblocks (neither is 16-byte aligned) into planes that the
// GEMV kernels read with aligned 128-bit loads.  Byte counts are unchanged.
#include "qdq_internal.cuh"

namespace qdq {
namespace {

constexpr int kPackThreads = 256;

__device__ __forceinline__ uint32_t load_u32_bytes(const uint8_t *p) {
  return uint32_t(p[0]) | (uint32_t(p[1]) << 8) | (uint32_t(p[2]) << 16) | (uint32_t(p[3]) << 24);
}

// One thread per Q8_0 block: 2 bytes of scale go to the d plane, 32 quant
// bytes to the q plane (block i of the matrix lands at q plane offset 32*i).
__global__ void q8_0_pack_kernel(const uint8_t *__restrict__ g, uint8_t *__restrict__ packed,
                                 int64_t n_blocks, int64_t q_plane_bytes) {
  uint16_t *dplane = reinterpret_cast<uint16_t *>(packed + q_plane_bytes);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_blocks;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint8_t *src = g + i * 34;
    dplane[i] = uint16_t(src[0] | (src[1] << 8));
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = load_u32_bytes(src + 2 + 4 * k);
    uint4 *dst = reinterpret_cast<uint4 *>(packed + i * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// 6-bit scale/min j of a GGML Q4_K superblock from its 12 packed bytes s[]:
// bytes 0..3 hold sc0..3 (low 6 bits) and the top 2 bits of sc4..7; bytes
// 4..7 hold m0..3 and the top 2 bits of m4..7; bytes 8..11 hold the low
// nibbles of sc4..7 (low half) and of m4..7 (high half).
__device__ __forceinline__ void ggml_q4k_scale_min(const uint8_t *s, int j, uint32_t &sc, uint32_t &m) {
  if (j < 4) {
    sc = s[j] & 63u;
    m = s[j + 4] & 63u;
  } else {
    sc = (s[j + 4] & 0x0Fu) | ((uint32_t(s[j - 4]) >> 6) << 4);
    m = (uint32_t(s[j + 4]) >> 4) | ((uint32_t(s[j]) >> 6) << 4);
  }
}

// One thread per Q4_K superblock.  Quants: GGML stores weight 64c+l (l<32) in
// the low nibble and weight 64c+32+l in the high nibble of byte 32c+l; the
// packed plane stores weight e in nibble (e & 1) of byte e/2.  Header record:
// d | dmin << 16, then the eight (sc_j, m_j) pairs as 12-bit fields.
__global__ void q4k_pack_kernel(const uint8_t *__restrict__ g, uint8_t *__restrict__ packed,
                                int64_t n_super, int64_t q_plane_bytes) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_super;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint8_t *src = g + i * 144;
    const uint8_t *s = src + 4;
    const uint8_t *qs = src + 16;

    uint32_t out[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) out[t] = 0;
#pragma unroll 4
    for (int e = 0; e < 256; ++e) {
      const int c = e >> 6, l = e & 63;
      const uint32_t byte = qs[32 * c + (l & 31)];
      const uint32_t q = (l < 32) ? (byte & 0x0Fu) : (byte >> 4);
      out[e >> 3] |= q << (4 * (e & 7));
    }
    uint4 *dst = reinterpret_cast<uint4 *>(packed + i * 128);
#pragma unroll
    for (int t = 0; t < 8; ++t) dst[t] = make_uint4(out[4 * t], out[4 * t + 1], out[4 * t + 2], out[4 * t + 3]);

    uint64_t lo = 0;   // bits 0..63 of the 96-bit field
    uint32_t hi = 0;   // bits 64..95
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t sc, m;
      ggml_q4k_scale_min(s, j, sc, m);
      const uint64_t f = uint64_t(sc | (m << 6));
      const int bit = 12 * j;
      if (bit + 12 <= 64) {
        lo |= f << bit;
      } else if (bit >= 64) {
        hi |= uint32_t(f << (bit - 64));
      } else {  // straddles bit 64
        lo |= f << bit;
        hi |= uint32_t(f >> (64 - bit));
      }
    }
    const uint32_t h0 = uint32_t(src[0]) | (uint32_t(src[1]) << 8) | (uint32_t(src[2]) << 16) |
                        (uint32_t(src[3]) << 24);
    uint4 *hdr = reinterpret_cast<uint4 *>(packed + q_plane_bytes + i * 16);
    *hdr = make_uint4(h0, uint32_t(lo), uint32_t(lo >> 32), hi);
  }
}

// Q8_0 dequant: w = d * q, exact in f32.  One thread per 16 weights.
__global__ void q8_0_dequant_kernel(const uint8_t *__restrict__ W, float *__restrict__ out, int64_t n_chunks,
                                    int64_t q_plane_bytes) {
  const __half *dplane = reinterpret_cast<const __half *>(W + q_plane_bytes);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_chunks;
       i += int64_t(gridDim.x) * blockDim.x) {
    const float d = __half2float(dplane[i >> 1]);
    const int8_t *q = reinterpret_cast<const int8_t *>(W + i * 16);
#pragma unroll
    for (int k = 0; k < 16; ++k) out[i * 16 + k] = __fmul_rn(d, float(q[k]));
  }
}

// Q4_K dequant: w = RN_f32(d*sc_j*q - dmin*m_j).  d*sc_j, (d*sc_j)*q and
// dmin*m_j are exact in f32; the subtraction is the one rounding.
__global__ void q4k_dequant_kernel(const uint8_t *__restrict__ W, float *__restrict__ out, int64_t n_sub,
                                   int64_t q_plane_bytes) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_sub;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t sb = i >> 3;
    const int j = int(i & 7);
    const uint4 h = *reinterpret_cast<const uint4 *>(W + q_plane_bytes + sb * 16);
    const uint64_t lo = uint64_t(h.y) | (uint64_t(h.z) << 32);
    const int bit = 12 * j;
    uint32_t f;
    if (bit + 12 <= 64) f = uint32_t(lo >> bit) & 0xFFFu;
    else if (bit >= 64) f = (h.w >> (bit - 64)) & 0xFFFu;
    else f = (uint32_t(lo >> bit) | (h.w << (64 - bit))) & 0xFFFu;
    const float sc = float(f & 63u), m = float(f >> 6);
    const float d = __half2float(__ushort_as_half(uint16_t(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(uint16_t(h.x >> 16)));
    const float D = __fmul_rn(d, sc), M = __fmul_rn(dmin, m);
    const uint4 qv = *reinterpret_cast<const uint4 *>(W + i * 16);
    const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float q = float((words[k >> 3] >> (4 * (k & 7))) & 0xFu);
      out[i * 32 + k] = __fsub_rn(__fmul_rn(D, q), M);
    }
  }
}

int grid_for(int64_t items) {
  int64_t g = (items + kPackThreads - 1) / kPackThreads;
  if (g > 65535LL * 16) g = 65535LL * 16;
  return int(g < 1 ? 1 : g);
}

}  // namespace

int launch_q8_0_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t s) {
  const int64_t nblk = int64_t(n_out) * (n_in / 32);
  q8_0_pack_kernel<<<grid_for(nblk), kPackThreads, 0, s>>>(static_cast<const uint8_t *>(ggml),
                                                            static_cast<uint8_t *>(packed), nblk,
                                                            int64_t(n_out) * n_in);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

int launch_q4k_pack(const void *ggml, void *packed, int n_out, int n_in, cudaStream_t s) {
  const int64_t nsb = int64_t(n_out) * (n_in / 256);
  q4k_pack_kernel<<<grid_for(nsb), kPackThreads, 0, s>>>(static_cast<const uint8_t *>(ggml),
                                                          static_cast<uint8_t *>(packed), nsb,
                                                          int64_t(n_out) * (n_in / 2));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

int launch_q8_0_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t s) {
  const int64_t n = int64_t(n_out) * (n_in / 16);
  q8_0_dequant_kernel<<<grid_for(n), kPackThreads, 0, s>>>(static_cast<const uint8_t *>(W), out, n,
                                                            int64_t(n_out) * n_in);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

int launch_q4k_dequant(const void *W, float *out, int n_out, int n_in, cudaStream_t s) {
  const int64_t n = int64_t(n_out) * (n_in / 32);
  q4k_dequant_kernel<<<grid_for(n), kPackThreads, 0, s>>>(static_cast<const uint8_t *>(W), out, n,
                                                           int64_t(n_out) * (n_in / 2));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QDQ_OK : fail_cuda(e);
}

}  // namespace qdq

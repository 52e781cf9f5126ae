// Allocation-free entry point: the Q4_K FFN block with residual, its
// intermediate activation vector kept in a fixed device array of this library
// instead of a caller-provided workspace.
//
// Who needs it: callers that may not allocate device memory themselves -- for
// example a plug-in inside a host application whose memory manager owns all of
// the GPU's memory through its own pool (a cudaMalloc there bypasses the pool's
// accounting and can fail once the pool has reserved the free memory), or a
// decode loop that must not pay for cudaMalloc/cudaFree, which can block on
// the device.  Such a caller passes only its inputs and outputs.
//
// The array lives in this file's device memory image, so every GPU that loads
// the library holds it (QDQ_NOALLOC_FFN_MAX_MID floats) until the process ends.
// Host code cannot use the array's name as a device address, so the first call
// on each device looks the address up with cudaGetSymbolAddress while that
// device is current and caches it; that first call should come before any
// stream capture.  The computation itself is the ordinary FFN path.
#include <mutex>

#include "qdq_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

// mid = silu(Wg x) * (Wu x) for up to QDQ_NOALLOC_FFN_MAX_MID floats
static __device__ __align__(256) float g_ffn_mid_scratch[QDQ_NOALLOC_FFN_MAX_MID];

std::mutex g_scratch_mu;
float *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_on_current_device(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return qdq::fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return QDQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ffn_mid_scratch);
    if (e != cudaSuccess) return qdq::fail_cuda(e);
    g_scratch_addr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_addr[dev];
  return QDQ_OK;
}

}  // namespace

extern "C" int qdq_q4k_ffn_residual_noalloc(const void *Wg, const void *Wu, const void *Wd, const float *x,
                                            const float *residual, float *out, int n_embd, int n_ff, int batch,
                                            cudaStream_t stream) {
  // the intermediate vector is batch x n_ff floats; it must fit the fixed array
  if (batch > 0 && n_ff > 0 && int64_t(batch) * n_ff > int64_t(QDQ_NOALLOC_FFN_MAX_MID)) return QDQ_ERR_SCRATCH;
  // then the same argument checks as the workspace entry point, all before any CUDA call
  int rc = qdq::check_ffn_residual(Wg, Wu, Wd, x, residual, out, nullptr, n_embd, n_ff, batch);
  if (rc != QDQ_OK) return rc;
  float *mid = nullptr;
  rc = scratch_on_current_device(&mid);
  if (rc != QDQ_OK) return rc;
  // Every element of mid is written by the SwiGLU kernel before the down
  // projection reads it, so nothing left from an earlier call needs clearing.
  // All calls share the one array: calls that overlap on the GPU race on it.
  return qdq_q4k_ffn_residual(Wg, Wu, Wd, x, residual, out, mid, n_embd, n_ff, batch, stream);
}

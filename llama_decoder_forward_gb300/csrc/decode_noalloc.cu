// decode_noalloc.cu - smol_decode_step_noalloc: the decode step with its
// scratch memory in a fixed device array owned by the library, for callers
// that cannot hand the library a workspace (see include/smol.h), and
// smol_decode_noalloc_status, which reads the status word kept in that array.
#include <mutex>

#include "common.cuh"

#define SMOL_API extern "C" __attribute__((visibility("default")))

namespace {

// Largest decode workspace served without a caller buffer.  The decode step
// on B sequences needs smol_workspace_bytes(cfg, SMOL_OP_DECODE, B, 1) bytes
// (about 5.1 MiB for SmolLM2-135M at B = 64 with max_pos 8192; most of it is
// the attention partials, B * H * 32 * hd fp32 values).
constexpr size_t kStaticWsBytes = 8u << 20;

// One copy exists on every device that loads the library, for the life of
// the process.  Calls share it: each call overwrites what the previous one
// left, and the decode step clears the parts that must start at zero itself.
// Its first word is the status word that the kernels' bounded waits write.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticWsBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device.  In host code the
// symbol's name is only a host-side handle, so the address is looked up with
// that device current.  Outside stream capture it is looked up on every call,
// so that a module reloaded after cudaDeviceReset is found at its new address;
// while `stream` is capturing, the address found by the last uncaptured call
// on this device is used (the lookup may load the module, which capture
// forbids), and a device never called before capture is refused.
int scratch_address(cudaStream_t stream, void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMOL_ERR_DEVICE;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SMOL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) return SMOL_ERR_CUDA;
    g_scratch_addr[dev] = p;
  } else if (!g_scratch_addr[dev]) {
    return SMOL_ERR_INVALID_ARG;
  }
  *out = g_scratch_addr[dev];
  return SMOL_OK;
}

}  // namespace

SMOL_API int smol_decode_step_noalloc(const smol_config *cfg, const void *packed, const int32_t *ids,
                                      const int32_t *cache_len, int B, const void *k_cache,
                                      const void *v_cache, int S_max, void *k_new, void *v_new,
                                      void *logits, void *stream) {
  const size_t need = smol_workspace_bytes(cfg, SMOL_OP_DECODE, B, 1);
  if (need > kStaticWsBytes) return SMOL_ERR_WORKSPACE;
  void *ws = nullptr;
  const int rc = scratch_address(static_cast<cudaStream_t>(stream), &ws);
  if (rc != SMOL_OK) return rc;
  return smol_decode_step(cfg, packed, ids, cache_len, B, k_cache, v_cache, S_max, k_new, v_new,
                          logits, ws, kStaticWsBytes, stream);
}

SMOL_API int smol_decode_noalloc_status(void *stream) {
  void *ws = nullptr;
  const int rc = scratch_address(static_cast<cudaStream_t>(stream), &ws);
  if (rc != SMOL_OK) return rc;
  return smol_workspace_status(ws, stream);
}

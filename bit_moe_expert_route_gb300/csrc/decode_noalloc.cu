// Batch-1 decode for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc: code that runs inside a
// host framework whose memory pool owns all device memory (a plug-in or
// custom op in someone else's runtime), and latency-critical serving loops
// where an allocation's implicit synchronisation or pool growth is not
// acceptable. moe_decode_gemv_w4_noalloc lets them run the decode path
// without passing a workspace: its scratch (router logits, top-k selection,
// SwiGLU activations, status words) lives in the array below, which is part
// of the library's device code. Every GPU that loads this library holds its
// own copy of the array until the process exits.
//
// The call forwards to moe_decode_gemv_w4 with this array as the workspace, so
// the kernels and the argument checks are the same ones.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 256 * 1024;

// The built-in scratch. In host code this name is only a stand-in for the
// symbol, not a device address: the device address comes from
// cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device; looked up once
// per device (the lookup may load this library's device code onto the device).
int scratch_on_current_device(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_decode_gemv_w4_noalloc(const uint16_t* x, const moe_weights_t* w,
                                          const moe_shape_t* shape, uint16_t* out,
                                          void* stream) {
  // the same argument checks as moe_decode_gemv_w4 first, so an unsupported
  // shape reads as MOE_ERR_SHAPE here too; then the scratch's size limit
  int rc = moe::decode_args_status(x, w, shape, out);
  if (rc != MOE_OK) return rc;
  if (moe_decode_workspace_bytes(shape) > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((rc = scratch_on_current_device(&scratch)) != MOE_OK) return rc;
  return moe_decode_gemv_w4(x, w, shape, out, scratch, kNoAllocScratchBytes, stream);
}

extern "C" int moe_decode_noalloc_device_status(void* stream, int32_t* device_status) {
  if (!device_status) return MOE_ERR_NULL;
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_get_device_status(scratch, stream, device_status);
}

extern "C" int moe_decode_noalloc_reset(void* stream) {
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  if (cudaMemsetAsync(scratch, 0, kNoAllocScratchBytes, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

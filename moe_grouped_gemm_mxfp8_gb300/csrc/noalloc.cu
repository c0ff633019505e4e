// Allocation-free form of the operator, for callers that must not allocate
// device memory themselves: the scratch space the kernels need lives in one
// file-scope device array that every GPU loading the library holds until the
// process exits.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "gmmfr.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

// Device scratch shared by every call of the allocation-free entry point.
// In host code this name is only a stand-in for the symbol: its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

gmmfr_status cuda_error(const char* what, cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return gmmfr::record_error(GMMFR_ERR_CUDA, msg);
}

// Device address of the scratch array on the current device.  Outside stream capture it is
// looked up on every call (a host-side table lookup), so that it is right again after the
// device's context has been destroyed and re-created; during capture, where a lookup could
// load the module inside the captured region, the address of an earlier call is used.
gmmfr_status scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return gmmfr::record_error(GMMFR_ERR_UNSUPPORTED, "device index above 63");
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_error("cudaStreamIsCapturing", e);
  std::lock_guard<std::mutex> lk(g_mu);
  if (cap != cudaStreamCaptureStatusNone) {
    if (!g_scratch_ptr[dev])
      return gmmfr::record_error(GMMFR_ERR_UNSUPPORTED,
                                 "the static-scratch entry point was first called inside a stream capture; make one "
                                 "call on this device before capturing");
    *out = g_scratch_ptr[dev];
    return GMMFR_OK;
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_static_scratch);
  if (e != cudaSuccess || !ptr) return cuda_error("cudaGetSymbolAddress of the static scratch", e);
  g_scratch_ptr[dev] = ptr;
  *out = ptr;
  return GMMFR_OK;
}

}  // namespace

extern "C" GMMFR_API gmmfr_status gmmfr_grouped_matmul_finalize_routing_static_scratch(
    const gmmfr_problem* problem, const gmmfr_tensor* x1, const gmmfr_tensor* pertoken_scale,
    const gmmfr_tensor* group_list, const gmmfr_tensor* logit, const gmmfr_tensor* row_index,
    const gmmfr_tensor* shared_input, const gmmfr_tensor* out, const void* prepared, size_t prepared_bytes,
    void* stream) {
  size_t need = 0;
  if (gmmfr_status st = gmmfr_workspace_size(problem, 1, &need)) return st;
  if (!prepared)
    return gmmfr::record_error(GMMFR_ERR_INVALID_ARG,
                               "the static-scratch entry point needs weights from gmmfr_prepare_weights");
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg), "problem needs %zu bytes of scratch; the static scratch holds %zu (16 MiB)", need,
             kStaticScratchBytes);
    return gmmfr::record_error(GMMFR_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  if (gmmfr_status st = scratch_address(static_cast<cudaStream_t>(stream), &scratch)) return st;
  // The operator overwrites every scratch word it reads (header, group table,
  // token scales, CSR) before reading it, so nothing has to be cleared here.
  return gmmfr_grouped_matmul_finalize_routing(problem, x1, nullptr, nullptr, pertoken_scale, group_list, logit,
                                               row_index, shared_input, nullptr, out, prepared, prepared_bytes,
                                               scratch, kStaticScratchBytes, stream);
}

extern "C" GMMFR_API gmmfr_status gmmfr_static_scratch_check_device_errors(void* stream, uint32_t* bits) {
  if (!bits) return gmmfr::record_error(GMMFR_ERR_INVALID_ARG, "bits is NULL");
  void* scratch = nullptr;
  if (gmmfr_status st = scratch_address(static_cast<cudaStream_t>(stream), &scratch)) return st;
  return gmmfr_check_device_errors(scratch, stream, bits);
}

// conv_noalloc.cu -- ssm_conv_bwd_noalloc: the conv1d backward for callers that cannot
// allocate device memory.
//
// ssm_conv_bwd needs a caller-provided scratch buffer (the per-tile partial sums of d_c and
// d_bias).  This variant keeps that scratch in a fixed array in the library's own device
// memory instead, so the caller passes only inputs and outputs.  Every GPU that loads the
// library holds the array until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "ssm.h"

namespace {

// The scratch of every ssm_conv_bwd_noalloc call on a device.  Host code must not use this
// name as an address: on the host it is only a stand-in for the symbol, so its device address
// is looked up with cudaGetSymbolAddress (once per device) and passed to the kernels.
static __device__ __align__(256) unsigned char g_conv_scratch[SSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_conv_scratch on the current device, looked up on the first call made
// with that device current.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SSM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_conv_scratch) != cudaSuccess || !p) return SSM_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SSM_OK;
}

}  // namespace

extern "C" int ssm_conv_bwd_noalloc(const void* sx, const float* c, const float* bias,
                                    const void* dout, void* d_sx, float* d_c, float* d_bias,
                                    int n_s, int d_inner, int n_t, int d_conv, int io,
                                    unsigned flags, void* stream) {
  if (n_s <= 0 || d_inner <= 0 || n_t <= 0 || d_conv <= 0) return SSM_ERR_INVALID_ARG;
  if (d_conv > SSM_MAX_D_CONV) return SSM_ERR_UNSUPPORTED;
  const size_t need = ssm_conv_workspace_size(n_s, d_inner, n_t, d_conv);
  if (need == 0) return SSM_ERR_INVALID_ARG;
  if (need > (size_t)SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_UNSUPPORTED;
  void* ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc != SSM_OK) return rc;
  // The partial sums are written in full by every call before they are read, so nothing in
  // the shared array has to be cleared first.
  return ssm_conv_bwd(sx, c, bias, dout, d_sx, d_c, d_bias, ws, (size_t)SSM_NOALLOC_SCRATCH_BYTES,
                      n_s, d_inner, n_t, d_conv, io, flags, stream);
}

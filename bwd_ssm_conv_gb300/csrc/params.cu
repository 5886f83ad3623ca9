// params.cu -- the A_log parameterisation of the scan (infotheory's mamba1 layer weights hold
// A_log and A = -exp(A_log), and its gradient path turns dA into dA_log = dA * A): A from A_log
// into scratch before a scan call, and dL/dA_log = dL/dA * A after the backward.
#include "common.cuh"
#include "kernels.cuh"

namespace ssm {

namespace {

__global__ void a_from_log_kernel(const float* __restrict__ a_log, float* __restrict__ a, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    a[i] = -expf(__ldg(a_log + i));
}

__global__ void scale_by_kernel(float* __restrict__ v, const float* __restrict__ s, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    v[i] *= __ldg(s + i);
}

int blocks_of(int n) { return n <= 0 ? 1 : (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024; }

}  // namespace

cudaError_t launch_a_from_log(const float* a_log, float* a, int n, cudaStream_t st) {
  a_from_log_kernel<<<blocks_of(n), 256, 0, st>>>(a_log, a, n), count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_scale_dA(float* d_a, const float* a, int n, cudaStream_t st) {
  scale_by_kernel<<<blocks_of(n), 256, 0, st>>>(d_a, a, n), count_launches(1);
  return cudaGetLastError();
}

}  // namespace ssm

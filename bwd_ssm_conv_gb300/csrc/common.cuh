// common.cuh -- helpers shared by the kernels of libssm_gb300 (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm.h"

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(v) = 2^(v * log2 e)

// ---- I/O element types --------------------------------------------------------------
template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}
template <typename T> __device__ __forceinline__ void st(T* p, float v);
template <> __device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);  // one round-to-nearest-even store from fp32
}

// ---- pointwise math -----------------------------------------------------------------
// 2^v by the SFU instruction (relative error ~2^-22; subnormal results flush to 0).
__device__ __forceinline__ float ex2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// 1/v by the SFU instruction (at most 1 ulp off; 1/inf = 0).
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// The denominator 1 + 2^(-v log2 e) lies in [1, inf], where the SFU reciprocal needs no fix-up.
__device__ __forceinline__ float sigmoidf_(float v) { return rcp_approx(1.0f + ex2(-v * kLog2e)); }
__device__ __forceinline__ float siluf_(float v) { return v * sigmoidf_(v); }
// d/dv silu(v) = s (1 + v (1 - s)),  s = sigmoid(v)   (silu_grad_from_sigmoid)
__device__ __forceinline__ float silu_gradf_(float v) {
  float s = sigmoidf_(v);
  return s * (1.0f + v * (1.0f - s));
}
// softplus with threshold 20 (identity above), and the derivative of that piecewise function.
__device__ __forceinline__ float softplusf_(float v) { return v > 20.0f ? v : log1pf(__expf(v)); }
__device__ __forceinline__ float softplus_gradf_(float v) {
  return v > 20.0f ? 1.0f : sigmoidf_(v);
}

// ---- packed fp32 pairs (fma/mul/add .rn.f32x2): one instruction for two lanes' worth ------
// On GB300 these run at the same FMA-pipe rate as two scalar ops but take one issue slot.
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// 2^v for both halves (two SFU operations).
__device__ __forceinline__ f2_t f2_ex2(f2_t v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  return f2_pack(ex2(lo), ex2(hi));
}

// ---- device status word (first 4 bytes of every scan workspace) ---------------------
// Holds 0 or the first error a kernel recorded.  Only ever written with atomicCAS from 0.
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

constexpr size_t kStatusBytes = 256;

// Number of kernels this library has enqueued in the process (ssm_kernel_launches).
void count_launches(int n);
__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace ssm

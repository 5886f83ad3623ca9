// decode.cu -- the single-token step of the path, fused into one launch: the conv ring-state
// roll, conv1d(+bias, SiLU) of the new input column and one step of the scan.  It is the
// per-token loop of infotheory's mamba1 runtime (forward_impl over one token with its conv
// ring buffer, depthwise_conv_step, and its recurrent state) and ggml's ssm_conv + ssm_scan
// with n_seq_tokens = 1 (ggmlR), with the arithmetic of conv.cu and scan_fwd.cu:
//   x   = act(bias + sum_{k<K-1} conv_state[k] c[k] + x_new c[K-1])   (rounded to the I/O type)
//   conv_state <- (conv_state[1..K-2], x_new)
//   h   = exp(delta A) h + delta x B,   y = (C . h + D x) silu(z)
// A group of tpc threads (a power of two <= 32, inside one warp) owns one (sequence, channel):
// each thread NS states; y is summed over the group with xor-shuffles.  The state and the conv
// state are updated in place, at row ids[b] (or b) of their arrays.
#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"

namespace ssm {

namespace {

constexpr int kDecodeThreads = 256;

// A value of the I/O type as fp32 (plain loads: the conv state is rewritten by this kernel).
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename IO, int NS, bool SCALAR_A>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_kernel(const ScanProblem p, int K, int silu, int tpc, const IO* __restrict__ x_new,
                   IO* conv_state, const float* __restrict__ c, const float* __restrict__ bias,
                   float* state, IO* __restrict__ y) {
  constexpr bool ACC = sizeof(IO) == 4;  // accurate decay form for fp32 I/O
  const long gid = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long total = (long)p.ns * p.HP * tpc;
  // no early return: every lane of a group reaches the shuffles (groups never straddle the end)
  const bool in_range = gid < total;
  const long cidx = in_range ? gid / tpc : 0;
  const int sg = (int)(gid - cidx * tpc);
  const int b = (int)(cidx / p.HP), ch = (int)(cidx - (long)b * p.HP);
  const int h = ch / p.P, g = h / (p.H / p.G), N = p.N;
  const unsigned gmask = group_mask(tpc);
  int row = b;
  bool ok = in_range;
  if (ok && p.ids) {
    row = __ldg(p.ids + b);
    if (row < 0 || row >= p.state_rows) {
      if (sg == 0) record_status(p.status, SSM_ERR_INVALID_ARG);
      ok = false;
    }
  }

  // ---- conv of the new column (the conv kernels' tap order: bias first, oldest input first) --
  IO* cs = conv_state + ((long)row * p.HP + ch) * (K - 1);
  float xv = 0.0f;
  IO xn_raw{};
  if (ok) {
    float pre = bias ? __ldg(bias + ch) : 0.0f;
    for (int k = 0; k + 1 < K; k++) pre = fmaf(to_f(cs[k]), __ldg(c + (long)ch * K + k), pre);
    xn_raw = x_new[(long)b * p.HP + ch];
    pre = fmaf(to_f(xn_raw), __ldg(c + (long)ch * K + K - 1), pre);
    const float act = silu ? siluf_(pre) : pre;
    if constexpr (sizeof(IO) == 4) xv = act;
    else xv = __bfloat162float(__float2bfloat16_rn(act));  // as stored by ssm_conv_fwd
  }
  __syncwarp(gmask);  // every lane of the group has read the old conv state
  if (ok && sg == 0 && K > 1) {  // roll: drop the oldest, append the new column
    for (int j = 0; j + 2 < K; j++) cs[j] = cs[j + 1];
    cs[K - 2] = xn_raw;
  }

  // ---- one scan step over this thread's states --------------------------------------------
  float acc = 0.0f;
  if (ok) {
    float dl = ld(reinterpret_cast<const IO*>(p.dt) + (long)b * p.H + h);
    if (p.softplus) dl = softplusf_(dl + (p.dt_bias ? __ldg(p.dt_bias + h) : 0.0f));
    const float dx = dl * xv;
    const IO* Br = reinterpret_cast<const IO*>(p.B) + ((long)b * p.G + g) * N;
    const IO* Cr = reinterpret_cast<const IO*>(p.C) + ((long)b * p.G + g) * N;
    float* sp = state + ((long)row * p.HP + ch) * N;
    const DecayCoef as = SCALAR_A ? decay_coef<ACC>(dl, __ldg(p.A + h) * kLog2e) : DecayCoef{0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < NS; j++) {
      const int n = sg * NS + j;
      if (n < N) {
        const DecayCoef a = SCALAR_A ? as : decay_coef<ACC>(dl, __ldg(p.A + (long)h * N + n) * kLog2e);
        const float hv = decay_step<ACC>(a, sp[n], dx * ld(Br + n));
        sp[n] = hv;
        acc = fmaf(ld(Cr + n), hv, acc);
      }
    }
  }
  for (int off = tpc >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(gmask, acc, off);
  if (ok && sg == 0) {
    float yv = fmaf(p.D ? __ldg(p.D + ch) : 0.0f, xv, acc);
    if (p.z) yv *= siluf_(ld(reinterpret_cast<const IO*>(p.z) + (long)b * p.HP + ch));
    if (p.check_finite && !isfinite(yv)) record_status(p.status, SSM_ERR_NONFINITE);
    st(y + (long)b * p.HP + ch, yv);
  }
}

template <typename IO, int NS>
cudaError_t launch_ns(const ScanProblem& p, int K, int silu, int tpc, const void* x_new,
                      void* conv_state, const float* c, const float* bias, float* state, void* y,
                      cudaStream_t st) {
  const long total = (long)p.ns * p.HP * tpc;
  const int blocks = (int)((total + kDecodeThreads - 1) / kDecodeThreads);
  if (p.a_per_state)
    decode_step_kernel<IO, NS, false><<<blocks, kDecodeThreads, 0, st>>>(
        p, K, silu, tpc, (const IO*)x_new, (IO*)conv_state, c, bias, state, (IO*)y);
  else
    decode_step_kernel<IO, NS, true><<<blocks, kDecodeThreads, 0, st>>>(
        p, K, silu, tpc, (const IO*)x_new, (IO*)conv_state, c, bias, state, (IO*)y);
  count_launches(1);
  return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_io(const ScanProblem& p, int K, int silu, const void* x_new, void* conv_state,
                      const float* c, const float* bias, float* state, void* y, cudaStream_t st) {
  // states per thread: the smallest of 4, 8, 16 that keeps a channel's group within a warp
  const int ns = p.N <= 128 ? 4 : (p.N <= 256 ? 8 : 16);
  int tpc = 1;
  while (tpc * ns < p.N) tpc <<= 1;
  switch (ns) {
    case 4: return launch_ns<IO, 4>(p, K, silu, tpc, x_new, conv_state, c, bias, state, y, st);
    case 8: return launch_ns<IO, 8>(p, K, silu, tpc, x_new, conv_state, c, bias, state, y, st);
    default: return launch_ns<IO, 16>(p, K, silu, tpc, x_new, conv_state, c, bias, state, y, st);
  }
}

}  // namespace

cudaError_t launch_decode_step(const ScanProblem& p, int K, int silu, const void* x_new,
                               void* conv_state, const float* c, const float* bias, float* state,
                               void* y, cudaStream_t st) {
  return p.io == SSM_BF16
             ? launch_io<__nv_bfloat16>(p, K, silu, x_new, conv_state, c, bias, state, y, st)
             : launch_io<float>(p, K, silu, x_new, conv_state, c, bias, state, y, st);
}

}  // namespace ssm

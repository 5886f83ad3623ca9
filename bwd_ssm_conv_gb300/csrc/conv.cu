// conv.cu -- causal depthwise conv1d (+bias, +SiLU): forward, backward, reductions.
//
// Forward (ggmlR test-ssm-rwkv.R, "ggml_ssm_conv matches a depthwise convolution computed
// in R"):  out[b][t][d] = act(sum_k sx[b][d][t+k] c[d][k] + bias[d]).  sx is time-fastest,
// out is channel-fastest, so every tile is transposed through shared memory: loads run
// along time, stores along channels, both coalesced.
//
// Backward (lattice-inference gdn_backward.rs step 5, ggmlR ssm_conv_back):
//   gp[t]      = dout[t] * silu'(pre[t])            (pre recomputed from sx)
//   d_sx[i]    = sum_k gp[i-k] c[k]                 (0 <= i-k < L)
//   d_c[d][k]  = sum_{b,t} gp[b][t][d] sx[b][d][t+k],   d_bias[d] = sum_{b,t} gp
// d_c / d_bias are summed per tile into the workspace and reduced in a fixed order.
#include "common.cuh"
#include "kernels.cuh"

namespace ssm {

constexpr int kConvTD = 32;   // channels per tile
constexpr int kConvTT = 64;   // time columns per tile
constexpr int kConvThreads = 256;

__host__ __device__ inline int odd_up(int v) { return v | 1; }

template <typename IO>
__global__ void __launch_bounds__(kConvThreads)
conv_fwd_kernel(const IO* __restrict__ sx, const float* __restrict__ c,
                const float* __restrict__ bias, IO* __restrict__ out, int D, int L, int K,
                int silu) {
  extern __shared__ float sm[];
  const int R = kConvTT + K - 1, Rp = odd_up(R), Kp = odd_up(K);
  float* s = sm;                        // [TD][Rp]   odd row stride: conflict-free column reads
  float* w = sm + kConvTD * Rp;         // [TD][Kp]
  const int d0 = blockIdx.x * kConvTD, t0 = blockIdx.y * kConvTT, b = blockIdx.z;
  const long W = (long)L + K - 1;
  const int tid = threadIdx.x;
  for (int i = tid; i < kConvTD * R; i += kConvThreads) {
    int r = i / R, col = i - r * R;
    int d = d0 + r;
    long t = (long)t0 + col;
    s[r * Rp + col] = (d < D && t < W) ? ld(sx + ((long)b * D + d) * W + t) : 0.0f;
  }
  for (int i = tid; i < kConvTD * K; i += kConvThreads) {
    int r = i / K, k = i - r * K;
    int d = d0 + r;
    w[r * Kp + k] = d < D ? __ldg(c + (long)d * K + k) : 0.0f;
  }
  __syncthreads();
  const int tx = tid & 31, ty = tid >> 5;
  const int d = d0 + tx;
  if (d >= D) return;
  const float bv = bias ? __ldg(bias + d) : 0.0f;
  for (int tt = ty; tt < kConvTT; tt += kConvThreads / 32) {
    int t = t0 + tt;
    if (t >= L) break;
    float acc = 0.0f;
    for (int k = 0; k < K; k++) acc = fmaf(s[tx * Rp + tt + k], w[tx * Kp + k], acc);
    acc += bv;
    st(out + ((long)b * L + t) * D + d, silu ? siluf_(acc) : acc);
  }
}

template <typename IO>
__global__ void conv_state_kernel(const IO* __restrict__ sx, IO* __restrict__ st_out, int n_s,
                                  int D, int L, int K) {
  const long total = (long)n_s * D * (K - 1);
  const long W = (long)L + K - 1;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    long row = i / (K - 1);
    int k = (int)(i - row * (K - 1));
    st(st_out + i, ld(sx + row * W + L + k));
  }
}

template <typename IO>
__global__ void __launch_bounds__(kConvThreads)
conv_bwd_kernel(const IO* __restrict__ sx, const float* __restrict__ c,
                const float* __restrict__ bias, const IO* __restrict__ dout,
                IO* __restrict__ d_sx, float* __restrict__ part, int D, int L, int K, int silu) {
  extern __shared__ float sm[];
  // The tile owns d_sx columns [i0, i0+TT) and, for the d_c partials, tokens [i0, i0+TT).
  const int Rs = odd_up(kConvTT + 2 * K - 2);   // sx columns i0-K+1 .. i0+TT+K-2
  const int Rg = odd_up(kConvTT + K - 1);       // gp tokens  i0-K+1 .. i0+TT-1
  const int Kp = odd_up(K);
  float* sxs = sm;                               // [TD][Rs]
  float* gps = sxs + kConvTD * Rs;               // [TD][Rg]
  float* w = gps + kConvTD * Rg;                 // [TD][Kp]
  const int d0 = blockIdx.x * kConvTD, i0 = blockIdx.y * kConvTT, b = blockIdx.z;
  const long W = (long)L + K - 1;
  const int tid = threadIdx.x;
  const int base = i0 - K + 1;                   // global column of local index 0
  const int ns = kConvTT + 2 * K - 2, ng = kConvTT + K - 1;
  for (int i = tid; i < kConvTD * ns; i += kConvThreads) {
    int r = i / ns, j = i - r * ns;
    int d = d0 + r;
    long col = (long)base + j;
    sxs[r * Rs + j] = (d < D && col >= 0 && col < W) ? ld(sx + ((long)b * D + d) * W + col) : 0.0f;
  }
  for (int i = tid; i < kConvTD * K; i += kConvThreads) {
    int r = i / K, k = i - r * K;
    int d = d0 + r;
    w[r * Kp + k] = d < D ? __ldg(c + (long)d * K + k) : 0.0f;
  }
  for (int i = tid; i < kConvTD * ng; i += kConvThreads) {  // dout is channel-fastest
    int tl = i / kConvTD, r = i - tl * kConvTD;
    int d = d0 + r;
    long t = (long)base + tl;
    gps[r * Rg + tl] = (d < D && t >= 0 && t < L) ? ld(dout + ((long)b * L + t) * D + d) : 0.0f;
  }
  __syncthreads();
  if (silu) {  // gp = dout * silu'(pre), pre recomputed (same tap order as the forward)
    for (int i = tid; i < kConvTD * ng; i += kConvThreads) {
      int r = i / ng, tl = i - r * ng;
      int d = d0 + r;
      long t = (long)base + tl;
      if (d >= D || t < 0 || t >= L) continue;
      float pre = 0.0f;
      for (int k = 0; k < K; k++) pre = fmaf(sxs[r * Rs + tl + k], w[r * Kp + k], pre);
      if (bias) pre += __ldg(bias + d);
      gps[r * Rg + tl] *= silu_gradf_(pre);
    }
    __syncthreads();
  }
  // d_sx columns [i0, i0+TT): warp lanes along time -> coalesced row stores
  const int lane = tid & 31, wid = tid >> 5;
  for (int r = wid; r < kConvTD; r += kConvThreads / 32) {
    int d = d0 + r;
    if (d >= D) continue;
    for (int il = lane; il < kConvTT; il += 32) {
      long i = (long)i0 + il;
      if (i >= W) break;
      float acc = 0.0f;
      for (int k = 0; k < K; k++) acc = fmaf(gps[r * Rg + il + K - 1 - k], w[r * Kp + k], acc);
      st(d_sx + ((long)b * D + d) * W + i, acc);
    }
  }
  // partial d_c[d][k] (k < K) and d_bias[d] (k == K) over the tokens this tile owns
  const int nt = gridDim.y;
  for (int i = tid; i < kConvTD * (K + 1); i += kConvThreads) {
    int r = i / (K + 1), k = i - r * (K + 1);
    int d = d0 + r;
    if (d >= D) continue;
    float acc = 0.0f;
    for (int tl = 0; tl < kConvTT; tl++) {
      long t = (long)i0 + tl;
      if (t >= L) break;
      float g = gps[r * Rg + tl + K - 1];
      acc = (k < K) ? fmaf(g, sxs[r * Rs + tl + K - 1 + k], acc) : acc + g;
    }
    part[(((long)b * nt + blockIdx.y) * D + d) * (K + 1) + k] = acc;
  }
}


// ---- d_conv <= 4: compile-time taps and division-free index math -------------------------
// Loads walk rows with whole warps (lane = column), so no per-element division is needed; the
// tap loops unroll.  Same tiles, results and partial layout as the general kernels above.
template <typename IO, int K>
__global__ void __launch_bounds__(kConvThreads)
conv_fwd_k_kernel(const IO* __restrict__ sx, const float* __restrict__ c,
                  const float* __restrict__ bias, IO* __restrict__ out, int D, int L, int silu) {
  constexpr int R = kConvTT + K - 1, Rp = R | 1;
  constexpr int kWarpsC = kConvThreads / 32;
  __shared__ float s[kConvTD * Rp];
  const int d0 = blockIdx.x * kConvTD, t0 = blockIdx.y * kConvTT, b = blockIdx.z;
  const long W = (long)L + K - 1;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int r = wid; r < kConvTD; r += kWarpsC) {
    const int d = d0 + r;
    const IO* row = sx + ((long)b * D + d) * W + t0;
    const long lim = W - t0;  // columns left in this row
#pragma unroll
    for (int col = lane; col < R; col += 32)
      s[r * Rp + col] = (d < D && col < lim) ? ld(row + col) : 0.0f;
  }
  const int d = d0 + lane;
  float w[K];
#pragma unroll
  for (int k = 0; k < K; k++) w[k] = d < D ? __ldg(c + (long)d * K + k) : 0.0f;
  const float bv = (bias && d < D) ? __ldg(bias + d) : 0.0f;
  __syncthreads();
  if (d >= D) return;
  const int tmax = min(kConvTT, L - t0);
  for (int tt = wid; tt < tmax; tt += kWarpsC) {
    float acc = bv;
#pragma unroll
    for (int k = 0; k < K; k++) acc = fmaf(s[lane * Rp + tt + k], w[k], acc);
    st(out + ((long)b * L + t0 + tt) * D + d, silu ? siluf_(acc) : acc);
  }
}

template <typename IO, int K>
__global__ void __launch_bounds__(kConvThreads)
conv_bwd_k_kernel(const IO* __restrict__ sx, const float* __restrict__ c,
                  const float* __restrict__ bias, const IO* __restrict__ dout,
                  IO* __restrict__ d_sx, float* __restrict__ part, int D, int L, int silu) {
  constexpr int NS_ = kConvTT + 2 * K - 2, Rs = NS_ | 1;  // sx columns i0-K+1 .. i0+TT+K-2
  constexpr int NG = kConvTT + K - 1, Rg = NG | 1;        // gp tokens  i0-K+1 .. i0+TT-1
  constexpr int kWarpsC = kConvThreads / 32;
  __shared__ float sxs[kConvTD * Rs];
  __shared__ float gps[kConvTD * Rg];
  const int d0 = blockIdx.x * kConvTD, i0 = blockIdx.y * kConvTT, b = blockIdx.z;
  const long W = (long)L + K - 1;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int base = i0 - K + 1;
  for (int r = wid; r < kConvTD; r += kWarpsC) {  // sx: rows along time
    const int d = d0 + r;
    const IO* row = sx + ((long)b * D + d) * W;
#pragma unroll
    for (int j = lane; j < NS_; j += 32) {
      const long col = (long)base + j;
      sxs[r * Rs + j] = (d < D && col >= 0 && col < W) ? ld(row + col) : 0.0f;
    }
  }
  {  // dout: channel-fastest rows per token; lane = channel
    const int d = d0 + lane;
    for (int tl = wid; tl < NG; tl += kWarpsC) {
      const long t = (long)base + tl;
      gps[lane * Rg + tl] = (d < D && t >= 0 && t < L) ? ld(dout + ((long)b * L + t) * D + d) : 0.0f;
    }
  }
  // each warp owns channel rows r = wid, wid + 8, ...: its taps in registers
  __syncthreads();
  if (silu) {  // gp = dout * silu'(pre), pre recomputed with the forward's tap order
    for (int r = wid; r < kConvTD; r += kWarpsC) {
      const int d = d0 + r;
      if (d >= D) continue;
      float w[K];
#pragma unroll
      for (int k = 0; k < K; k++) w[k] = __ldg(c + (long)d * K + k);
      const float bv = bias ? __ldg(bias + d) : 0.0f;
#pragma unroll
      for (int tl = lane; tl < NG; tl += 32) {
        const long t = (long)base + tl;
        if (t < 0 || t >= L) continue;
        float pre = bv;
#pragma unroll
        for (int k = 0; k < K; k++) pre = fmaf(sxs[r * Rs + tl + k], w[k], pre);
        gps[r * Rg + tl] *= silu_gradf_(pre);
      }
    }
    __syncthreads();
  }
  const int nt = gridDim.y;
  for (int r = wid; r < kConvTD; r += kWarpsC) {
    const int d = d0 + r;
    if (d >= D) continue;
    float w[K];
#pragma unroll
    for (int k = 0; k < K; k++) w[k] = __ldg(c + (long)d * K + k);
    // d_sx columns [i0, i0+TT): lanes along time -> coalesced row stores
#pragma unroll
    for (int il = lane; il < kConvTT; il += 32) {
      const long i = (long)i0 + il;
      if (i < W) {
        float acc = 0.0f;
#pragma unroll
        for (int k = 0; k < K; k++) acc = fmaf(gps[r * Rg + il + K - 1 - k], w[k], acc);
        st(d_sx + ((long)b * D + d) * W + i, acc);
      }
    }
    // partial d_c[d][k] and d_bias[d] over the tokens this tile owns: lanes over tokens, then
    // a fixed-order warp sum
    float pk[K + 1];
#pragma unroll
    for (int k = 0; k <= K; k++) pk[k] = 0.0f;
#pragma unroll
    for (int tl = lane; tl < kConvTT; tl += 32) {
      if ((long)i0 + tl < L) {
        const float g = gps[r * Rg + tl + K - 1];
#pragma unroll
        for (int k = 0; k < K; k++) pk[k] = fmaf(g, sxs[r * Rs + tl + K - 1 + k], pk[k]);
        pk[K] += g;
      }
    }
#pragma unroll
    for (int k = 0; k <= K; k++) {
      float v = pk[k];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) part[(((long)b * nt + blockIdx.y) * D + d) * (K + 1) + k] = v;
    }
  }
}

// d_c[d][k] and d_bias[d] = sum over (sequence, tile) partials.  A block = 32 outputs x 8
// slices of the (sequence, tile) range; slices combine in shared memory in a fixed order.
constexpr int kRedOut = 32, kRedSlices = 8;
__global__ void __launch_bounds__(kRedOut * kRedSlices)
conv_reduce_kernel(const float* __restrict__ part, float* __restrict__ d_c,
                   float* __restrict__ d_bias, int n_s, int nt, int D, int K) {
  __shared__ float sred[kRedSlices][kRedOut];
  const long total = (long)D * (K + 1);
  const int lo = threadIdx.x % kRedOut, sl = threadIdx.x / kRedOut;
  const long o = (long)blockIdx.x * kRedOut + lo;
  const long terms = (long)n_s * nt;
  float acc = 0.0f;
  if (o < total)
    for (long j = sl; j < terms; j += kRedSlices) acc += part[j * total + o];
  sred[sl][lo] = acc;
  __syncthreads();
  if (sl == 0 && o < total) {
    float v = 0.0f;
    for (int q = 0; q < kRedSlices; q++) v += sred[q][lo];
    const int d = (int)(o / (K + 1)), k = (int)(o - (long)d * (K + 1));
    if (k < K) d_c[(long)d * K + k] = v;
    else if (d_bias) d_bias[d] = v;
  }
}

// ---- host launchers ----------------------------------------------------------------------
size_t conv_bwd_ws_bytes(int n_s, int D, int L, int K) {
  long W = (long)L + K - 1;
  long nt = (W + kConvTT - 1) / kConvTT;
  return align_up(sizeof(float) * (size_t)n_s * nt * D * (K + 1), 256);
}

template <typename IO>
static cudaError_t conv_fwd_t(const void* sx, const float* c, const float* bias, void* out,
                              void* cs, int n_s, int D, int L, int K, int silu, cudaStream_t st) {
  dim3 grid((D + kConvTD - 1) / kConvTD, (L + kConvTT - 1) / kConvTT, n_s);
  const IO* x = (const IO*)sx;
  IO* o = (IO*)out;
  switch (K) {
    case 1: conv_fwd_k_kernel<IO, 1><<<grid, kConvThreads, 0, st>>>(x, c, bias, o, D, L, silu); break;
    case 2: conv_fwd_k_kernel<IO, 2><<<grid, kConvThreads, 0, st>>>(x, c, bias, o, D, L, silu); break;
    case 3: conv_fwd_k_kernel<IO, 3><<<grid, kConvThreads, 0, st>>>(x, c, bias, o, D, L, silu); break;
    case 4: conv_fwd_k_kernel<IO, 4><<<grid, kConvThreads, 0, st>>>(x, c, bias, o, D, L, silu); break;
    default: {
      size_t smem = sizeof(float) * (kConvTD * odd_up(kConvTT + K - 1) + kConvTD * odd_up(K));
      conv_fwd_kernel<IO><<<grid, kConvThreads, smem, st>>>(x, c, bias, o, D, L, K, silu);
    }
  }
  count_launches(1);
  if (cs && K > 1) {
    long total = (long)n_s * D * (K - 1);
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    conv_state_kernel<IO><<<blocks, 256, 0, st>>>((const IO*)sx, (IO*)cs, n_s, D, L, K), count_launches(1);
  }
  return cudaGetLastError();
}

template <typename IO>
static cudaError_t conv_bwd_t(const void* sx, const float* c, const float* bias, const void* dout,
                              void* d_sx, float* d_c, float* d_bias, void* ws, int n_s, int D,
                              int L, int K, int silu, cudaStream_t st) {
  long W = (long)L + K - 1;
  int nt = (int)((W + kConvTT - 1) / kConvTT);
  dim3 grid((D + kConvTD - 1) / kConvTD, nt, n_s);
  size_t smem = sizeof(float) * (kConvTD * odd_up(kConvTT + 2 * K - 2) +
                                 kConvTD * odd_up(kConvTT + K - 1) + kConvTD * odd_up(K));
  float* part = (float*)ws;
  const IO* x = (const IO*)sx;
  const IO* g = (const IO*)dout;
  IO* dx = (IO*)d_sx;
  switch (K) {
    case 1: conv_bwd_k_kernel<IO, 1><<<grid, kConvThreads, 0, st>>>(x, c, bias, g, dx, part, D, L, silu); break;
    case 2: conv_bwd_k_kernel<IO, 2><<<grid, kConvThreads, 0, st>>>(x, c, bias, g, dx, part, D, L, silu); break;
    case 3: conv_bwd_k_kernel<IO, 3><<<grid, kConvThreads, 0, st>>>(x, c, bias, g, dx, part, D, L, silu); break;
    case 4: conv_bwd_k_kernel<IO, 4><<<grid, kConvThreads, 0, st>>>(x, c, bias, g, dx, part, D, L, silu); break;
    default:
      conv_bwd_kernel<IO><<<grid, kConvThreads, smem, st>>>(x, c, bias, g, dx, part, D, L, K, silu);
  }
  count_launches(1);
  const long total = (long)D * (K + 1);
  const int blocks = (int)((total + kRedOut - 1) / kRedOut);
  conv_reduce_kernel<<<blocks, kRedOut * kRedSlices, 0, st>>>(part, d_c, d_bias, n_s, nt, D, K),
      count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_conv_fwd(const void* sx, const float* c, const float* bias, void* out, void* cs,
                            int n_s, int D, int L, int K, int io, int silu, cudaStream_t st) {
  return io == SSM_BF16 ? conv_fwd_t<__nv_bfloat16>(sx, c, bias, out, cs, n_s, D, L, K, silu, st)
                        : conv_fwd_t<float>(sx, c, bias, out, cs, n_s, D, L, K, silu, st);
}

cudaError_t launch_conv_bwd(const void* sx, const float* c, const float* bias, const void* dout,
                            void* d_sx, float* d_c, float* d_bias, void* ws, int n_s, int D, int L,
                            int K, int io, int silu, cudaStream_t st) {
  return io == SSM_BF16
             ? conv_bwd_t<__nv_bfloat16>(sx, c, bias, dout, d_sx, d_c, d_bias, ws, n_s, D, L, K,
                                         silu, st)
             : conv_bwd_t<float>(sx, c, bias, dout, d_sx, d_c, d_bias, ws, n_s, D, L, K, silu, st);
}

}  // namespace ssm

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
#include <type_traits>

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


// ---- d_conv <= 4, backward: one thread streams 32 tokens of one channel ----------------
// A tile = 32 channels (one per lane) x 256 tokens (8 warps x 32).  Each thread walks its 32
// tokens in order with the taps, the last d_conv inputs and the last d_conv input gradients in
// registers, so every tap sum, SiLU' and d_c term is computed once from registers.  Lanes run
// along channels, so the channel-fastest dout rows are read coalesced straight from global
// memory; the time-fastest sx and d_sx rows go through shared memory, moved with aligned
// 16-byte accesses (row starts have any alignment: a row holds L + d_conv - 1 elements) and
// scalar ones only at partial groups.
constexpr int kSeg = 32;                       // tokens per thread
constexpr int kSegWarps = 8;
constexpr int kSegThreads = 32 * kSegWarps;
constexpr int kSegTT = kSeg * kSegWarps;       // tokens per tile
constexpr int kSegRows = 32;                   // channels per tile

template <typename IO>
__device__ __forceinline__ void unpack16(const uint4 u, float* v) {
  if constexpr (sizeof(IO) == 4) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {  // bf16 -> fp32 is exact: the bits move up 16 places
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}
template <typename IO>
__device__ __forceinline__ uint4 pack16(const float* v) {
  if constexpr (sizeof(IO) == 4) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);  // RNE, as st()
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Copies columns [c0, c0 + NC) of rows d0 .. d0+31 of a time-fastest [..][W] array into
// s[r][0..NC) (row stride SP floats, odd) as fp32; zero outside [0, W) and for rows >= D.
// One row per lane (32 rows per shared store instruction, conflict-free with the odd stride),
// groups gi = wid, wid + 8, ... of 16 bytes aligned in global memory; a group partly outside
// the row is read element by element.  Every load of a thread is issued before its first
// shared store, so the groups' round trips overlap.
template <typename IO, int NC, int SP>
__device__ __forceinline__ void rows_to_smem(const IO* base, int d0, int D, long c0, long W,
                                             float* s, int wid, int lane) {
  constexpr int V = 16 / sizeof(IO);
  constexpr int NG = (NC + V - 1) / V + 1;  // groups covering NC columns at any alignment
  constexpr int KG = (NG + kSegWarps - 1) / kSegWarps;
  const int d = d0 + lane;
  const IO* row = base + (long)(d < D ? d : 0) * W;
  const int ph = (int)(((uintptr_t)(row + c0) & 15) / sizeof(IO));
  uint4 raw[KG];
#pragma unroll
  for (int k = 0; k < KG; k++) {
    const int gi = wid + kSegWarps * k;
    const long cs = c0 - ph + (long)gi * V;  // column of the group's first element
    raw[k] = make_uint4(0u, 0u, 0u, 0u);
    if (d >= D || gi >= NG || cs - c0 >= NC) continue;
    if (cs >= 0 && cs + V <= W) {
      raw[k] = __ldg(reinterpret_cast<const uint4*>(row + cs));
    } else {  // a partial group: its elements inside [0, W), the rest zero
      using B = typename std::conditional<sizeof(IO) == 2, unsigned short, unsigned>::type;
      const B* bits = reinterpret_cast<const B*>(row);
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < V; e++) {
        if (cs + e < 0 || cs + e >= W) continue;
        const uint32_t v = __ldg(bits + cs + e);
        if constexpr (sizeof(IO) == 2) w[e / 2] |= v << (16 * (e % 2));
        else w[e] = v;
      }
      raw[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  if (d >= D) return;
  float* srow = s + lane * SP;
#pragma unroll
  for (int k = 0; k < KG; k++) {
    const int gi = wid + kSegWarps * k;
    const int j0 = gi * V - ph;  // the group's first element's index in s
    if (gi >= NG || j0 >= NC) continue;
    float v[V];
    unpack16<IO>(raw[k], v);
#pragma unroll
    for (int e = 0; e < V; e++)
      if (j0 + e >= 0 && j0 + e < NC) srow[j0 + e] = v[e];
  }
}

// ---- d_conv <= 4, forward: one lane streams 16 tokens of two adjacent channels -----------
// A tile = 64 channels (a pair per lane) x 128 tokens (8 warps x 16).  The pair's arithmetic
// runs in packed fp32 pairs (fma/mul/add.rn.f32x2; each half rounds as the scalar sequence
// would) and leaves as one 4-byte (bf16) or 8-byte (fp32) store per token, so a warp store
// writes 128 or 256 contiguous bytes.  The time-fastest sx rows go through shared memory as
// interleaved fp32 pairs (row 2p in .x, row 2p+1 in .y), one 8-byte read per token and lane;
// the odd pair stride keeps each half-warp's reads on distinct banks.  Rows are moved one per
// lane with aligned 16-byte loads (scalar ones only at partial groups).
constexpr int kPairSeg = 16;                      // tokens per thread
constexpr int kPairTT = kPairSeg * kSegWarps;     // tokens per tile
constexpr int kPairRows = 64;                     // channels per tile

template <typename IO, int K, bool SILU>
__global__ void __launch_bounds__(kSegThreads)
conv_fwd_pair_kernel(const IO* __restrict__ sx, const float* __restrict__ c,
                     const float* __restrict__ bias, IO* __restrict__ out, int D, int L,
                     int ovec) {
  constexpr int NC = kPairTT + K - 1;             // staged columns i0 .. i0+NC-1
  constexpr int SP = NC | 1;                      // pair stride (float2), odd
  constexpr int V = 16 / sizeof(IO);
  constexpr int NG = (NC + V - 1) / V + 1;        // groups covering NC columns at any alignment
  __shared__ float2 s2[kPairRows / 2 * SP];
  float* sf = reinterpret_cast<float*>(s2);
  const int d0 = blockIdx.x * kPairRows, i0 = blockIdx.y * kPairTT, b = blockIdx.z;
  const int W = L + K - 1;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // every load a thread makes is issued before the first shared store: slot (rp, k) = row
  // lane + 32 rp, group wid + 8 k
  constexpr int KG = (NG + kSegWarps - 1) / kSegWarps;
  uint4 raw[kPairRows / 32][KG];
  int ph[kPairRows / 32];
#pragma unroll
  for (int rp = 0; rp < kPairRows / 32; rp++) {
    const int d = d0 + lane + 32 * rp;
    const IO* row = sx + ((long)b * D + (d < D ? d : 0)) * W;
    ph[rp] = (int)(((uintptr_t)(row + i0) & 15) / sizeof(IO));
#pragma unroll
    for (int k = 0; k < KG; k++) {
      const int gi = wid + kSegWarps * k;
      const int cs = i0 - ph[rp] + gi * V;        // column of the group's first element
      raw[rp][k] = make_uint4(0u, 0u, 0u, 0u);
      if (d >= D || gi >= NG || cs - i0 >= NC) continue;
      if (cs >= 0 && cs + V <= W) {
        raw[rp][k] = __ldg(reinterpret_cast<const uint4*>(row + cs));
      } else {  // a partial group: its elements inside [0, W), the rest zero
        using B = typename std::conditional<sizeof(IO) == 2, unsigned short, unsigned>::type;
        const B* bits = reinterpret_cast<const B*>(row);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < V; e++) {
          if (cs + e < 0 || cs + e >= W) continue;
          const uint32_t v = __ldg(bits + cs + e);
          if constexpr (sizeof(IO) == 2) w[e / 2] |= v << (16 * (e % 2));
          else w[e] = v;
        }
        raw[rp][k] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
#pragma unroll
  for (int rp = 0; rp < kPairRows / 32; rp++) {
    const int r = lane + 32 * rp;
    if (d0 + r >= D) continue;
    float* dst = sf + (r >> 1) * 2 * SP + (r & 1);  // column i0 + j at dst[2 j]
#pragma unroll
    for (int k = 0; k < KG; k++) {
      const int gi = wid + kSegWarps * k;
      const int j0 = gi * V - ph[rp];
      if (gi >= NG || j0 >= NC) continue;
      float v[V];
      unpack16<IO>(raw[rp][k], v);
#pragma unroll
      for (int e = 0; e < V; e++)
        if (j0 + e >= 0 && j0 + e < NC) dst[2 * (j0 + e)] = v[e];
    }
  }
  __syncthreads();
  const int d = d0 + 2 * lane, s0 = i0 + wid * kPairSeg;
  if (d >= D || s0 >= L) return;
  const bool has1 = d + 1 < D;
  f2_t w2[K];
#pragma unroll
  for (int k = 0; k < K; k++)
    w2[k] = f2_pack(__ldg(c + (long)d * K + k), has1 ? __ldg(c + (long)(d + 1) * K + k) : 0.0f);
  const f2_t b2 = bias ? f2_pack(__ldg(bias + d), has1 ? __ldg(bias + d + 1) : 0.0f) : 0ull;
  const float2* xr = s2 + lane * SP + wid * kPairSeg;  // column s0 + u + k at xr[u + k]
  IO* o = out + ((long)b * L + s0) * D + d;
  const bool pair = ovec && has1;
  f2_t xw[K];
#pragma unroll
  for (int k = 1; k < K; k++) xw[k] = f2_pack(xr[k - 1].x, xr[k - 1].y);
  auto token = [&](int u) {
#pragma unroll
    for (int k = 0; k + 1 < K; k++) xw[k] = xw[k + 1];
    const float2 xv = xr[u + K - 1];
    xw[K - 1] = f2_pack(xv.x, xv.y);
    f2_t acc = b2;
#pragma unroll
    for (int k = 0; k < K; k++) acc = f2_fma(xw[k], w2[k], acc);
    float lo, hi;
    if constexpr (SILU) {  // silu(v) = v / (1 + 2^(-v log2 e)): the scalar steps, paired
      float e0, e1;
      f2_unpack(f2_mul(acc, f2_pack(-kLog2e, -kLog2e)), e0, e1);
      f2_unpack(f2_add(f2_pack(ex2(e0), ex2(e1)), f2_pack(1.0f, 1.0f)), e0, e1);
      acc = f2_mul(acc, f2_pack(rcp_approx(e0), rcp_approx(e1)));
    }
    f2_unpack(acc, lo, hi);
    IO* ot = o + (long)u * D;
    if (pair) {
      if constexpr (sizeof(IO) == 2) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // RNE, as st()
        *reinterpret_cast<__nv_bfloat162*>(ot) = h;
      } else {
        *reinterpret_cast<float2*>(ot) = make_float2(lo, hi);
      }
    } else {
      st(ot, lo);
      if (has1) st(ot + 1, hi);
    }
  };
  const int n = min(kPairSeg, L - s0);
  if (n == kPairSeg) {
#pragma unroll
    for (int u = 0; u < kPairSeg; u++) token(u);
  } else {
    for (int u = 0; u < n; u++) token(u);
  }
}

// 4 blocks per SM for bf16; fp32's twice as many staging registers would spill there, so 3
template <typename IO, int K, bool SILU>
__global__ void __launch_bounds__(kSegThreads, sizeof(IO) == 2 ? 4 : 3)
conv_bwd_seg_kernel(const IO* __restrict__ sx, const float* __restrict__ c,
                    const float* __restrict__ bias, const IO* __restrict__ dout,
                    IO* __restrict__ d_sx, float* __restrict__ part, int D, int L) {
  // sx columns i0-K+1 .. i0+TT+K-2 (inputs of tokens i0-K+1 .. i0+TT-1); later reused for the
  // d_sx tile (columns i0 .. i0+TT-1).
  constexpr int NC = kSegTT + 2 * K - 2, SP = NC | 1;
  constexpr int NU = kSeg + K - 1;  // steps per thread: K-1 tokens before the segment, then it
  __shared__ float s[kSegRows * SP];
  __shared__ float red[(K + 1) * kSegWarps * 32];
  const int d0 = blockIdx.x * kSegRows, i0 = blockIdx.y * kSegTT, b = blockIdx.z;
  const long W = (long)L + K - 1;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int d = d0 + lane, s0 = i0 + wid * kSeg;
  const bool active = d < D && s0 < W;
  // dout of tokens s0-K+1+u (zero outside [0, L)), issued before the sx tile so that both
  // loads are in flight together
  float dv[NU];
  const int t_first = s0 - (K - 1);
  if (active && t_first >= 0 && t_first + NU <= L) {  // interior segment: no per-token checks
    const IO* dp = dout + ((long)b * L + t_first) * D + d;
#pragma unroll
    for (int u = 0; u < NU; u++) dv[u] = ld(dp + (long)u * D);
  } else {
#pragma unroll
    for (int u = 0; u < NU; u++) {
      const int t = t_first + u;
      dv[u] = (active && t >= 0 && t < L) ? ld(dout + ((long)b * L + t) * D + d) : 0.0f;
    }
  }
  rows_to_smem<IO, NC, SP>(sx + (long)b * D * W, d0, D, (long)i0 - (K - 1), W, s, wid, lane);
  __syncthreads();
  float ox[kSeg];
  float pk[K + 1];
#pragma unroll
  for (int k = 0; k <= K; k++) pk[k] = 0.0f;
  if (active) {
    float w[K];
#pragma unroll
    for (int k = 0; k < K; k++) w[k] = __ldg(c + (long)d * K + k);
    const float bv = bias ? __ldg(bias + d) : 0.0f;
    const float* xr = s + lane * SP + wid * kSeg;  // input column t_first + u + k at xr[u + k]
    float xw[K], gw[K];
#pragma unroll
    for (int k = 1; k < K; k++) xw[k] = xr[k - 1];
#pragma unroll
    for (int k = 0; k < K; k++) gw[k] = 0.0f;
#pragma unroll
    for (int u = 0; u < NU; u++) {
#pragma unroll
      for (int k = 0; k + 1 < K; k++) xw[k] = xw[k + 1];
      xw[K - 1] = xr[u + K - 1];
      float g = dv[u];
      if constexpr (SILU) {  // pre recomputed with the forward's tap order
        float pre = bv;
#pragma unroll
        for (int k = 0; k < K; k++) pre = fmaf(xw[k], w[k], pre);
        g *= silu_gradf_(pre);
      }
#pragma unroll
      for (int k = K - 1; k > 0; k--) gw[k] = gw[k - 1];
      gw[0] = g;  // gw[k] = gp of token t - k
      if (u >= K - 1) {  // token t = s0 + u - K + 1 of the segment: d_sx[t], d_c terms
        float acc = 0.0f;
#pragma unroll
        for (int k = 0; k < K; k++) acc = fmaf(gw[k], w[k], acc);
        ox[u - (K - 1)] = acc;
#pragma unroll
        for (int k = 0; k < K; k++) pk[k] = fmaf(g, xw[k], pk[k]);  // g = 0 past L
        pk[K] += g;
      }
    }
  }
#pragma unroll
  for (int k = 0; k <= K; k++) red[(k * kSegWarps + wid) * 32 + lane] = pk[k];
  __syncthreads();  // every thread is done with the sx tile
  constexpr int SO = kSegTT | 1;
  if (active) {
#pragma unroll
    for (int u = 0; u < kSeg; u++) s[lane * SO + wid * kSeg + u] = ox[u];
  }
  const int nt = gridDim.y;
  if (threadIdx.x < (K + 1) * 32) {  // fixed-order sum over the tile's 8 segments
    const int k = threadIdx.x >> 5, dd = d0 + lane;
    float v = 0.0f;
#pragma unroll
    for (int q = 0; q < kSegWarps; q++) v += red[(k * kSegWarps + q) * 32 + lane];
    if (dd < D) part[(((long)b * nt + blockIdx.y) * D + dd) * (K + 1) + k] = v;
  }
  __syncthreads();
  // d_sx rows: columns [i0, min(i0 + TT, W)), 16-byte aligned groups + scalar edges.  8 lanes
  // share a row (4 rows per warp, 8 warps: all 32 rows in one pass), so every warp store
  // writes 4 runs of 128 contiguous bytes (measured faster than one row per lane, whose 32
  // scattered 16-byte pieces per store cost more than the 2-way shared-memory conflicts here).
  constexpr int V = 16 / sizeof(IO);
  constexpr int NG = (kSegTT + V - 1) / V + 1;
  constexpr int LPR = 8;
  const int n = (int)min((long)kSegTT, W - i0);
  const int r = wid * (32 / LPR) + lane / LPR;  // this lane's row of the tile
  const int dd = d0 + r;
  IO* row = d_sx + ((long)b * D + dd) * W + i0;
  const int ph = (int)(((uintptr_t)row & 15) / sizeof(IO));
  for (int gi = lane % LPR; gi < NG && dd < D; gi += LPR) {
    const int j0 = gi * V - ph;
    if (j0 >= n) break;
    const float* src = s + r * SO + j0;
    if (j0 >= 0 && j0 + V <= n) {
      float v[V];
#pragma unroll
      for (int e = 0; e < V; e++) v[e] = src[e];
      *reinterpret_cast<uint4*>(row + j0) = pack16<IO>(v);
    } else {
#pragma unroll
      for (int e = 0; e < V; e++)
        if (j0 + e >= 0 && j0 + e < n) st(row + j0 + e, src[e]);
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
// One partial of d_c and d_bias per (sequence, time tile, channel): the tile is the one
// conv_bwd_t launches with (kSegTT tokens for d_conv <= 4, kConvTT above).
static int conv_bwd_tile(int K) { return K <= 4 ? kSegTT : kConvTT; }

size_t conv_bwd_ws_bytes(int n_s, int D, int L, int K) {
  long W = (long)L + K - 1;
  const int tt = conv_bwd_tile(K);
  long nt = (W + tt - 1) / tt;
  return align_up(sizeof(float) * (size_t)n_s * nt * D * (K + 1), 256);
}

template <typename IO>
static cudaError_t conv_fwd_t(const void* sx, const float* c, const float* bias, void* out,
                              void* cs, int n_s, int D, int L, int K, int silu, cudaStream_t st) {
  dim3 grid((D + kConvTD - 1) / kConvTD, (L + kConvTT - 1) / kConvTT, n_s);
  const IO* x = (const IO*)sx;
  IO* o = (IO*)out;
  const dim3 gpair((D + kPairRows - 1) / kPairRows, (L + kPairTT - 1) / kPairTT, n_s);
  // a lane's two channels leave in one store when out and D keep every pair aligned
  const int ovec = D % 2 == 0 && ((uintptr_t)out % (2 * sizeof(IO))) == 0;
#define SSM_CONV_PAIR(KK)                                                                        \
  silu ? conv_fwd_pair_kernel<IO, KK, true><<<gpair, kSegThreads, 0, st>>>(x, c, bias, o, D, L, ovec) \
       : conv_fwd_pair_kernel<IO, KK, false><<<gpair, kSegThreads, 0, st>>>(x, c, bias, o, D, L, ovec)
  switch (K) {
    case 1: SSM_CONV_PAIR(1); break;
    case 2: SSM_CONV_PAIR(2); break;
    case 3: SSM_CONV_PAIR(3); break;
    case 4: SSM_CONV_PAIR(4); break;
    default: {
      size_t smem = sizeof(float) * (kConvTD * odd_up(kConvTT + K - 1) + kConvTD * odd_up(K));
      conv_fwd_kernel<IO><<<grid, kConvThreads, smem, st>>>(x, c, bias, o, D, L, K, silu);
    }
  }
#undef SSM_CONV_PAIR
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
  const int tt = conv_bwd_tile(K);
  int nt = (int)((W + tt - 1) / tt);
  dim3 grid((D + kConvTD - 1) / kConvTD, nt, n_s);
  size_t smem = sizeof(float) * (kConvTD * odd_up(kConvTT + 2 * K - 2) +
                                 kConvTD * odd_up(kConvTT + K - 1) + kConvTD * odd_up(K));
  float* part = (float*)ws;
  const IO* x = (const IO*)sx;
  const IO* g = (const IO*)dout;
  IO* dx = (IO*)d_sx;
  switch (K) {
    case 1: silu ? conv_bwd_seg_kernel<IO, 1, true><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L)
                 : conv_bwd_seg_kernel<IO, 1, false><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L); break;
    case 2: silu ? conv_bwd_seg_kernel<IO, 2, true><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L)
                 : conv_bwd_seg_kernel<IO, 2, false><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L); break;
    case 3: silu ? conv_bwd_seg_kernel<IO, 3, true><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L)
                 : conv_bwd_seg_kernel<IO, 3, false><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L); break;
    case 4: silu ? conv_bwd_seg_kernel<IO, 4, true><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L)
                 : conv_bwd_seg_kernel<IO, 4, false><<<grid, kSegThreads, 0, st>>>(x, c, bias, g, dx, part, D, L); break;
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

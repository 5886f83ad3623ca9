// scan_fwd_ssd.cu -- forward scan of the Mamba-2 form (one A per head) in chunked matrix form on
// the tensor cores: tcgen05.mma kind::tf32 with operands in shared memory and accumulators in
// tensor memory.  Applies to bf16 I/O, head_dim a multiple of 64, d_state 128 and a checkpoint
// interval that is a multiple of 64 (ggmlR's ssm_scan with a [1, n_head] A; infotheory's
// mamba1 forward_impl recurrence with one decay shared by a head's states).
//
// With one decay per (token, head), a_t = 2^(lambda_t), lambda_t = delta_t A log2(e), and
// Lambda_t = sum of lambda_s over the chunk's tokens s <= t, the recurrence
//   h_t = a_t h_{t-1} + (delta_t x_t) B_t^T,   y_t = h_t C_t
// has over a chunk of 64 tokens the closed form (the affine steps composed, as the associative
// scan of kizzasi's backprop_ssm composes them)
//   y_t   = sum_{s <= t} 2^(Lambda_t - Lambda_s) (C_t . B_s) delta_s x_s + 2^(Lambda_t) h_start C_t
//   h_end = 2^(Lambda_end) h_start + sum_s 2^(Lambda_end - Lambda_s) delta_s x_s B_s^T
// Three launches:
//   1. ssd_state_kernel, per (sequence, head, chunk, 64 channels): the chunk's own end state
//      S = (w B)^T X (w_s = delta_s 2^(Lambda_end - Lambda_s)) as a 128 x 64 x 64 product
//      (rows: states), and the chunk decay 2^(Lambda_end);
//   2. ssd_pass_kernel, per state element: start states h_start(c+1) = 2^(Lambda_end(c))
//      h_start(c) + S(c) in chunk order, in fp32; checkpoints and the final state fall out;
//   3. ssd_out_kernel, per (sequence, head, chunk, 32 channels): G = C B^T (64 x 64 x 128) and
//      Y' = C h_start^T (64 x 32 x 128); then W = G o (delta_s 2^(Lambda_t - Lambda_s))_{s <= t}
//      and Y = W X (64 x 32 x 64); y_t = Y_t + 2^(Lambda_t) Y'_t, then D x and the gate.
// x, B and C (bf16) are exact in tf32, and so is G.  The computed operands (w B, W, the start
// states) are fp32 values split into two tf32 terms, v = hi + lo with hi = tf32(v) and
// lo = tf32(v - hi), and each product they enter is taken twice (hi and lo against the exact
// operand): a single tf32 rounding (2^-11) of the terms of a nearly cancelling sum measured
// 0.07-0.18 of error near zero outputs in the floored metric, above the bf16 gate of 2e-2.
// fp32 I/O stays on the recurrence kernels (its 1e-4 gate needs the full fp32 recurrence).
#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"
#include "tma.cuh"
#include "tmem.cuh"

namespace ssm {

namespace {

constexpr int kQ = 64;    // tokens per chunk
constexpr int kSP = 64;   // channels per block of the state kernel
constexpr int kSPo = 32;  // channels per block of the output kernel
constexpr int kSN = 128;  // d_state
constexpr int kSsdThreads = 128;

struct SsdArgs {
  ScanProblem p;
  int nchq, npb;   // chunks of kQ tokens; channel blocks per head of the launch
  float* S;        // [ns][H][nchq][P][N]: chunk end states (launch 1), then start states (2)
  float* dec;      // [ns][H][nchq]: 2^(Lambda_end) of every chunk
  float* state_out;
  float* ckpt;
  __nv_bfloat16* y;
};

struct Unit { int b, h, c, pb, g, t0, p0; };

__device__ __forceinline__ Unit unit_of(const SsdArgs& a, int block_channels) {
  const ScanProblem& p = a.p;
  int u = blockIdx.x;
  Unit r;
  r.pb = u % a.npb; u /= a.npb;
  r.c = u % a.nchq; u /= a.nchq;
  r.h = u % p.H;
  r.b = u / p.H;
  r.g = r.h / (p.H / p.G);
  r.t0 = r.c * kQ;
  r.p0 = r.pb * block_channels;
  return r;
}

// v as two tf32 terms: hi = tf32(v), lo = tf32(v - hi) (hi + lo = v to about 2^-22).
__device__ __forceinline__ void split_tf32(float v, float& hi, float& lo) {
  hi = tc::tf32_rn(v);
  lo = tc::tf32_rn(v - hi);
}

// delta of the chunk's tokens and the inclusive log2-decay Lambda (threads 0..63; tokens past
// the sequence end have delta 0 and leave Lambda unchanged).  Within a chunk |Lambda| stays
// around 10^2 at most, so fp32 prefix sums keep each exponent to about 1e-5.
__device__ __forceinline__ void chunk_log_decay(const SsdArgs& a, const Unit& u, float* sDl,
                                                float* sLam, float* sCarry) {
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x;
  if (tid < kQ) {
    const int t = u.t0 + tid;
    float dl = 0.0f;
    if (t < p.L) {
      dl = ld(reinterpret_cast<const __nv_bfloat16*>(p.dt) + ((long)u.b * p.L + t) * p.H + u.h);
      if (p.softplus) dl = softplusf_(dl + (p.dt_bias ? __ldg(p.dt_bias + u.h) : 0.0f));
    }
    float v = dl * (__ldg(p.A + u.h) * kLog2e);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float w = __shfl_up_sync(0xffffffffu, v, o);
      if ((tid & 31) >= o) v += w;
    }
    sDl[tid] = dl;
    sLam[tid] = v;
    if (tid == 31) sCarry[0] = v;
  }
  __syncthreads();
  if (tid >= 32 && tid < kQ) sLam[tid] += sCarry[0];
  __syncthreads();
}

// 8 bf16 (16 bytes, aligned) as fp32; zeros when !in.
__device__ __forceinline__ void ld8_bf16(const __nv_bfloat16* q, bool in, float (&v)[8]) {
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  if (in) u = __ldg(reinterpret_cast<const uint4*>(q));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void sts16(unsigned char* base, uint32_t off, float a0, float a1,
                                      float a2, float a3) {
  *reinterpret_cast<float4*>(base + off) = make_float4(a0, a1, a2, a3);
}

// Staging into K-major tiles.  Every store writes one 16-byte core-matrix row, and the 8 lanes
// of a store phase take 8 consecutive tile rows, so that they hit 8 different bank groups.

// Each staging step issues all of a thread's global loads before its first shared store (the
// stores go through generic pointers, which the compiler would otherwise keep ordered after
// the loads that follow them).

// X^T of the chunk's CH channels [p][s] (K = 64 tokens), exact.  Thread: channel tid % CH,
// 16 CH / 128 of the 16 token groups.
template <int CH>
struct XtRegs { float v[16 * CH / kSsdThreads][4]; };
template <int CH>
__device__ __forceinline__ void load_xt(const SsdArgs& a, const Unit& u, XtRegs<CH>& r) {
  const ScanProblem& p = a.p;
  constexpr int KPT = 16 * CH / kSsdThreads;  // token groups per thread
  const int tid = threadIdx.x, pp = tid % CH, kh = tid / CH;
  const __nv_bfloat16* xc = reinterpret_cast<const __nv_bfloat16*>(p.x) + u.h * p.P + u.p0 + pp;
#pragma unroll
  for (int q = 0; q < KPT; q++)
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int t = u.t0 + 4 * (KPT * kh + q) + j;
      r.v[q][j] = t < p.L ? ld(xc + ((long)u.b * p.L + t) * p.HP) : 0.0f;
    }
}
template <int CH>
__device__ __forceinline__ void store_xt(const XtRegs<CH>& r, unsigned char* tile) {
  constexpr int KPT = 16 * CH / kSsdThreads;
  const int tid = threadIdx.x, pp = tid % CH, kh = tid / CH;
#pragma unroll
  for (int q = 0; q < KPT; q++)
    sts16(tile, tc::kmajor_row16(pp, KPT * kh + q, kQ), r.v[q][0], r.v[q][1], r.v[q][2], r.v[q][3]);
}

// Rows [t0, t0 + 64) of a [token][G][128] bf16 matrix (B or C) as a K-major tile (rows =
// tokens, K = 128 states), exact.  Thread: token tid % 64, half of the states.
__device__ __forceinline__ void load_rows(const SsdArgs& a, const Unit& u, const void* m,
                                          uint4 (&raw)[8]) {
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x, tr = tid & 63, nh = tid >> 6, t = u.t0 + tr;
  const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(m) +
                                                   (((long)u.b * p.L + t) * p.G + u.g) * kSN + 64 * nh);
#pragma unroll
  for (int j = 0; j < 8; j++) raw[j] = t < p.L ? __ldg(q + j) : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void store_rows(const uint4 (&raw)[8], unsigned char* tile) {
  const int tid = threadIdx.x, tr = tid & 63, nh = tid >> 6;
#pragma unroll
  for (int j = 0; j < 8; j++) {
    const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    sts16(tile, tc::kmajor_row16(tr, 16 * nh + 2 * j, kSN), v[0], v[1], v[2], v[3]);
    sts16(tile, tc::kmajor_row16(tr, 16 * nh + 2 * j + 1, kSN), v[4], v[5], v[6], v[7]);
  }
}

// ---- launch 1: chunk end states -------------------------------------------------------------
// Shared memory: (w B)^T [128 n][64 s] as hi and lo tiles (32 KB each), X^T [64 p][64 s] 16 KB,
// then small arrays.  Two blocks per SM.
constexpr uint32_t kStateTileA = kSN * kQ * 4, kStateTileX = kSP * kQ * 4;
constexpr uint32_t kStateSmem = 2 * kStateTileA + kStateTileX + 4 * kQ * 4 + 64;
constexpr uint32_t kStateTmCols = 64;

__global__ void __launch_bounds__(kSsdThreads) ssd_state_kernel(const __grid_constant__ SsdArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const ScanProblem& p = a.p;
  unsigned char* sAh = smem;
  unsigned char* sAl = smem + kStateTileA;
  unsigned char* sX = sAl + kStateTileA;
  float* sDl = reinterpret_cast<float*>(sX + kStateTileX);
  float* sLam = sDl + kQ;
  float* sW = sLam + kQ;
  float* sCarry = sW + kQ;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sCarry + kQ);
  uint32_t* tbase = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  const Unit u = unit_of(a, kSP);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(tbase, kStateTmCols);
  chunk_log_decay(a, u, sDl, sLam, sCarry);  // (its barriers also publish tbase and bar)
  if (tid < kQ) sW[tid] = sDl[tid] * ex2(sLam[kQ - 1] - sLam[tid]);
  __syncthreads();
  // (w B)^T [n][s] as hi + lo: thread = state n, all 64 tokens (loads first)
  {
    const __nv_bfloat16* bc = reinterpret_cast<const __nv_bfloat16*>(p.B) + (long)u.g * kSN + tid;
    float bv[kQ];
#pragma unroll
    for (int s = 0; s < kQ; s++) {
      const int t = u.t0 + s;
      bv[s] = t < p.L ? ld(bc + ((long)u.b * p.L + t) * p.G * kSN) : 0.0f;
    }
    XtRegs<kSP> xr;
    load_xt<kSP>(a, u, xr);
#pragma unroll
    for (int k4 = 0; k4 < kQ / 4; k4++) {
      float hi[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; j++) split_tf32(bv[4 * k4 + j] * sW[4 * k4 + j], hi[j], lo[j]);
      sts16(sAh, tc::kmajor_row16(tid, k4, kQ), hi[0], hi[1], hi[2], hi[3]);
      sts16(sAl, tc::kmajor_row16(tid, k4, kQ), lo[0], lo[1], lo[2], lo[3]);
    }
    store_xt<kSP>(xr, sX);
  }
  fence_async_shared();
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tm = *tbase;
  if (tid == 0) {  // D[n][p] = sum_s (w B)^T[n][s] X^T[p][s], hi and lo terms
    constexpr uint32_t id = tc::idesc_tf32(kSN, kSP);
    tc::mma_tf32_k(tm, smem_u32(sAh), smem_u32(sX), kQ, id, false);
    tc::mma_tf32_k(tm, smem_u32(sAl), smem_u32(sX), kQ, id, true);
    tc::mma_commit(bar);
  }
  const bool ok = mbar_wait(bar, 0);
  tmem_fence_after_sync();
  if (__syncthreads_or(!ok)) {
    if (tid == 0) record_status(p.status, SSM_ERR_TIMEOUT);
  } else {  // row n = tid (lane n of the M = 128 accumulator), columns p
    const int n = tid;
    float* dst = a.S + ((((long)u.b * p.H + u.h) * a.nchq + u.c) * p.P + u.p0) * kSN + n;
#pragma unroll
    for (int half = 0; half < 2; half++) {
      float v[32];
      tmem_ld32(tm + ((uint32_t)(32 * warp) << 16) + 32u * half, v);
#pragma unroll
      for (int j = 0; j < 32; j++) dst[(long)(32 * half + j) * kSN] = v[j];
    }
    if (u.pb == 0 && tid == 0) a.dec[((long)u.b * p.H + u.h) * a.nchq + u.c] = ex2(sLam[kQ - 1]);
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, kStateTmCols);
}

// ---- launch 2: start states in chunk order ----------------------------------------------------
// One thread per state element walks the chunks in order; the chunk states are read 8 chunks at
// a time so that their loads are in flight together (one at a time, each chunk waited on the
// previous one's load).
constexpr int kPassBatch = 8;

__global__ void ssd_pass_kernel(const __grid_constant__ SsdArgs a) {
  const ScanProblem& p = a.p;
  const long total = (long)p.ns * p.H * p.P * kSN;
  float* __restrict__ S = a.S;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i % kSN);
    const long r = i / kSN;
    const int pp = (int)(r % p.P);
    const int h = (int)((r / p.P) % p.H), b = (int)(r / ((long)p.P * p.H));
    const int ch = h * p.P + pp;
    const float* row = start_row(p, b);
    float hv = row ? row[(long)ch * kSN + n] : 0.0f;
    const long cstride = (long)p.P * kSN;  // between consecutive chunks of one element
    float* sp = S + (((long)b * p.H + h) * a.nchq * p.P + pp) * kSN + n;
    const float* dp = a.dec + ((long)b * p.H + h) * a.nchq;
    for (int c0 = 0; c0 < a.nchq; c0 += kPassBatch) {
      float sv[kPassBatch], dv[kPassBatch];
#pragma unroll
      for (int j = 0; j < kPassBatch; j++) {
        const bool in = c0 + j < a.nchq;
        sv[j] = in ? sp[(c0 + j) * cstride] : 0.0f;
        dv[j] = in ? __ldg(dp + c0 + j) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kPassBatch; j++) {
        const int c = c0 + j;
        if (c >= a.nchq) break;
        sp[c * cstride] = hv;  // the start state of chunk c
        if (a.ckpt && (c * kQ) % p.chunk == 0)
          a.ckpt[(((long)b * p.n_chunks + c * kQ / p.chunk) * p.HP + ch) * kSN + n] = hv;
        hv = fmaf(dv[j], hv, sv[j]);
      }
    }
    if (a.state_out) a.state_out[((long)b * p.HP + ch) * kSN + n] = hv;
  }
}

// ---- launch 3: outputs ----------------------------------------------------------------------
// Shared memory: C [64 t][128 n] 32 KB; B [64 s][128 n] 32 KB, after G the hi and lo tiles of W
// [64 t][64 s]; X^T [32 p][64 s] 8 KB; h_start^T [32 p][128 n] as hi and lo tiles (16 KB
// each).  Two blocks per SM; tensor memory: G (64 columns), Y' and Y (32 each).
constexpr uint32_t kOutC = kQ * kSN * 4, kOutB = kQ * kSN * 4, kOutX = kSPo * kQ * 4,
                   kOutH = kSPo * kSN * 4, kOutW = kQ * kQ * 4;
constexpr uint32_t kOutSmem = kOutC + kOutB + kOutX + 2 * kOutH + 3 * kQ * 4 + 64;
constexpr uint32_t kOutTmCols = 128;
constexpr uint32_t kTmG = 0, kTmYs = 64, kTmY = 96;

__global__ void __launch_bounds__(kSsdThreads) ssd_out_kernel(const __grid_constant__ SsdArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const ScanProblem& p = a.p;
  unsigned char* sC = smem;
  unsigned char* sB = sC + kOutC;  // B, then W hi (first 16 KB) and W lo
  unsigned char* sX = sB + kOutB;
  unsigned char* sHh = sX + kOutX;
  unsigned char* sHl = sHh + kOutH;
  float* sDl = reinterpret_cast<float*>(sHl + kOutH);
  float* sLam = sDl + kQ;
  float* sCarry = sLam + kQ;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sCarry + kQ);  // [2]
  uint32_t* tbase = reinterpret_cast<uint32_t*>(bar + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Unit u = unit_of(a, kSPo);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(tbase, kOutTmCols);
  // every staging load first: C, B, X^T and h_start^T (thread = channel tid % 32, a quarter
  // of the states, as hi + lo)
  uint4 craw[8], braw[8];
  load_rows(a, u, p.C, craw);
  load_rows(a, u, p.B, braw);
  XtRegs<kSPo> xr;
  load_xt<kSPo>(a, u, xr);
  float4 hv4[8];
  {
    const int pp = tid & 31, nq = tid >> 5;
    const float4* hs = reinterpret_cast<const float4*>(
        a.S + ((((long)u.b * p.H + u.h) * a.nchq + u.c) * p.P + u.p0 + pp) * kSN + 32 * nq);
#pragma unroll
    for (int k = 0; k < 8; k++) hv4[k] = hs[k];
  }
  chunk_log_decay(a, u, sDl, sLam, sCarry);
  store_rows(craw, sC);
  store_rows(braw, sB);
  store_xt<kSPo>(xr, sX);
  {
    const int pp = tid & 31, nq = tid >> 5;
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const float4 v = hv4[k];
      float h[4], l[4];
      split_tf32(v.x, h[0], l[0]);
      split_tf32(v.y, h[1], l[1]);
      split_tf32(v.z, h[2], l[2]);
      split_tf32(v.w, h[3], l[3]);
      sts16(sHh, tc::kmajor_row16(pp, 8 * nq + k, kSN), h[0], h[1], h[2], h[3]);
      sts16(sHl, tc::kmajor_row16(pp, 8 * nq + k, kSN), l[0], l[1], l[2], l[3]);
    }
  }
  fence_async_shared();
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tm = *tbase;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  if (tid == 0) {
    // G[t][s] = C_t . B_s;  Y'[t][p] = C_t . h_start[p] (hi and lo terms)
    tc::mma_tf32_k(tm + kTmG, smem_u32(sC), smem_u32(sB), kSN, tc::idesc_tf32(kQ, kQ), false);
    constexpr uint32_t id32 = tc::idesc_tf32(kQ, kSPo);
    tc::mma_tf32_k(tm + kTmYs, smem_u32(sC), smem_u32(sHh), kSN, id32, false);
    tc::mma_tf32_k(tm + kTmYs, smem_u32(sC), smem_u32(sHl), kSN, id32, true);
    tc::mma_commit(&bar[0]);
  }
  bool ok = mbar_wait(&bar[0], 0);
  tmem_fence_after_sync();
  if (!__syncthreads_or(!ok)) {
    // W[t][s] = G[t][s] delta_s 2^(Lambda_t - Lambda_s) for s <= t, as hi + lo in B's space;
    // row t = 16 warp + lane (lanes < 16 of the M = 64 accumulator)
    unsigned char* sWh = sB;
    unsigned char* sWl = sB + kOutW;
    const int t = 16 * warp + (lane & 15);
#pragma unroll
    for (int half = 0; half < 2; half++) {
      float g[32];
      tmem_ld32(tm + kTmG + lane_base + 32u * half, g);
      if (lane < 16) {
#pragma unroll
        for (int q4 = 0; q4 < 8; q4++) {
          float wh[4], wl[4];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            const int s = 32 * half + 4 * q4 + j;
            const float w = s <= t ? g[4 * q4 + j] * sDl[s] * ex2(sLam[t] - sLam[s]) : 0.0f;
            split_tf32(w, wh[j], wl[j]);
          }
          sts16(sWh, tc::kmajor_row16(t, 8 * half + q4, kQ), wh[0], wh[1], wh[2], wh[3]);
          sts16(sWl, tc::kmajor_row16(t, 8 * half + q4, kQ), wl[0], wl[1], wl[2], wl[3]);
        }
      }
    }
    fence_async_shared();
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (tid == 0) {  // Y[t][p] = sum_s W[t][s] X^T[p][s], hi and lo terms
      constexpr uint32_t id32 = tc::idesc_tf32(kQ, kSPo);
      tc::mma_tf32_k(tm + kTmY, smem_u32(sWh), smem_u32(sX), kQ, id32, false);
      tc::mma_tf32_k(tm + kTmY, smem_u32(sWl), smem_u32(sX), kQ, id32, true);
      tc::mma_commit(&bar[1]);
    }
    ok = mbar_wait(&bar[1], 0);
    tmem_fence_after_sync();
    if (!__syncthreads_or(!ok)) {
      // y_t = Y_t + 2^(Lambda_t) Y'_t (+ D x)(* silu(z)); row t = 16 warp + lane (lanes < 16)
      const int tt = u.t0 + t;
      const bool store = lane < 16 && tt < p.L && a.y;
      const float e = ex2(sLam[t]);
      const long yrow = ((long)u.b * p.L + tt) * p.HP + u.h * p.P + u.p0;
      const __nv_bfloat16* X = reinterpret_cast<const __nv_bfloat16*>(p.x);
      const __nv_bfloat16* Z = reinterpret_cast<const __nv_bfloat16*>(p.z);
      float yv[32], ys[32];
      tmem_ld32(tm + kTmY + lane_base, yv);
      tmem_ld32(tm + kTmYs + lane_base, ys);
      if (store) {
#pragma unroll
        for (int q8 = 0; q8 < kSPo / 8; q8++) {
          const int p8 = 8 * q8;
          float xv[8], zv[8], o[8];
          if (p.D) ld8_bf16(X + yrow + p8, true, xv);
          if (Z) ld8_bf16(Z + yrow + p8, true, zv);
#pragma unroll
          for (int j = 0; j < 8; j++) {
            float v = fmaf(e, ys[p8 + j], yv[p8 + j]);
            if (p.D) v = fmaf(__ldg(p.D + u.h * p.P + u.p0 + p8 + j), xv[j], v);
            if (Z) v *= siluf_(zv[j]);
            if (p.check_finite && !isfinite(v)) record_status(p.status, SSM_ERR_NONFINITE);
            o[j] = v;
          }
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            const __nv_bfloat162 hb = __floats2bfloat162_rn(o[2 * j], o[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&hb);
          }
          *reinterpret_cast<uint4*>(a.y + yrow + p8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    } else if (tid == 0) {
      record_status(p.status, SSM_ERR_TIMEOUT);
    }
  } else if (tid == 0) {
    record_status(p.status, SSM_ERR_TIMEOUT);
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, kOutTmCols);
}

bool aligned16(const void* q) { return q == nullptr || ((uintptr_t)q & 15) == 0; }

// The shape test alone sizes the workspace (the sizing calls carry no pointers); a launch also
// needs the pointers the kernels read with 16-byte loads aligned.
bool ssd_shape_ok(const ScanProblem& p) {
  return p.chunked && !p.a_per_state && p.io == SSM_BF16 && p.N == kSN && p.P % kSP == 0 &&
         p.chunk % kQ == 0 && p.H % p.G == 0 && !p.sx;
}
bool ssd_applies(const ScanProblem& p) {
  return ssd_shape_ok(p) && p.x && aligned16(p.x) && aligned16(p.B) && aligned16(p.C) &&
         aligned16(p.z);
}

size_t ssd_bytes(const ScanProblem& p, size_t* off_dec) {
  const int nchq = (p.L + kQ - 1) / kQ;
  size_t off = kStatusBytes;
  off = align_up(off + sizeof(float) * (size_t)p.ns * p.H * nchq * p.P * kSN, 256);
  *off_dec = off;
  off = align_up(off + sizeof(float) * (size_t)p.ns * p.H * nchq, 256);
  return off;
}

}  // namespace

size_t scan_fwd_ssd_ws_bytes(const ScanProblem& p) {
  size_t od;
  return ssd_shape_ok(p) ? ssd_bytes(p, &od) : 0;
}

cudaError_t launch_scan_fwd_ssd(const ScanProblem& p, void* y, float* state_out, float* ckpt,
                                void* ws, cudaStream_t st) {
  if (!ssd_applies(p) || !aligned16(y)) return cudaErrorNotSupported;
  size_t off_dec;
  ssd_bytes(p, &off_dec);
  SsdArgs a{};
  a.p = p;
  a.nchq = (p.L + kQ - 1) / kQ;
  a.npb = p.P / kSP;  // the state kernel's channel blocks; the output kernel's below
  a.S = reinterpret_cast<float*>((char*)ws + kStatusBytes);
  a.dec = reinterpret_cast<float*>((char*)ws + off_dec);
  a.state_out = state_out;
  a.ckpt = ckpt;
  a.y = reinterpret_cast<__nv_bfloat16*>(y);
  cudaError_t e = cudaFuncSetAttribute(ssd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kStateSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ssd_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kOutSmem);
  if (e != cudaSuccess) return e;
  const long units = (long)p.ns * p.H * a.nchq * a.npb;
  ssd_state_kernel<<<(unsigned)units, kSsdThreads, kStateSmem, st>>>(a), count_launches(1);
  const long total = (long)p.ns * p.H * p.P * kSN;
  const long nb = (total + 255) / 256;
  ssd_pass_kernel<<<(unsigned)(nb < 8192 ? nb : 8192), 256, 0, st>>>(a), count_launches(1);
  if (y) {  // (checkpoints only: the start states are all there is to compute)
    SsdArgs ao = a;
    ao.npb = p.P / kSPo;
    const long units_o = (long)p.ns * p.H * a.nchq * ao.npb;
    ssd_out_kernel<<<(unsigned)units_o, kSsdThreads, kOutSmem, st>>>(ao), count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace ssm

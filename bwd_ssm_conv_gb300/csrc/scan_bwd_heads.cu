// scan_bwd_heads.cu -- backward scan for the Mamba-2 form: one A per head, head_dim a multiple of
// 32, d_state 128 (ggmlR's ssm_scan_back with a [1, n_head] A; the adjoint of infotheory's
// mamba1/model.rs accumulate_token_step_gradients with the decay shared by a head's states).
//
// A block = 128 threads = 32 channels of one head x 128 states, one sequence, one time segment;
// a thread holds a 4-channel x 8-state tile (the forward's tile, scan_fwd_heads.cu).  Per chunk
// (last to first): level 1 walks the chunk's 16-token tiles forward from the checkpoint and keeps
// the state at every 8-token half-tile start (global scratch); level 2 walks the tiles in
// reverse, and per half-tile recomputes its 8 states into tensor memory (a thread's 32 states x
// 8 tokens: 256 columns of its lane, half the SM's, which register pressure leaves at 2 blocks
// per SM anyway) and runs the adjoint over them, reading each h_{t-1} back with one 32-column
// load:
//   dh = gy C + carry,  carry <- a dh,  w = carry h_prev
//   dx = gy D + delta sum_n dh B,  ddelta_head = sum_p x sum_n dh B + A sum_{p,n} w,
//   dA_head += delta sum_{p,n} w,  dB_t = sum_{h,p} dh delta x,  dC_t = sum_{h,p} gy h
// The sums over a channel's states close inside the warp (transposed shuffles); dB/dC are summed
// over the warp's two channel groups by shuffle and over the block's warps in shared memory every
// 4 tokens, in a fixed order, then over blocks by reduce_bc_kernel.  Segments, their adjoint carry
// and the d_s0 reduction are the general backward's (scan_bwd.cu).
#include "scan_bwd.cuh"
#include "tmem.cuh"

namespace ssm {

namespace {

constexpr int kBhThreads = 128;
constexpr int kBhWarps = kBhThreads / 32;
constexpr int kBhP = 32;     // channels per block
constexpr int kBhN = 128;    // d_state
constexpr int kBhTP = 4;     // channels per thread
constexpr int kBhTN = 8;     // states per thread
constexpr int kBhTile = 16;  // tokens per tile
constexpr int kBhSub = 8;    // tokens per half-tile (the history held in tensor memory)
constexpr uint32_t kBhTmCols = 256;  // 8 records x 32 states per lane
constexpr int kBhGrp = 4;    // tokens per shared-memory dB/dC sum
constexpr int kBhTS = kBhTP * kBhTN;  // states per thread

struct BhArgs {
  BwdArgs a;       // problem, gradients, segment buffers of the general plan
  int bph;         // blocks per head (P / 32)
  int bpg;         // blocks per group ((H / G) * bph)
  int vec;         // x, dy, z, B, C allow 4-element vector loads
  float* bnd;      // [blocks][S][half-tiles per chunk][threads][32]  half-tile start states
  float* part_dd;  // [ns * L][H][bph]   d delta partial of the block (before softplus')
  float* dA_blk;   // [ns][S][H][bph]
};

// Shared memory of one tile (floats).
struct BhSmem {
  float x[kBhTile][kBhP], gy[kBhTile][kBhP], dlx[kBhTile][kBhP], dyg[kBhTile][kBhP];
  float B[kBhTile][kBhN], C[kBhTile][kBhN];
  float tc[kBhTile][4];                   // (decay c, delta, softplus', decay s)
  float q[kBhTile][kBhP][2];              // per channel: sum_n dh B, sum_n C h
  float w[kBhTile][kBhWarps];             // per warp: sum of w over its states
  float red[kBhGrp][kBhWarps][2 * kBhN];  // per warp: dB (0..127), dC (128..255)
  float dd[kBhThreads];                   // per thread: dD accumulators, then dA
};

// 4 consecutive values (16 bytes of fp32, 8 of bf16; aligned) as fp32.
template <typename IO>
__device__ __forceinline__ float4 bh_ld4(const IO* p) {
  if constexpr (sizeof(IO) == 4) {
    return __ldg(reinterpret_cast<const float4*>(p));
  } else {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  }
}

template <typename IO>
__device__ __forceinline__ float bh_ld(const IO* p) {
  if constexpr (sizeof(IO) == 4) return __ldg(reinterpret_cast<const float*>(p));
  else return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p)));
}

// Loads tokens [t0, t0 + cnt) of this block: x, delta (and decay) always; dy, z, C and the
// per-(token, channel) adjoint inputs when `adjoint`.  Tokens past cnt are zero.
template <typename IO, bool ACC>
__device__ void bh_load_tile(const BhArgs& A, BhSmem& S, long tok0, int cnt, int ch0, int h,
                             int g, float A2, float bias, bool adjoint) {
  const ScanProblem& p = A.a.p;
  const int tid = threadIdx.x;
  __syncthreads();  // every thread is done with the previous tile
  if (tid < kBhTile) {
    float dl = 0.0f, spg = 1.0f;
    if (tid < cnt) {
      const float raw = bh_ld(reinterpret_cast<const IO*>(p.dt) + (tok0 + tid) * p.H + h);
      if (p.softplus) {
        dl = softplusf_(raw + bias);
        spg = softplus_gradf_(raw + bias);
      } else {
        dl = raw;
      }
    }
    const DecayCoef k = decay_coef<ACC, true>(dl, A2);
    S.tc[tid][0] = k.c;
    S.tc[tid][3] = k.s;
    S.tc[tid][1] = dl;
    S.tc[tid][2] = spg;
  }
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int idx = tid; idx < kBhTile * kBhP / 4; idx += kBhThreads) {  // 4 channels per item
    const int i = idx / (kBhP / 4), c = (idx - i * (kBhP / 4)) * 4;
    const long off = (tok0 + i) * p.HP + ch0 + c;
    const bool in = i < cnt;
    float xs[4], gys[4], dygs[4];
    float4 v = zero4, dv = zero4, zv4 = zero4;
    if (in) {
      if (A.vec) {
        v = bh_ld4(reinterpret_cast<const IO*>(p.x) + off);
        if (adjoint) dv = bh_ld4(reinterpret_cast<const IO*>(A.a.g.dy) + off);
        if (adjoint && p.z) zv4 = bh_ld4(reinterpret_cast<const IO*>(p.z) + off);
      } else {
        const IO* xp = reinterpret_cast<const IO*>(p.x) + off;
        v = make_float4(bh_ld(xp), bh_ld(xp + 1), bh_ld(xp + 2), bh_ld(xp + 3));
        if (adjoint) {
          const IO* yp = reinterpret_cast<const IO*>(A.a.g.dy) + off;
          dv = make_float4(bh_ld(yp), bh_ld(yp + 1), bh_ld(yp + 2), bh_ld(yp + 3));
          if (p.z) {
            const IO* zp = reinterpret_cast<const IO*>(p.z) + off;
            zv4 = make_float4(bh_ld(zp), bh_ld(zp + 1), bh_ld(zp + 2), bh_ld(zp + 3));
          }
        }
      }
    }
    xs[0] = v.x; xs[1] = v.y; xs[2] = v.z; xs[3] = v.w;
    const float dys[4] = {dv.x, dv.y, dv.z, dv.w}, zs[4] = {zv4.x, zv4.y, zv4.z, zv4.w};
#pragma unroll
    for (int e = 0; e < 4; e++) {
      gys[e] = dys[e];
      dygs[e] = 0.0f;
      if (adjoint && p.z && in) {
        const float sg = sigmoidf_(zs[e]);
        gys[e] = dys[e] * zs[e] * sg;
        dygs[e] = dys[e] * sg * (1.0f + zs[e] * (1.0f - sg));
      }
    }
    *reinterpret_cast<float4*>(&S.x[i][c]) = v;
    if (adjoint) {
      *reinterpret_cast<float4*>(&S.gy[i][c]) = make_float4(gys[0], gys[1], gys[2], gys[3]);
      *reinterpret_cast<float4*>(&S.dyg[i][c]) = make_float4(dygs[0], dygs[1], dygs[2], dygs[3]);
    }
  }
  for (int idx = tid; idx < kBhTile * kBhN / 4; idx += kBhThreads) {  // 4 states per item
    const int i = idx / (kBhN / 4), n = (idx - i * (kBhN / 4)) * 4;
    const long off = ((tok0 + i) * p.G + g) * kBhN + n;
    const bool in = i < cnt;
    const IO* bp = reinterpret_cast<const IO*>(p.B) + off;
    const IO* cp = reinterpret_cast<const IO*>(p.C) + off;
    float4 bv = zero4, cv = zero4;
    if (in) {
      bv = A.vec ? bh_ld4(bp) : make_float4(bh_ld(bp), bh_ld(bp + 1), bh_ld(bp + 2), bh_ld(bp + 3));
      if (adjoint)
        cv = A.vec ? bh_ld4(cp) : make_float4(bh_ld(cp), bh_ld(cp + 1), bh_ld(cp + 2), bh_ld(cp + 3));
    }
    *reinterpret_cast<float4*>(&S.B[i][n]) = bv;
    if (adjoint) *reinterpret_cast<float4*>(&S.C[i][n]) = cv;
  }
  __syncthreads();
  for (int idx = tid; idx < kBhTile * kBhP; idx += kBhThreads) {
    const int i = idx / kBhP, c = idx - i * kBhP;
    S.dlx[i][c] = S.tc[i][1] * S.x[i][c];
  }
  __syncthreads();
}

// Sum over the 16 state-group lanes (bits 0..3) of 8 per-lane values, transposed over bits 3, 2
// and 1: lane with bits (3,2,1) = k ends with the total of value k (bit 0 lanes agree).
__device__ __forceinline__ float bh_sum16_transposed(const float (&v)[8], int lane) {
  const bool u3 = lane & 8, u2 = lane & 4, u1 = lane & 2;
  float w[4], x[2];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const float snd = u3 ? v[k] : v[k + 4], kp = u3 ? v[k + 4] : v[k];
    w[k] = kp + __shfl_xor_sync(0xffffffffu, snd, 8);
  }
#pragma unroll
  for (int k = 0; k < 2; k++) {
    const float snd = u2 ? w[k] : w[k + 2], kp = u2 ? w[k + 2] : w[k];
    x[k] = kp + __shfl_xor_sync(0xffffffffu, snd, 4);
  }
  const float snd = u1 ? x[0] : x[1], kp = u1 ? x[1] : x[0];
  float y = kp + __shfl_xor_sync(0xffffffffu, snd, 2);
  return y + __shfl_xor_sync(0xffffffffu, y, 1);
}

// A thread's 32 states to / from 32 columns of its tensor-memory lane (one warp-wide access).
__device__ __forceinline__ void bh_tm_store(uint32_t taddr, const f2_t (&v)[kBhTP][kBhTN / 2]) {
  uint32_t r[32];
#pragma unroll
  for (int c = 0; c < kBhTP; c++)
#pragma unroll
    for (int q = 0; q < kBhTN / 2; q++) {
      float lo, hi;
      f2_unpack(v[c][q], lo, hi);
      r[c * kBhTN + 2 * q] = __float_as_uint(lo);
      r[c * kBhTN + 2 * q + 1] = __float_as_uint(hi);
    }
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void bh_tm_load(uint32_t taddr, f2_t (&v)[kBhTP][kBhTN / 2]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int c = 0; c < kBhTP; c++)
#pragma unroll
    for (int q = 0; q < kBhTN / 2; q++)
      v[c][q] = f2_pack(__uint_as_float(r[c * kBhTN + 2 * q]),
                        __uint_as_float(r[c * kBhTN + 2 * q + 1]));
}

// A thread's 32 states (4 channels x 8 states as 16 pairs) to / from a scratch slot.
__device__ __forceinline__ void bh_store(float* slot, const f2_t (&v)[kBhTP][kBhTN / 2]) {
  float4* d = reinterpret_cast<float4*>(slot);
#pragma unroll
  for (int c = 0; c < kBhTP; c++)
#pragma unroll
    for (int q = 0; q < kBhTN / 2; q += 2) {
      float a0, a1, a2, a3;
      f2_unpack(v[c][q], a0, a1);
      f2_unpack(v[c][q + 1], a2, a3);
      d[c * 2 + q / 2] = make_float4(a0, a1, a2, a3);
    }
}
__device__ __forceinline__ void bh_load(const float* slot, f2_t (&v)[kBhTP][kBhTN / 2]) {
  const float4* d = reinterpret_cast<const float4*>(slot);
#pragma unroll
  for (int c = 0; c < kBhTP; c++)
#pragma unroll
    for (int q = 0; q < kBhTN / 2; q += 2) {
      const float4 u = d[c * 2 + q / 2];
      v[c][q] = f2_pack(u.x, u.y);
      v[c][q + 1] = f2_pack(u.z, u.w);
    }
}

template <typename IO>
__global__ void __launch_bounds__(kBhThreads)
scan_bwd_heads_kernel(const BhArgs A) {
  constexpr bool ACC = sizeof(IO) == 4;  // accurate decay form for fp32 I/O
  constexpr int TT = kBhTile, N = kBhN;
  const BwdArgs& a = A.a;
  const ScanProblem& p = a.p;
  __shared__ __align__(16) BhSmem S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ng = lane & 15, pgl = lane >> 4;
  const int pl0 = warp * 8 + pgl * kBhTP;  // first of the thread's 4 channels, within the block
  const int n0 = ng * kBhTN;               // first of its 8 states
  const int h = blockIdx.x / A.bph, pb = blockIdx.x - h * A.bph;
  const int ch0 = h * p.P + pb * kBhP;
  const int hpg = p.H / p.G, g = h / hpg;
  const int big = (h - g * hpg) * A.bph + pb;  // the block's index within its group
  const int s = blockIdx.y, b = blockIdx.z;
  const int c_first = s * a.seg_chunks, c_last = min(a.nch_b, c_first + a.seg_chunks) - 1;
  const float Ah = __ldg(p.A + h), A2 = Ah * kLog2e;
  const float bias = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + h) : 0.0f;
  const int hpc_chunk = a.chunk_b / kBhSub;
  const long blk = ((long)b * a.S + s) * gridDim.x + blockIdx.x;
  float* bnd = A.bnd + blk * hpc_chunk * kBhThreads * kBhTS;
  auto bnd_slot = [&](int j) { return bnd + ((long)j * kBhThreads + tid) * kBhTS; };
  // the half-tile history: record k (the state after token k of the half-tile) in columns
  // 32 k .. 32 k + 31 of this thread's lane
  __shared__ uint32_t sTmem;
  __syncwarp();
  if (warp == 0) tmem_alloc(&sTmem, kBhTmCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tm = sTmem + ((uint32_t)(warp * 32) << 16);

  f2_t carry[kBhTP][kBhTN / 2];
#pragma unroll
  for (int c = 0; c < kBhTP; c++) {
    const long row = (long)(ch0 + pl0 + c) * N + n0;
#pragma unroll
    for (int q = 0; q < kBhTN / 2; q++) {
      float v0 = 0.0f, v1 = 0.0f;
      if (a.S > 1) {
        const float* src = a.segend + ((long)b * a.S + s) * p.HP * N + row + 2 * q;
        v0 = src[0];
        v1 = src[1];
      } else if (a.g.d_state_out) {
        const float* src = a.g.d_state_out + (long)b * p.HP * N + row + 2 * q;
        v0 = __ldg(src);
        v1 = __ldg(src + 1);
      }
      carry[c][q] = f2_pack(v0, v1);
    }
  }
  float dA_acc = 0.0f, dD_acc = 0.0f;

  for (int ck = c_last; ck >= c_first; ck--) {
    const int t0c = ck * a.chunk_b, t1c = min(p.L, t0c + a.chunk_b);
    const int nt = (t1c - t0c + TT - 1) / TT;
    // ---- level 1: the chunk forward from its checkpoint, keeping every tile's start --------
    f2_t hv[kBhTP][kBhTN / 2];
    {
      const float* src = a.ckpt + ((long)b * a.nch_b + ck) * p.HP * N;
#pragma unroll
      for (int c = 0; c < kBhTP; c++)
#pragma unroll
        for (int q = 0; q < kBhTN / 2; q++) {
          const float* r = src + (long)(ch0 + pl0 + c) * N + n0 + 2 * q;
          hv[c][q] = f2_pack(r[0], r[1]);
        }
    }
    for (int j = 0; j < nt; j++) {
      const int t0 = t0c + j * TT, cnt = min(TT, t1c - t0);
      bh_load_tile<IO, ACC>(A, S, (long)b * p.L + t0, cnt, ch0, h, g, A2, bias, false);
      for (int i = 0; i < cnt; i++) {
        if (i % kBhSub == 0) bh_store(bnd_slot(2 * j + i / kBhSub), hv);
        const DecayCoef2 cf2 = decay_pair(DecayCoef{S.tc[i][0], S.tc[i][3]});
        const float4 b0 = *reinterpret_cast<const float4*>(&S.B[i][n0]);
        const float4 b1 = *reinterpret_cast<const float4*>(&S.B[i][n0 + 4]);
        const f2_t B2[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                            f2_pack(b1.z, b1.w)};
        const float4 dx = *reinterpret_cast<const float4*>(&S.dlx[i][pl0]);
        const float dxs[4] = {dx.x, dx.y, dx.z, dx.w};
#pragma unroll
        for (int c = 0; c < kBhTP; c++) {
          const f2_t dx2 = f2_pack(dxs[c], dxs[c]);
#pragma unroll
          for (int q = 0; q < kBhTN / 2; q++) hv[c][q] = step2<ACC>(cf2, hv[c][q], f2_mul(dx2, B2[q]));
        }
      }
    }
    // ---- level 2: tiles in reverse; per half-tile, recompute into tensor memory, then the
    // adjoint over it ----------------------------------------------------------------------
    for (int j = nt - 1; j >= 0; j--) {
      const int t0 = t0c + j * TT, cnt = min(TT, t1c - t0);
      const long tok0 = (long)b * p.L + t0;
      bh_load_tile<IO, ACC>(A, S, tok0, cnt, ch0, h, g, A2, bias, true);
      for (int hf = (cnt - 1) / kBhSub; hf >= 0; hf--) {
        const int i_lo = hf * kBhSub, i_hi = min(cnt, i_lo + kBhSub);
        bh_load(bnd_slot(2 * j + hf), hv);
        for (int i = i_lo; i < i_hi; i++) {
          const DecayCoef2 cf2 = decay_pair(DecayCoef{S.tc[i][0], S.tc[i][3]});
          const float4 b0 = *reinterpret_cast<const float4*>(&S.B[i][n0]);
          const float4 b1 = *reinterpret_cast<const float4*>(&S.B[i][n0 + 4]);
          const f2_t B2[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                              f2_pack(b1.z, b1.w)};
          const float4 dx = *reinterpret_cast<const float4*>(&S.dlx[i][pl0]);
          const float dxs[4] = {dx.x, dx.y, dx.z, dx.w};
#pragma unroll
          for (int c = 0; c < kBhTP; c++) {
            const f2_t dx2 = f2_pack(dxs[c], dxs[c]);
#pragma unroll
            for (int q = 0; q < kBhTN / 2; q++) hv[c][q] = step2<ACC>(cf2, hv[c][q], f2_mul(dx2, B2[q]));
          }
          if (i + 1 < i_hi) bh_tm_store(tm + 32u * (uint32_t)(i - i_lo), hv);
        }
        tmem_wait_st();
        // hv = the state after the half-tile's last token: h_t of its first adjoint step
        for (int i = i_hi - 1; i >= i_lo; i--) {
          f2_t hp[kBhTP][kBhTN / 2];  // h_{t-1}
          if (i > i_lo) bh_tm_load(tm + 32u * (uint32_t)(i - 1 - i_lo), hp);
          else bh_load(bnd_slot(2 * j + hf), hp);
          const DecayCoef2 cf2 = decay_pair(DecayCoef{S.tc[i][0], S.tc[i][3]});
          const float dl = S.tc[i][1];
          const float4 b0 = *reinterpret_cast<const float4*>(&S.B[i][n0]);
          const float4 b1 = *reinterpret_cast<const float4*>(&S.B[i][n0 + 4]);
          const float4 c0 = *reinterpret_cast<const float4*>(&S.C[i][n0]);
          const float4 c1 = *reinterpret_cast<const float4*>(&S.C[i][n0 + 4]);
          const f2_t B2[4] = {f2_pack(b0.x, b0.y), f2_pack(b0.z, b0.w), f2_pack(b1.x, b1.y),
                              f2_pack(b1.z, b1.w)};
          const f2_t C2[4] = {f2_pack(c0.x, c0.y), f2_pack(c0.z, c0.w), f2_pack(c1.x, c1.y),
                              f2_pack(c1.z, c1.w)};
          const float4 gyv = *reinterpret_cast<const float4*>(&S.gy[i][pl0]);
          const float4 dlxv = *reinterpret_cast<const float4*>(&S.dlx[i][pl0]);
          const float gys[4] = {gyv.x, gyv.y, gyv.z, gyv.w};
          const float dlxs[4] = {dlxv.x, dlxv.y, dlxv.z, dlxv.w};
          f2_t dB2[4] = {0ull, 0ull, 0ull, 0ull}, dC2[4] = {0ull, 0ull, 0ull, 0ull}, w2 = 0ull;
          float v8[8];
#pragma unroll
          for (int c = 0; c < kBhTP; c++) {
            const f2_t gy2 = f2_pack(gys[c], gys[c]), dlx2 = f2_pack(dlxs[c], dlxs[c]);
            f2_t sb = 0ull, yp = 0ull;
#pragma unroll
            for (int q = 0; q < kBhTN / 2; q++) {
              const f2_t dh = f2_fma(gy2, C2[q], carry[c][q]);
              sb = f2_fma(dh, B2[q], sb);
              dB2[q] = f2_fma(dh, dlx2, dB2[q]);
              dC2[q] = f2_fma(gy2, hv[c][q], dC2[q]);
              yp = f2_fma(C2[q], hv[c][q], yp);
              const f2_t cn = apply2<ACC>(cf2, dh);
              w2 = f2_fma(cn, hp[c][q], w2);
              carry[c][q] = cn;
            }
            v8[c] = f2_sum(sb);
            v8[4 + c] = f2_sum(yp);
          }
          const float wsum = f2_sum(w2);
          dA_acc = fmaf(dl, wsum, dA_acc);
          // per channel: sum over the 128 states (lanes 0..15 of the half-warp)
          const float tot = bh_sum16_transposed(v8, lane);
          if ((lane & 1) == 0) {
            const int k = ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
            S.q[i][pl0 + (k & 3)][k >> 2] = tot;
          }
          // dB, dC: sum over the warp's two channel groups (lane bit 4), transposed
          {
            const bool u4 = lane & 16;
            float r[8];
#pragma unroll
            for (int q = 0; q < 4; q++) {
              float b_lo, b_hi, c_lo, c_hi;
              f2_unpack(dB2[q], b_lo, b_hi);
              f2_unpack(dC2[q], c_lo, c_hi);
              r[2 * q] = (u4 ? c_lo : b_lo) + __shfl_xor_sync(0xffffffffu, u4 ? b_lo : c_lo, 16);
              r[2 * q + 1] = (u4 ? c_hi : b_hi) + __shfl_xor_sync(0xffffffffu, u4 ? b_hi : c_hi, 16);
            }
            float* dst = &S.red[i % kBhGrp][warp][(u4 ? N : 0) + n0];
            *reinterpret_cast<float4*>(dst) = make_float4(r[0], r[1], r[2], r[3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(r[4], r[5], r[6], r[7]);
          }
          // sum of w over the warp
          float wv = wsum;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) wv += __shfl_xor_sync(0xffffffffu, wv, off);
          if (lane == 0) S.w[i][warp] = wv;
#pragma unroll
          for (int c = 0; c < kBhTP; c++)
#pragma unroll
            for (int q = 0; q < kBhTN / 2; q++) hv[c][q] = hp[c][q];
          if (i % kBhGrp == 0) {  // tokens i .. i+3 complete: dB, dC of the block, fixed order
            __syncthreads();
            for (int o = tid; o < kBhGrp * 2 * N; o += kBhThreads) {
              const int k = o / (2 * N), r = o - k * 2 * N;
              if (i + k < cnt) {
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < kBhWarps; w++) v += S.red[k][w][r];
                a.part_bc[(((tok0 + i + k) * p.G + g) * A.bpg + big) * 2 * N + r] = v;
              }
            }
            __syncthreads();
          }
        }
      }
      // ---- epilogue of the tile: dx, dz per (token, channel); the block's d delta per token --
      for (int idx = tid; idx < cnt * kBhP; idx += kBhThreads) {
        const int i = idx / kBhP, c = idx - i * kBhP;  // c == tid % 32 for every item
        const float sB = S.q[i][c][0], yp = S.q[i][c][1], xv = S.x[i][c], gy = S.gy[i][c];
        const float Dv = p.D ? __ldg(p.D + ch0 + c) : 0.0f;
        const long off = (tok0 + i) * p.HP + ch0 + c;
        const float dxv = fmaf(gy, Dv, S.tc[i][1] * sB);
        const float dzv = p.z ? S.dyg[i][c] * fmaf(Dv, xv, yp) : 0.0f;
        if (p.check_finite && !(isfinite(dxv) && isfinite(dzv)))
          record_status(p.status, SSM_ERR_NONFINITE);
        st(reinterpret_cast<IO*>(a.g.d_x) + off, dxv);
        if (p.z && a.g.d_z) st(reinterpret_cast<IO*>(a.g.d_z) + off, dzv);
        dD_acc = fmaf(gy, xv, dD_acc);
      }
      for (int i = warp; i < cnt; i += kBhWarps) {
        float v = S.x[i][lane] * S.q[i][lane][0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) {
          float wt = 0.0f;
#pragma unroll
          for (int w = 0; w < kBhWarps; w++) wt += S.w[i][w];
          A.part_dd[((tok0 + i) * p.H + h) * A.bph + pb] = fmaf(Ah, wt, v);
        }
      }
    }
  }

  // ---- per block: dD per channel, dA of the head, d s0 ---------------------------------------
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(sTmem, kBhTmCols);
  S.dd[tid] = dD_acc;
  __syncthreads();
  if (tid < kBhP && a.g.d_D) {
    float v = 0.0f;
#pragma unroll
    for (int k = 0; k < kBhThreads / kBhP; k++) v += S.dd[tid + k * kBhP];
    a.dD_part[((long)b * a.S + s) * p.HP + ch0 + tid] = v;
  }
  __syncthreads();
  S.dd[tid] = dA_acc;
  __syncthreads();
  if (tid == 0) {
    float v = 0.0f;
    for (int k = 0; k < kBhThreads; k++) v += S.dd[k];
    A.dA_blk[(((long)b * a.S + s) * p.H + h) * A.bph + pb] = v;
  }
  if (s == 0) {
#pragma unroll
    for (int c = 0; c < kBhTP; c++)
#pragma unroll
      for (int q = 0; q < kBhTN / 2; q++) {
        float* d = a.dh0 + ((long)b * p.HP + ch0 + pl0 + c) * N + n0 + 2 * q;
        f2_unpack(carry[c][q], d[0], d[1]);
      }
  }
}

// d_dt[tok][h] = softplus'(pre) * sum over the head's blocks of the d delta partials.  With a
// d_dt_bias wanted, d_dt also goes back into the first partial for reduce_heads_params_kernel.
template <typename IO>
__global__ void reduce_heads_ddt_kernel(const BhArgs A) {
  const ScanProblem& p = A.a.p;
  const long total = (long)p.ns * p.L * p.H;
  const IO* dt = reinterpret_cast<const IO*>(p.dt);
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int h = (int)(i % p.H);
    float* src = A.part_dd + i * A.bph;
    float v = 0.0f;
    for (int k = 0; k < A.bph; k++) v += src[k];
    if (p.softplus) v *= softplus_gradf_(bh_ld(dt + i) + (p.dt_bias ? __ldg(p.dt_bias + h) : 0.0f));
    st(reinterpret_cast<IO*>(A.a.g.d_dt) + i, v);
    src[0] = v;
  }
}

// One block per head: dA (over sequences, segments, blocks), d_dt_bias (over tokens) and dD of
// the head's channels (over sequences, segments); strided partial sums, then a fixed-order tree.
constexpr int kRhThreads = 256;
__global__ void __launch_bounds__(kRhThreads) reduce_heads_params_kernel(const BhArgs A) {
  const BwdArgs& a = A.a;
  const ScanProblem& p = a.p;
  __shared__ float sm[kRhThreads];
  const int h = blockIdx.x, tid = threadIdx.x;
  auto block_sum = [&](float v) {
    sm[tid] = v;
    __syncthreads();
    for (int w = kRhThreads / 2; w > 0; w >>= 1) {
      if (tid < w) sm[tid] += sm[tid + w];
      __syncthreads();
    }
    const float r = sm[0];
    __syncthreads();
    return r;
  };
  float v = 0.0f;
  const int nA = p.ns * a.S * A.bph;
  for (int k = tid; k < nA; k += kRhThreads) {
    const int pb = k % A.bph, bs = k / A.bph;
    v += A.dA_blk[((long)bs * p.H + h) * A.bph + pb];
  }
  const float dA = block_sum(v);
  if (tid == 0) a.g.d_A[h] = dA;
  if (a.g.d_dt_bias) {
    v = 0.0f;
    for (long tok = tid; tok < (long)p.ns * p.L; tok += kRhThreads)
      v += A.part_dd[(tok * p.H + h) * A.bph];
    const float db = block_sum(v);
    if (tid == 0) a.g.d_dt_bias[h] = db;
  }
  if (a.g.d_D) {
    for (int pp = tid; pp < p.P; pp += kRhThreads) {
      const int ch = h * p.P + pp;
      float d = 0.0f;
      for (int bs = 0; bs < p.ns * a.S; bs++) d += a.dD_part[(long)bs * p.HP + ch];
      a.g.d_D[ch] = d;
    }
  }
}

}  // namespace

bool bwd_heads_applies(const ScanProblem& p, int chunk_b) {
  return !p.a_per_state && p.P % kBhP == 0 && p.N == kBhN && chunk_b % kBhTile == 0;
}

int bwd_heads_blocks(const ScanProblem& p) { return p.ns * p.H * (p.P / kBhP); }

size_t bwd_heads_scratch_floats(const ScanProblem& p, int S, int chunk_b) {
  const size_t blocks = (size_t)bwd_heads_blocks(p) * S;
  return blocks * (size_t)(chunk_b / kBhSub) * kBhThreads * kBhTS;
}

// Main pass and reductions of the Mamba-2-form backward (segments' local adjoint and carry
// already done by the caller when a.S > 1).  scratch: bwd_heads_scratch_floats floats.
cudaError_t launch_bwd_heads(const BwdArgs& a, float* scratch, cudaStream_t st) {
  const ScanProblem& p = a.p;
  BhArgs A;
  A.a = a;
  A.bph = p.P / kBhP;
  A.bpg = (p.H / p.G) * A.bph;
  A.a.bpg = A.bpg;  // part_bc is laid out per head-tiled block
  const size_t blocks = (size_t)bwd_heads_blocks(p) * a.S;
  (void)blocks;
  A.bnd = scratch;
  A.part_dd = a.ddt_part;
  const uintptr_t al = p.io == SSM_BF16 ? 8 : 16;
  auto ok = [&](const void* q) { return q == nullptr || ((uintptr_t)q % al) == 0; };
  A.vec = ok(p.x) && ok(a.g.dy) && ok(p.z) && ok(p.B) && ok(p.C);
  A.dA_blk = a.dA_part;
  const dim3 grid(p.H * A.bph, a.S, p.ns);
  // Each block holds kBhTmCols of the SM's 512 columns of tensor memory; unused dynamic shared
  // memory keeps a third block off the SM (it would only wait in the allocation).
  const void* kern = p.io == SSM_BF16 ? reinterpret_cast<const void*>(scan_bwd_heads_kernel<__nv_bfloat16>)
                                      : reinterpret_cast<const void*>(scan_bwd_heads_kernel<float>);
  cudaFuncAttributes fa;
  int dev = 0, smem_sm = 0, reserved = 0;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e != cudaSuccess) return e;
  const int max_blocks = (int)(512u / kBhTmCols);
  const long need = (long)smem_sm / (max_blocks + 1) + 1 - (long)fa.sharedSizeBytes - reserved;
  const size_t dyn = need > 0 ? (size_t)need : 0;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  if (p.io == SSM_BF16)
    scan_bwd_heads_kernel<__nv_bfloat16><<<grid, kBhThreads, dyn, st>>>(A), count_launches(1);
  else
    scan_bwd_heads_kernel<float><<<grid, kBhThreads, dyn, st>>>(A), count_launches(1);
  const long nbc = (long)p.ns * p.L * p.G * 2 * p.N;
  const int bbc = (int)((nbc + 255) / 256 < 8192 ? (nbc + 255) / 256 : 8192);
  const long ndt = (long)p.ns * p.L * p.H;
  const int bdt = (int)((ndt + 255) / 256 < 8192 ? (ndt + 255) / 256 : 8192);
  if (p.io == SSM_BF16) {
    reduce_bc_kernel<__nv_bfloat16><<<bbc, 256, 0, st>>>(A.a), count_launches(1);
    reduce_heads_ddt_kernel<__nv_bfloat16><<<bdt, 256, 0, st>>>(A), count_launches(1);
  } else {
    reduce_bc_kernel<float><<<bbc, 256, 0, st>>>(A.a), count_launches(1);
    reduce_heads_ddt_kernel<float><<<bdt, 256, 0, st>>>(A), count_launches(1);
  }
  reduce_heads_params_kernel<<<p.H, kRhThreads, 0, st>>>(A), count_launches(1);
  return cudaGetLastError();
}

}  // namespace ssm

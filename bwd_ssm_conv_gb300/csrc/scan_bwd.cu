// scan_bwd.cu -- selective scan backward from per-chunk checkpoints.
//
// Per token, in reverse (infotheory mamba1/model.rs accumulate_token_step_gradients; the
// reverse adjoint dh_t = C^T dy_t + a_{t+1} dh_{t+1} of kizzasi-model ssm_backward):
//   gy = dy silu(z)              dz = dy y_pre silu'(z)
//   dh = gy C + carry            dC += gy h_t          (summed over the channels of a group)
//   dB += dh delta x             dx  = gy D + delta sum_n dh B
//   w  = (a dh) h_{t-1}          ddelta = sum_n A w + x sum_n dh B
//   dA += delta w                dD += gy x            carry = a dh
//
// Gradient checkpointing (GradientCheckpointedSSM of backprop_ssm.rs; the TBPTT replay of
// online_train_segment_tbptt): a block walks its chunks last to first.  For each chunk it
// recomputes the states forward from the checkpoint, keeping the state at every 8-token
// sub-chunk start in shared memory (level 1); then, sub-chunk by sub-chunk in reverse, it
// recomputes 8 tokens keeping h and a in registers (level 2) and runs the adjoint over them.
// Unlike the segment loop printed on the kizzasi page, the adjoint carried out of a later
// chunk seeds dh at this chunk's LAST token (it is added to the C^T dy term there), not the
// chunk's initial-state gradient.
//
// Time parallelism for long sequences: segments of whole chunks, with the adjoint at each
// segment end found by the same three-launch composition as the forward (local adjoint from
// zero, sequential carry, main pass).  Cross-channel sums (dB, dC) and sums over time (dA,
// dD, d dt_bias) go through per-block partials in the workspace and a fixed-order reduce.
#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"
#include "scan_bwd.cuh"

namespace ssm {

template <typename IO, bool SCALAR_A, bool FULL>
__global__ void __launch_bounds__(kScanThreads)
scan_bwd_kernel(const BwdArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;  // accurate decay form for fp32 I/O
  extern __shared__ float4 smem4[];
  const ScanProblem& p = a.p;
  const Lane l = lane_of(a);
  const int N = p.N, Npad = l.tpc * kBwdNS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kScanThreads / 32;
  const int s = blockIdx.y, b = blockIdx.z;
  const unsigned gmask = group_mask(l.tpc);
  const int nsub_max = (a.chunk_b + kTsub - 1) / kTsub;
  float4* bnd = smem4;                                        // [nsub_max][threads]
  float* red = reinterpret_cast<float*>(smem4 + nsub_max * kScanThreads);  // [Tsub][warps][2][Npad]

  const IO* x = (const IO*)p.x;
  const IO* dt = (const IO*)p.dt;
  const IO* Bm = (const IO*)p.B;
  const IO* Cm = (const IO*)p.C;
  const IO* z = (const IO*)p.z;
  const IO* dy = (const IO*)a.g.dy;

  float An[kBwdNS], A2[kBwdNS];
#pragma unroll
  for (int j = 0; j < kBwdNS; j++) {
    const bool in = l.valid && (FULL || l.n0 + j < N);
    An[j] = in ? (SCALAR_A ? __ldg(p.A + l.h) : __ldg(p.A + (long)l.h * N + l.n0 + j)) : 0.0f;
    A2[j] = An[j] * kLog2e;
  }
  float carry[kBwdNS];
  {
    const long si = ((long)b * a.S + s) * p.HP + l.ch;
#pragma unroll
    for (int j = 0; j < kBwdNS; j++) {
      const bool in = l.valid && (FULL || l.n0 + j < N);
      float v = 0.0f;
      if (in) {
        if (a.S > 1) v = a.segend[si * N + l.n0 + j];
        else if (a.g.d_state_out) v = __ldg(a.g.d_state_out + ((long)b * p.HP + l.ch) * N + l.n0 + j);
      }
      carry[j] = v;
    }
  }
  float dA_acc[kBwdNS] = {0.f, 0.f, 0.f, 0.f};
  float dD_acc = 0.0f, dtb_acc = 0.0f;
  const float Dv = (l.valid && p.D) ? __ldg(p.D + l.ch) : 0.0f;
  const float bias = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + l.h) : 0.0f;
  const long gbase = (long)l.g * N + l.n0;  // offset of this thread's states inside a B/C token row

  const int c_first = s * a.seg_chunks;
  const int c_last = min(a.nch_b, c_first + a.seg_chunks) - 1;
  for (int ck = c_last; ck >= c_first; ck--) {
    const int t0 = ck * a.chunk_b, t1 = min(p.L, t0 + a.chunk_b);
    const int nsub = (t1 - t0 + kTsub - 1) / kTsub;
    // ---- level 1: states at every sub-chunk start, from the checkpoint -------------------
    float hs[kBwdNS];
    {
      const float* src = a.ckpt + (((long)b * a.nch_b + ck) * p.HP + l.ch) * N + l.n0;
#pragma unroll
      for (int j = 0; j < kBwdNS; j++)
        hs[j] = (l.valid && (FULL || l.n0 + j < N)) ? src[j] : 0.0f;
    }
    for (int k = 0; k < nsub; k++) {
      bnd[k * kScanThreads + threadIdx.x] = make_float4(hs[0], hs[1], hs[2], hs[3]);
      const int ts = t0 + k * kTsub, te = min(t1, ts + kTsub);
      for (int t = ts; t < te; t++) {
        const long tok = (long)b * p.L + t;
        float pre;
        const float dl = delta_of(p, dt, tok, l.h, bias, &pre);
        const float xv = l.valid ? ld(x + tok * p.HP + l.ch) : 0.0f;
        float Bv[kBwdNS];
        load_row<IO, kBwdNS, FULL>(Bm + tok * p.G * N + gbase, N - l.n0, Bv);
        const float dx = dl * xv;
        const DecayCoef as = SCALAR_A ? decay_coef<ACC, true>(dl, A2[0]) : DecayCoef{0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < kBwdNS; j++)
          hs[j] = decay_step<ACC>(SCALAR_A ? as : decay_coef<ACC, true>(dl, A2[j]), hs[j], dx * Bv[j]);
      }
    }
    // ---- level 2: per sub-chunk, last to first --------------------------------------------
    for (int k = nsub - 1; k >= 0; k--) {
      const int ts = t0 + k * kTsub;
      const int cnt = min(kTsub, t1 - ts);
      float hh[kTsub + 1][kBwdNS], dls[kTsub], xs[kTsub], pres[kTsub];
      DecayCoef aa[kTsub][kBwdNS];
      {
        const float4 v = bnd[k * kScanThreads + threadIdx.x];
        hh[0][0] = v.x; hh[0][1] = v.y; hh[0][2] = v.z; hh[0][3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < kTsub; i++) {
        if (i < cnt) {
          const long tok = (long)b * p.L + ts + i;
          float pre;
          const float dl = delta_of(p, dt, tok, l.h, bias, &pre);
          const float xv = l.valid ? ld(x + tok * p.HP + l.ch) : 0.0f;
          float Bv[kBwdNS];
          load_row<IO, kBwdNS, FULL>(Bm + tok * p.G * N + gbase, N - l.n0, Bv);
          const float dx = dl * xv;
          const DecayCoef as = SCALAR_A ? decay_coef<ACC, true>(dl, A2[0]) : DecayCoef{0.0f, 0.0f};
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) {
            aa[i][j] = SCALAR_A ? as : decay_coef<ACC, true>(dl, A2[j]);
            hh[i + 1][j] = decay_step<ACC>(aa[i][j], hh[i][j], dx * Bv[j]);
          }
          dls[i] = dl; xs[i] = xv; pres[i] = pre;
        } else {
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) {  // the identity step, a = 1
            aa[i][j] = ACC ? DecayCoef{0.0f, 1.0f} : DecayCoef{1.0f, 0.0f};
            hh[i + 1][j] = hh[i][j];
          }
          dls[i] = 0.0f; xs[i] = 0.0f; pres[i] = 0.0f;
        }
      }
#pragma unroll
      for (int i = kTsub - 1; i >= 0; i--) {
        if (i < cnt) {  // cnt is uniform over the block: no divergence around the shuffles
          const long tok = (long)b * p.L + ts + i;
          float Bv[kBwdNS], Cv[kBwdNS];
          load_row<IO, kBwdNS, FULL>(Bm + tok * p.G * N + gbase, N - l.n0, Bv);
          load_row<IO, kBwdNS, FULL>(Cm + tok * p.G * N + gbase, N - l.n0, Cv);
          const float dyv = l.valid ? ld(dy + tok * p.HP + l.ch) : 0.0f;
          float gy = dyv, ypre = 0.0f, zv = 0.0f;
          if (z) {
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < kBwdNS; j++) part = fmaf(Cv[j], hh[i + 1][j], part);
            for (int off = l.tpc >> 1; off > 0; off >>= 1)
              part += __shfl_xor_sync(gmask, part, off);
            ypre = fmaf(Dv, xs[i], part);
            zv = l.valid ? ld(z + tok * p.HP + l.ch) : 0.0f;
            gy = dyv * siluf_(zv);
          }
          const float dlx = dls[i] * xs[i];
          float sB = 0.0f, sAw = 0.0f, dBp[kBwdNS], dCp[kBwdNS];
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) {
            const float dh = fmaf(gy, Cv[j], carry[j]);
            dCp[j] = gy * hh[i + 1][j];
            sB = fmaf(dh, Bv[j], sB);
            dBp[j] = dh * dlx;
            const float cn = decay_apply<ACC>(aa[i][j], dh);
            const float w = cn * hh[i][j];
            sAw = fmaf(An[j], w, sAw);
            dA_acc[j] = fmaf(dls[i], w, dA_acc[j]);
            carry[j] = cn;
          }
          for (int off = l.tpc >> 1; off > 0; off >>= 1) {
            sB += __shfl_xor_sync(gmask, sB, off);
            sAw += __shfl_xor_sync(gmask, sAw, off);
          }
          const float dxv = fmaf(gy, Dv, dls[i] * sB);
          const float ddl = fmaf(xs[i], sB, sAw);
          const float ddt = p.softplus ? ddl * softplus_gradf_(pres[i]) : ddl;
          dD_acc = fmaf(gy, xs[i], dD_acc);
          if (l.sg == 0 && l.valid) {
            st((IO*)a.g.d_x + tok * p.HP + l.ch, dxv);
            const float dzv = z ? dyv * ypre * silu_gradf_(zv) : 0.0f;
            if (p.check_finite && !(isfinite(dxv) && isfinite(ddl) && isfinite(dzv)))
              record_status(p.status, SSM_ERR_NONFINITE);
            if (z && a.g.d_z) st((IO*)a.g.d_z + tok * p.HP + l.ch, dzv);
            if (p.P == 1) st((IO*)a.g.d_dt + tok * p.H + l.h, ddt);
            else a.ddt_part[tok * p.HP + l.ch] = ddl;
            dtb_acc += ddt;
          }
          // dB, dC: sum over the channels of this warp (lanes that hold the same states)
          for (int off = 16; off >= l.tpc; off >>= 1) {
#pragma unroll
            for (int j = 0; j < kBwdNS; j++) {
              dBp[j] += __shfl_xor_sync(0xffffffffu, dBp[j], off);
              dCp[j] += __shfl_xor_sync(0xffffffffu, dCp[j], off);
            }
          }
          if (lane < l.tpc) {
            float* rb = red + ((i * kWarps + warp) * 2) * Npad + l.n0;
#pragma unroll
            for (int j = 0; j < kBwdNS; j++) { rb[j] = dBp[j]; rb[Npad + j] = dCp[j]; }
          }
        }
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < cnt * 2 * N; idx += kScanThreads) {
        const int i = idx / (2 * N), r = idx - i * 2 * N;
        const int q = r / N, n = r - q * N;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; w++) v += red[((i * kWarps + w) * 2 + q) * Npad + n];
        const long tok = (long)b * p.L + ts + i;
        a.part_bc[((tok * p.G + l.g) * a.bpg + l.blk) * 2 * N + r] = v;
      }
      __syncthreads();
    }
  }

  if (l.valid) {
    const long si = ((long)b * a.S + s) * p.HP + l.ch;
#pragma unroll
    for (int j = 0; j < kBwdNS; j++) {
      if (FULL || l.n0 + j < N) {
        a.dA_part[si * N + l.n0 + j] = dA_acc[j];
        if (s == 0) a.dh0[((long)b * p.HP + l.ch) * N + l.n0 + j] = carry[j];
      }
    }
    if (l.sg == 0) {
      a.dD_part[si] = dD_acc;
      a.dtb_part[si] = dtb_acc;
    }
  }
}

// Local adjoint of segments 1..S-1: the gradient reaching the state just before the
// segment from the segment's own outputs (zero adjoint at its end), and sum(delta).
template <typename IO, bool SCALAR_A, bool FULL>
__global__ void __launch_bounds__(kScanThreads)
scan_bwd_local_kernel(const BwdArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;
  const ScanProblem& p = a.p;
  const Lane l = lane_of(a);
  const int N = p.N;
  const int s = blockIdx.y + 1, b = blockIdx.z;
  const unsigned gmask = group_mask(l.tpc);
  (void)gmask;
  const IO* dt = (const IO*)p.dt;
  const IO* Cm = (const IO*)p.C;
  const IO* z = (const IO*)p.z;
  const IO* dy = (const IO*)a.g.dy;
  float A2[kBwdNS];
#pragma unroll
  for (int j = 0; j < kBwdNS; j++) {
    const bool in = l.valid && (FULL || l.n0 + j < N);
    A2[j] = in ? (SCALAR_A ? __ldg(p.A + l.h) : __ldg(p.A + (long)l.h * N + l.n0 + j)) * kLog2e
               : 0.0f;
  }
  const float bias = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + l.h) : 0.0f;
  const long gbase = (long)l.g * N + l.n0;
  float c[kBwdNS] = {0.f, 0.f, 0.f, 0.f};
  float sumd = 0.0f;
  const int t_begin = s * a.seg_chunks * a.chunk_b;
  const int t_end = min(p.L, t_begin + a.seg_chunks * a.chunk_b);
  for (int t = t_end - 1; t >= t_begin; t--) {
    const long tok = (long)b * p.L + t;
    float pre;
    const float dl = delta_of(p, dt, tok, l.h, bias, &pre);
    float Cv[kBwdNS];
    load_row<IO, kBwdNS, FULL>(Cm + tok * p.G * N + gbase, N - l.n0, Cv);
    float gy = l.valid ? ld(dy + tok * p.HP + l.ch) : 0.0f;
    if (z) gy *= siluf_(l.valid ? ld(z + tok * p.HP + l.ch) : 0.0f);
    const DecayCoef as = SCALAR_A ? decay_coef<ACC, true>(dl, A2[0]) : DecayCoef{0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < kBwdNS; j++)
      c[j] = decay_apply<ACC>(SCALAR_A ? as : decay_coef<ACC, true>(dl, A2[j]), fmaf(gy, Cv[j], c[j]));
    sumd += dl;
  }
  if (l.valid) {
    const long si = ((long)b * a.S + s) * p.HP + l.ch;
#pragma unroll
    for (int j = 0; j < kBwdNS; j++)
      if (FULL || l.n0 + j < N) a.dhloc[si * N + l.n0 + j] = c[j];
    if (l.sg == 0) a.sumd[si] = sumd;
  }
}

// Adjoint at every segment end, composing segments from the last: end[s-1] =
// exp(A sum_delta[s]) end[s] + local[s]; the last segment ends at d_state_out.
constexpr int kCarryBatch = 8;
__global__ void scan_bwd_carry_kernel(const BwdArgs a) {
  const ScanProblem& p = a.p;
  const long total = (long)p.ns * p.HP * p.N;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i % p.N);
    const long bc = i / p.N;
    const int ch = (int)(bc % p.HP), b = (int)(bc / p.HP);
    const int h = ch / p.P;
    const float A2 = (p.a_per_state ? __ldg(p.A + (long)h * p.N + n) : __ldg(p.A + h)) * kLog2e;
    float c = a.g.d_state_out ? __ldg(a.g.d_state_out + i) : 0.0f;
    // segments S-1 .. 0, kCarryBatch at a time: their decays and local adjoints do not depend
    // on c, so their loads go out together ahead of the composition
    for (int s0 = a.S - 1; s0 >= 0; s0 -= kCarryBatch) {
      float dk[kCarryBatch], lv[kCarryBatch];
#pragma unroll
      for (int j = 0; j < kCarryBatch; j++) {
        const int s = s0 - j;
        const long si = ((long)b * a.S + s) * p.HP + ch;
        dk[j] = s > 0 ? ex2(A2 * a.sumd[si]) : 0.0f;
        lv[j] = s > 0 ? a.dhloc[si * p.N + n] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kCarryBatch; j++) {
        const int s = s0 - j;
        if (s < 0) break;
        a.segend[(((long)b * a.S + s) * p.HP + ch) * p.N + n] = c;
        if (s > 0) c = fmaf(dk[j], c, lv[j]);
      }
    }
  }
}

// Local adjoint of segments 1..S-1 for the Mamba-2 form (one A per head, d_state 128, head_dim
// a multiple of 16): the same reverse-time scan c <- a_t (c + gy_t C_t^T) from a zero adjoint at
// the segment's end, and sum(delta), as scan_bwd_local_kernel (same operations in the same
// order, so the same bits), on a head-tiled block: 16 channels x 128 states, each thread 4
// channels x 4 states in packed pairs.  A tile's 16 C rows, gy values and decays are staged in
// shared memory once and shared by the block, where the per-channel kernel read the group's C
// row from global memory for every channel.  (Blocks of 16 channels rather than 32: the grid
// is small, and twice the blocks measured 0.8 % faster on the whole backward.)
constexpr int kHlThreads = 128, kHlTT = 16, kHlCB = 16, kHlN = 128;
template <typename IO>
__global__ void __launch_bounds__(kHlThreads) scan_bwd_heads_local_kernel(const BwdArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;
  __shared__ __align__(16) float sC[kHlTT][kHlN];   // C rows of the tile's tokens
  __shared__ __align__(16) float sG[kHlTT][kHlCB];  // gy = dy silu(z)
  __shared__ float2 sK[kHlTT];                      // the decay coefficient (c, s)
  __shared__ float sDl[kHlTT];                      // delta
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x, cg = tid >> 5, sg = tid & 31;
  const int ch0 = blockIdx.x * kHlCB, h = ch0 / p.P, g = h / (p.H / p.G);
  const int s = blockIdx.y + 1, b = blockIdx.z;
  const IO* dt = (const IO*)p.dt;
  const IO* Cm = (const IO*)p.C;
  const IO* z = (const IO*)p.z;
  const IO* dy = (const IO*)a.g.dy;
  const float A2 = __ldg(p.A + h) * kLog2e;
  const float bias = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + h) : 0.0f;
  const int t_begin = s * a.seg_chunks * a.chunk_b;
  const int t_end = min(p.L, t_begin + a.seg_chunks * a.chunk_b);
  f2_t c2[4][2];  // channels ch0 + 4 cg + i, states 4 sg + 2 q, +1
#pragma unroll
  for (int i = 0; i < 4; i++) c2[i][0] = c2[i][1] = 0ull;
  float sumd = 0.0f;
  for (int te = t_end; te > t_begin; te -= kHlTT) {
    const int t0 = max(t_begin, te - kHlTT), cnt = te - t0;
    __syncthreads();  // every thread is done with the previous tile
    for (int idx = tid; idx < cnt * (kHlN / 4); idx += kHlThreads) {
      const int i = idx / (kHlN / 4), n4 = (idx - i * (kHlN / 4)) * 4;
      const IO* src = Cm + (((long)b * p.L + t0 + i) * p.G + g) * kHlN + n4;
      *reinterpret_cast<float4*>(&sC[i][n4]) = make_float4(ld(src), ld(src + 1), ld(src + 2), ld(src + 3));
    }
    for (int idx = tid; idx < cnt * kHlCB; idx += kHlThreads) {
      const int i = idx / kHlCB, c = idx - i * kHlCB;
      const long e = ((long)b * p.L + t0 + i) * p.HP + ch0 + c;
      float gy = ld(dy + e);
      if (z) gy *= siluf_(ld(z + e));
      sG[i][c] = gy;
    }
    if (tid < cnt) {
      float pre;
      const float dl = delta_of(p, dt, (long)b * p.L + t0 + tid, h, bias, &pre);
      const DecayCoef k = decay_coef<ACC, true>(dl, A2);
      sK[tid] = make_float2(k.c, k.s);
      sDl[tid] = dl;
    }
    __syncthreads();
    for (int i = cnt - 1; i >= 0; i--) {
      const float4 cv = *reinterpret_cast<const float4*>(&sC[i][sg * 4]);
      const float4 gv = *reinterpret_cast<const float4*>(&sG[i][cg * 4]);
      const float2 kk = sK[i];
      const DecayCoef2 k2 = decay_pair(DecayCoef{kk.x, kk.y});
      const f2_t C2[2] = {f2_pack(cv.x, cv.y), f2_pack(cv.z, cv.w)};
      const float gys[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int ci = 0; ci < 4; ci++) {
        const f2_t gy2 = f2_pack(gys[ci], gys[ci]);
#pragma unroll
        for (int q = 0; q < 2; q++) c2[ci][q] = apply2<ACC>(k2, f2_fma(gy2, C2[q], c2[ci][q]));
      }
      sumd += sDl[i];
    }
  }
#pragma unroll
  for (int ci = 0; ci < 4; ci++) {
    const long si = ((long)b * a.S + s) * p.HP + ch0 + cg * 4 + ci;
    float v[4];
    f2_unpack(c2[ci][0], v[0], v[1]);
    f2_unpack(c2[ci][1], v[2], v[3]);
    *reinterpret_cast<float4*>(a.dhloc + si * kHlN + sg * 4) = make_float4(v[0], v[1], v[2], v[3]);
    if (sg == 0) a.sumd[si] = sumd;
  }
}

// ---- fixed-order reductions --------------------------------------------------------------
// dA, dD and d dt_bias: the sums of the per-(sequence, segment) partials.  A block = kParOut
// outputs x kParSlices slices of each output's terms; slice sl adds terms sl, sl + kParSlices,
// ... in order and the slices combine in shared memory in a fixed order, so the result is the
// same bits on every run.  (One thread per output left most SMs idle and each thread on a long
// chain of strided loads.)
constexpr int kParOut = 32, kParSlices = 8;
__global__ void __launch_bounds__(kParOut * kParSlices) reduce_params_kernel(const BwdArgs a) {
  __shared__ float sred[kParSlices][kParOut];
  const ScanProblem& p = a.p;
  const int nA = p.a_per_state ? p.H * p.N : p.H;
  const long total = (long)nA + p.HP + p.H;
  const int lo = threadIdx.x % kParOut, sl = threadIdx.x / kParOut;
  const long i = (long)blockIdx.x * kParOut + lo;
  const int bs = p.ns * a.S;  // (sequence, segment) partials
  float v = 0.0f;
  bool want = i < total;
  if (want && i < nA) {  // dA: over sequences, segments, head_dim (and states in the scalar form)
    const int h = p.a_per_state ? (int)(i / p.N) : (int)i;
    const int n_lo = p.a_per_state ? (int)(i % p.N) : 0;
    const int nn = p.a_per_state ? 1 : p.N;
    if (p.P == 1 && nn == 1) {  // one term per (sequence, segment): a plain strided sum
      const float* src = a.dA_part + i;
      const long stride = (long)kParSlices * p.HP * p.N;
      int j = sl;
      for (; j + 3 * kParSlices < bs; j += 4 * kParSlices) {  // 4 loads in flight, same order
        const float* q0 = src + (long)j * p.HP * p.N;
        const float t0 = q0[0], t1 = q0[stride], t2 = q0[2 * stride], t3 = q0[3 * stride];
        v += t0; v += t1; v += t2; v += t3;
      }
      for (; j < bs; j += kParSlices) v += src[(long)j * p.HP * p.N];
    } else {
      const int terms = bs * p.P * nn;  // term (b s, pp, n), n fastest
      for (int j = sl; j < terms; j += kParSlices) {
        const int n = n_lo + j % nn, pp = (j / nn) % p.P, q = j / (nn * p.P);
        v += a.dA_part[((long)q * p.HP + h * p.P + pp) * p.N + n];
      }
    }
  } else if (want && i < nA + p.HP) {  // dD
    const int ch = (int)(i - nA);
    want = a.g.d_D != nullptr;
    if (want)
      for (int j = sl; j < bs; j += kParSlices) v += a.dD_part[(long)j * p.HP + ch];
  } else if (want) {  // d dt_bias (head_dim == 1; the head_dim > 1 case is reduce_ddt_kernel's)
    const int h = (int)(i - nA - p.HP);
    want = a.g.d_dt_bias != nullptr && p.P == 1;
    if (want)
      for (int j = sl; j < bs; j += kParSlices) v += a.dtb_part[(long)j * p.HP + h];
  }
  sred[sl][lo] = v;
  __syncthreads();
  if (sl != 0 || !want) return;
  float t = 0.0f;
#pragma unroll
  for (int q = 0; q < kParSlices; q++) t += sred[q][lo];
  if (i < nA) a.g.d_A[i] = t;
  else if (i < nA + p.HP) a.g.d_D[i - nA] = t;
  else a.g.d_dt_bias[i - nA - p.HP] = t;
}

// head_dim > 1: d_dt[b][t][h] = softplus'(pre) * sum_p ddelta_p
template <typename IO>
__global__ void reduce_ddt_kernel(const BwdArgs a) {
  const ScanProblem& p = a.p;
  const long total = (long)p.ns * p.L * p.H;
  const IO* dt = (const IO*)p.dt;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int h = (int)(i % p.H);
    const long tok = i / p.H;
    float v = 0.0f;
    for (int pp = 0; pp < p.P; pp++) v += a.ddt_part[tok * p.HP + h * p.P + pp];
    if (p.softplus) {
      const float pre = ld(dt + i) + (p.dt_bias ? __ldg(p.dt_bias + h) : 0.0f);
      v *= softplus_gradf_(pre);
    }
    st((IO*)a.g.d_dt + i, v);
  }
}

template <typename IO>
__global__ void reduce_dtb_kernel(const BwdArgs a) {  // head_dim > 1, softplus
  const ScanProblem& p = a.p;
  const IO* dt = (const IO*)p.dt;
  for (int h = blockIdx.x * blockDim.x + threadIdx.x; h < p.H; h += gridDim.x * blockDim.x) {
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.0f;
    float v = 0.0f;
    for (long tok = 0; tok < (long)p.ns * p.L; tok++) {
      float s = 0.0f;
      for (int pp = 0; pp < p.P; pp++) s += a.ddt_part[tok * p.HP + h * p.P + pp];
      v += s * softplus_gradf_(ld(dt + tok * p.H + h) + bias);
    }
    a.g.d_dt_bias[h] = v;
  }
}

// d_s0[row] = sum over the sequences that start from row (zero if none).
__global__ void reduce_ds0_kernel(const BwdArgs a) {
  const ScanProblem& p = a.p;
  const long per_row = (long)p.HP * p.N;
  const long total = (long)p.state_rows * per_row;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int row = (int)(i / per_row);
    const long e = i - (long)row * per_row;
    float v = 0.0f;
    for (int b = 0; b < p.ns; b++) {
      const int rb = p.ids ? __ldg(p.ids + b) : b;
      if (rb == row) v += a.dh0[(long)b * per_row + e];
    }
    a.g.d_s0[i] = v;
  }
}

// ---- host side -------------------------------------------------------------------------

// Time segments of the head-tiled Mamba-2-form path: none when the (sequence, head, 32-channel
// block) grid alone has this many blocks per SM, else enough to reach it.
constexpr long kBwdHeadsBlocksPerSM = 3;

static BwdPlan plan_bwd(const ScanProblem& p, int num_sms) {
  BwdPlan q{};
  int ns;
  state_split(p.N, kBwdNS, &ns, &q.tpc);
  q.gc = (p.H / p.G) * p.P;
  const int cpb = kScanThreads / q.tpc;
  q.bpg = (q.gc + cpb - 1) / cpb;
  q.chunk_b = p.chunk <= kMaxBwdChunk ? p.chunk : kDefaultChunk;
  q.nch_b = (p.L + q.chunk_b - 1) / q.chunk_b;
  q.heads = bwd_heads_applies(p, q.chunk_b);
  long S;
  if (q.heads) {  // the head-tiled path: blocks of 32 channels x 128 states
    const long base = bwd_heads_blocks(p);
    S = base >= kBwdHeadsBlocksPerSM * num_sms
            ? 1 : (kBwdHeadsBlocksPerSM * num_sms + base - 1) / base;
  } else {
    q.tma_tt = bwd_tma_tile(p, q.chunk_b, q.gc);
    // the TMA path's blocks hold more channels (fewer, longer chains)
    const long blocks = q.tma_tt ? (long)p.ns * p.G * (q.gc / bwd_tma_channels_per_block())
                                 : (long)p.ns * p.G * q.bpg;
    const long base_threads = blocks * kScanThreads;
    const long target = (long)num_sms * kBwdTargetThreadsPerSM;
    S = base_threads >= (long)num_sms * kBwdNoSplitThreadsPerSM
            ? 1 : (target + base_threads - 1) / base_threads;
  }
  if (S > q.nch_b) S = q.nch_b;
  if (S < 1) S = 1;
  // Without time segments the (sequence, channel block) chains alone fill the GPU, but as whole
  // launches they quantise into waves (e.g. 768 chains on 456 resident blocks = 1.68 waves).
  // The TMA path then runs persistent blocks over (chain, chunk) units instead: every chunk
  // is a segment, and no local adjoint pass is needed because each unit waits for the start
  // adjoint of the chunk after it, which a unit taken earlier from the queue produces.  A
  // chain's units run one after another, so min(chains, resident blocks) blocks work at a
  // time; time segments keep every block busy but add a local adjoint pass, about 1.37x the
  // work (measured: 2 segments on 16 x 2048 x 1536 bf16).  So the persistent mode is also taken
  // when the chains fill at least 3/4 of the resident blocks, though not 512 threads per SM.
  const long chains = q.tma_tt ? (long)p.ns * p.G * (q.gc / bwd_tma_channels_per_block()) : 0;
  const long resident = (long)num_sms * kBwdTmaBlocksPerSM;
  q.persist = q.tma_tt && q.nch_b >= 2 && (S == 1 || 4 * chains >= 3 * resident);
  if (q.persist) S = q.nch_b;
  q.seg_chunks = (int)((q.nch_b + S - 1) / S);
  q.S = (q.nch_b + q.seg_chunks - 1) / q.seg_chunks;

  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  ScanProblem pf = p;
  pf.chunk = q.chunk_b;
  pf.n_chunks = q.nch_b;
  q.fwd_bytes = scan_fwd_ws_bytes(pf, num_sms);
  q.off_fwd = take(q.fwd_bytes);
  const size_t F = sizeof(float);
  q.off_ckpt = take(F * (size_t)p.ns * q.nch_b * p.HP * p.N);
  const size_t segst = F * (size_t)p.ns * q.S * p.HP * p.N;
  const size_t segch = F * (size_t)p.ns * q.S * p.HP;
  q.off_dhloc = take(segst);
  q.off_segend = take(segst);
  q.off_sumd = take(segch);
  q.off_part_bc = take(F * (size_t)p.ns * p.L * p.G * q.bpg * 2 * p.N);
  q.off_dA = take(segst);
  q.off_dD = take(segch);
  q.off_dtb = take(segch);
  q.off_ddt = take(p.P > 1 ? F * (size_t)p.ns * p.L * p.HP : 0);
  q.off_dh0 = take(F * (size_t)p.ns * p.HP * p.N);
  if (q.tma_tt && q.persist)  // queue counter, unit flags, finished-unit counts
    q.off_queue = take(sizeof(int) * (size_t)bwd_tma_queue_ints(p, q.nch_b, chains));
  if (q.heads) q.off_mh = take(F * bwd_heads_scratch_floats(p, q.S, q.chunk_b));
  q.bytes = off;
  const int nsub_max = (q.chunk_b + kTsub - 1) / kTsub;
  q.smem = sizeof(float4) * (size_t)nsub_max * kScanThreads +
           sizeof(float) * (size_t)kTsub * (kScanThreads / 32) * 2 * q.tpc * kBwdNS;
  return q;
}

size_t scan_bwd_ws_bytes(const ScanProblem& p, int num_sms) { return plan_bwd(p, num_sms).bytes; }

static int blocks_for(long total) {
  long nb = (total + 255) / 256;
  if (nb > 8192) nb = 8192;
  if (nb < 1) nb = 1;
  return (int)nb;
}

template <typename IO, bool SCALAR_A, bool FULL>
static cudaError_t launch_bwd_t(BwdArgs a, const BwdPlan& q, char* w, cudaStream_t st) {
  const ScanProblem& p = a.p;
  // the persistent TMA path needs no local adjoint pass; if its pointers do not allow TMA, the
  // general kernels take the same segments with one
  const bool tma = bwd_tma_ready(a, q);
  const bool persist = q.persist && tma;
  if (a.S > 1 && !persist) {
    cudaError_t e = q.tma_tt ? launch_bwd_tma_local(a, q, w, st) : cudaErrorNotSupported;
    if (e == cudaErrorNotSupported && q.heads && p.P % kHlCB == 0 && p.N == kHlN) {
      scan_bwd_heads_local_kernel<IO><<<dim3(p.HP / kHlCB, a.S - 1, p.ns), kHlThreads, 0, st>>>(a),
          count_launches(1);
      e = cudaSuccess;
    }
    if (e == cudaErrorNotSupported) {
      dim3 g1(p.G * a.bpg, a.S - 1, p.ns);
      scan_bwd_local_kernel<IO, SCALAR_A, FULL><<<g1, kScanThreads, 0, st>>>(a), count_launches(1);
    } else if (e != cudaSuccess) {
      return e;
    }
    scan_bwd_carry_kernel<<<blocks_for((long)p.ns * p.HP * p.N), 256, 0, st>>>(a), count_launches(1);
  }
  if (q.heads) {
    cudaError_t e = launch_bwd_heads(a, (float*)(w + q.off_mh), st);
    if (e != cudaSuccess) return e;
    if (a.g.d_s0 && a.dh0 != a.g.d_s0)
      reduce_ds0_kernel<<<blocks_for((long)p.state_rows * p.HP * p.N), 256, 0, st>>>(a), count_launches(1);
    return cudaGetLastError();
  }
  cudaError_t e = cudaErrorNotSupported;
  if (tma) {
    BwdArgs at = a;
    at.bpg = a.gc / bwd_tma_channels_per_block();  // its dB/dC partials are per block
    e = launch_bwd_tma_main(at, q, w, st);
    if (e == cudaSuccess) a.bpg = at.bpg;
  }
  if (e == cudaErrorNotSupported) {
    auto kern = scan_bwd_kernel<IO, SCALAR_A, FULL>;
    if (q.smem > 48 * 1024) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)q.smem);
      if (e != cudaSuccess) return e;
    }
    dim3 g2(p.G * a.bpg, a.S, p.ns);
    kern<<<g2, kScanThreads, q.smem, st>>>(a), count_launches(1);
  } else if (e != cudaSuccess) {
    return e;
  }
  if (!(persist && e == cudaSuccess))  // (the persistent TMA kernel sums dB, dC in its queue)
    reduce_bc_kernel<IO><<<blocks_for((long)p.ns * p.L * p.G * 2 * p.N), 256, 0, st>>>(a), count_launches(1);
  const long nparams = (long)(p.a_per_state ? p.H * p.N : p.H) + p.HP + p.H;
  reduce_params_kernel<<<(int)((nparams + kParOut - 1) / kParOut), kParOut * kParSlices, 0, st>>>(a),
      count_launches(1);
  if (p.P > 1) {
    reduce_ddt_kernel<IO><<<blocks_for((long)p.ns * p.L * p.H), 256, 0, st>>>(a), count_launches(1);
    if (p.softplus && a.g.d_dt_bias) reduce_dtb_kernel<IO><<<blocks_for(p.H), 256, 0, st>>>(a), count_launches(1);
  }
  if (a.g.d_s0 && a.dh0 != a.g.d_s0)
    reduce_ds0_kernel<<<blocks_for((long)p.state_rows * p.HP * p.N), 256, 0, st>>>(a), count_launches(1);
  return cudaGetLastError();
}

template <typename IO>
static cudaError_t launch_bwd_io(const BwdArgs& a, const BwdPlan& q, bool full, char* w,
                                 cudaStream_t st) {
  if (!a.p.a_per_state)
    return full ? launch_bwd_t<IO, true, true>(a, q, w, st) : launch_bwd_t<IO, true, false>(a, q, w, st);
  return full ? launch_bwd_t<IO, false, true>(a, q, w, st) : launch_bwd_t<IO, false, false>(a, q, w, st);
}

cudaError_t launch_scan_bwd(const ScanProblem& p, const float* ckpt, const ScanGrads& g, void* ws,
                            int num_sms, cudaStream_t st) {
  const BwdPlan q = plan_bwd(p, num_sms);
  char* w = (char*)ws;
  BwdArgs a{};
  a.p = p;
  a.g = g;
  a.chunk_b = q.chunk_b;
  a.nch_b = q.nch_b;
  a.S = q.S;
  a.seg_chunks = q.seg_chunks;
  a.tpc = q.tpc;
  a.bpg = q.bpg;
  a.gc = q.gc;
  a.ckpt = ckpt;
  if (!ckpt || p.chunk != q.chunk_b) {  // (re)compute checkpoints at interval chunk_b
    ScanProblem pf = p;
    pf.chunk = q.chunk_b;
    pf.n_chunks = q.nch_b;
    float* ck = (float*)(w + q.off_ckpt);
    cudaError_t e = launch_scan_fwd(pf, nullptr, nullptr, ck, w + q.off_fwd, num_sms, st);
    if (e != cudaSuccess) return e;
    a.ckpt = ck;
  }
  a.dhloc = (float*)(w + q.off_dhloc);
  a.segend = (float*)(w + q.off_segend);
  a.sumd = (float*)(w + q.off_sumd);
  a.part_bc = (float*)(w + q.off_part_bc);
  a.dA_part = (float*)(w + q.off_dA);
  a.dD_part = (float*)(w + q.off_dD);
  a.dtb_part = (float*)(w + q.off_dtb);
  a.ddt_part = (float*)(w + q.off_ddt);
  // the start-state adjoints, one row per sequence; when sequence b's initial state is row b
  // (no ids, one row per sequence) they are d_s0 itself and no sum runs.  Every path writes
  // each element once, from the unit or segment that ends at the sequence start.
  a.dh0 = (!p.ids && p.state_rows == p.ns && g.d_s0) ? g.d_s0 : (float*)(w + q.off_dh0);
  const bool full = rows_vectorizable(p, kBwdNS, q.tpc);
  return p.io == SSM_BF16 ? launch_bwd_io<__nv_bfloat16>(a, q, full, w, st)
                          : launch_bwd_io<float>(a, q, full, w, st);
}

}  // namespace ssm

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
#include "tma.cuh"

namespace ssm {

constexpr int kBwdNS = 4;          // states per thread
constexpr int kTsub = 8;           // tokens of state history held in registers
constexpr int kMaxBwdChunk = 512;  // larger checkpoint intervals are re-checkpointed at 256
constexpr int kDefaultChunk = 256;

struct BwdArgs {
  ScanProblem p;
  ScanGrads g;
  const float* ckpt;  // checkpoints at interval chunk_b
  int chunk_b, nch_b;
  int S, seg_chunks;  // segments of whole chunks
  int tpc, bpg, gc;   // threads per channel, blocks per group, channels per group
  float* dhloc;       // [ns][S][HP][N]
  float* segend;      // [ns][S][HP][N]
  float* sumd;        // [ns][S][HP]
  float* part_bc;     // [ns*L][G][bpg][2][N]
  float* dA_part;     // [ns][S][HP][N]
  float* dD_part;     // [ns][S][HP]
  float* dtb_part;    // [ns][S][HP]
  float* ddt_part;    // [ns*L][HP]   (head_dim > 1 only)
  float* dh0;         // [ns][HP][N]
};

struct Lane {
  int tpc, cl, sg, g, blk, cig, ch, h, n0;
  bool valid;
};

__device__ __forceinline__ Lane lane_of(const BwdArgs& a) {
  Lane l;
  l.tpc = a.tpc;
  l.cl = threadIdx.x / l.tpc;
  l.sg = threadIdx.x - l.cl * l.tpc;
  l.g = blockIdx.x / a.bpg;
  l.blk = blockIdx.x - l.g * a.bpg;
  l.cig = l.blk * (kScanThreads / l.tpc) + l.cl;
  l.valid = l.cig < a.gc;
  l.ch = l.g * a.gc + (l.valid ? l.cig : 0);
  l.h = l.ch / a.p.P;
  l.n0 = l.sg * kBwdNS;
  return l;
}

template <typename IO>
__device__ __forceinline__ float delta_of(const ScanProblem& p, const IO* dt, long tok, int h,
                                          float bias, float* pre) {
  const float raw = ld(dt + tok * p.H + h);
  if (p.softplus) {
    *pre = raw + bias;
    return softplusf_(*pre);
  }
  *pre = raw;
  return raw;
}

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
        const float as = SCALAR_A ? decay_coef<ACC>(dl, A2[0]) : 0.0f;
#pragma unroll
        for (int j = 0; j < kBwdNS; j++)
          hs[j] = decay_step<ACC>(SCALAR_A ? as : decay_coef<ACC>(dl, A2[j]), hs[j], dx * Bv[j]);
      }
    }
    // ---- level 2: per sub-chunk, last to first --------------------------------------------
    for (int k = nsub - 1; k >= 0; k--) {
      const int ts = t0 + k * kTsub;
      const int cnt = min(kTsub, t1 - ts);
      float hh[kTsub + 1][kBwdNS], aa[kTsub][kBwdNS], dls[kTsub], xs[kTsub], pres[kTsub];
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
          const float as = SCALAR_A ? decay_coef<ACC>(dl, A2[0]) : 0.0f;
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) {
            aa[i][j] = SCALAR_A ? as : decay_coef<ACC>(dl, A2[j]);
            hh[i + 1][j] = decay_step<ACC>(aa[i][j], hh[i][j], dx * Bv[j]);
          }
          dls[i] = dl; xs[i] = xv; pres[i] = pre;
        } else {
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) { aa[i][j] = ACC ? 0.0f : 1.0f; hh[i + 1][j] = hh[i][j]; }
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
            if (z && a.g.d_z) st((IO*)a.g.d_z + tok * p.HP + l.ch, dyv * ypre * silu_gradf_(zv));
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
    const float as = SCALAR_A ? decay_coef<ACC>(dl, A2[0]) : 0.0f;
#pragma unroll
    for (int j = 0; j < kBwdNS; j++)
      c[j] = decay_apply<ACC>(SCALAR_A ? as : decay_coef<ACC>(dl, A2[j]), fmaf(gy, Cv[j], c[j]));
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
    for (int s = a.S - 1; s >= 0; s--) {
      const long si = ((long)b * a.S + s) * p.HP + ch;
      a.segend[si * p.N + n] = c;
      if (s > 0) c = fmaf(ex2(A2 * a.sumd[si]), c, a.dhloc[si * p.N + n]);
    }
  }
}

// ---- fixed-order reductions --------------------------------------------------------------
template <typename IO>
__global__ void reduce_bc_kernel(const BwdArgs a) {
  const ScanProblem& p = a.p;
  const long total = (long)p.ns * p.L * p.G * 2 * p.N;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int r = (int)(i % (2 * p.N));
    const long tg = i / (2 * p.N);  // tok * G + g
    const float* src = a.part_bc + tg * a.bpg * 2 * p.N + r;
    float v = 0.0f;
    for (int k = 0; k < a.bpg; k++) v += src[(long)k * 2 * p.N];
    const int q = r / p.N, n = r - q * p.N;
    st((IO*)(q == 0 ? a.g.d_B : a.g.d_C) + tg * p.N + n, v);
  }
}

__global__ void reduce_params_kernel(const BwdArgs a) {
  const ScanProblem& p = a.p;
  const int nA = p.a_per_state ? p.H * p.N : p.H;
  const long total = (long)nA + p.HP + p.H;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    if (i < nA) {  // dA: over sequences, segments, head_dim (and states in the scalar form)
      const int h = p.a_per_state ? (int)(i / p.N) : (int)i;
      const int n_lo = p.a_per_state ? (int)(i % p.N) : 0;
      const int n_hi = p.a_per_state ? n_lo + 1 : p.N;
      float v = 0.0f;
      for (int b = 0; b < p.ns; b++)
        for (int s = 0; s < a.S; s++)
          for (int pp = 0; pp < p.P; pp++)
            for (int n = n_lo; n < n_hi; n++)
              v += a.dA_part[(((long)b * a.S + s) * p.HP + h * p.P + pp) * p.N + n];
      a.g.d_A[i] = v;
    } else if (i < nA + p.HP) {  // dD
      const int ch = (int)(i - nA);
      if (!a.g.d_D) continue;
      float v = 0.0f;
      for (int b = 0; b < p.ns; b++)
        for (int s = 0; s < a.S; s++) v += a.dD_part[((long)b * a.S + s) * p.HP + ch];
      a.g.d_D[ch] = v;
    } else {  // d dt_bias (head_dim == 1; the head_dim > 1 case is reduce_ddt_kernel's)
      const int h = (int)(i - nA - p.HP);
      if (!a.g.d_dt_bias || p.P != 1) continue;
      float v = 0.0f;
      for (int b = 0; b < p.ns; b++)
        for (int s = 0; s < a.S; s++) v += a.dtb_part[((long)b * a.S + s) * p.HP + h];
      a.g.d_dt_bias[h] = v;
    }
  }
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

// ---- TMA-staged main kernel: Mamba-1 layout, d_state 16 ----------------------------------
// Same arithmetic and workspace outputs as scan_bwd_kernel, with its inputs streamed as
// [tile][32 channels] tiles (x, dt, z, dy) and [tile][16] tiles (B, C) through a ring of
// shared-memory stages filled by cp.async.bulk.tensor, and dx, dz, ddt leaving as TMA-stored
// tiles.  Per chunk the schedule is: level-1 tiles forward (x, dt, B), then level-2 tiles in
// reverse (all inputs).  Sub-chunk start states go to a per-block region of global scratch
// (they are re-read by the same thread shortly after, from L2).  The dB/dC sums over the 8
// channels of a warp use a transposed butterfly: each of the 3 levels halves the values a
// lane holds, so the 8 partials (4 dB, 4 dC) of 8 lanes become 1 finished sum per lane in
// 7 shuffles instead of 24.
constexpr int kBwdStages = 3;

struct BwdTma {
  CUtensorMap mx, mdt, mz, mdy, mb, mc, mdx, mdz, mddt;
  int tt;  // tile tokens: divides chunk_b, multiple of kTsub
  uint32_t bytes_l1, bytes_l2;
  uint32_t off_x, off_dt, off_z, off_dy, off_b, off_c, stage_stride;
  uint32_t off_out, out_tile, out_stride, off_red, off_bar;
  float4* bnd;  // global scratch: [blocks][chunk_b / kTsub][threads]
};

// v holds 8 partials; lanes that differ in bits 2..4 hold other channels.  Returns the sum over
// those 8 lanes of the partial with original index (lane >> 2) & 7.
__device__ __forceinline__ float reduce8_transposed(float (&v)[8], int lane) {
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float send = up ? v[i] : v[i + 4], keep = up ? v[i + 4] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 2; i++) {
      const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  const bool up = lane & 4;
  const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
  return keep + __shfl_xor_sync(0xffffffffu, send, 4);
}

template <typename IO>
__device__ __forceinline__ float lds_f(const IO* p) {
  if constexpr (sizeof(IO) == 4) return *reinterpret_cast<const float*>(p);
  else return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}
template <typename IO>
__device__ __forceinline__ void sts_f(IO* p, float v) {
  if constexpr (sizeof(IO) == 4) *reinterpret_cast<float*>(p) = v;
  else *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}
template <typename IO>
__device__ __forceinline__ void lds4(const IO* p, float (&o)[4]) {
  if constexpr (sizeof(IO) == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162* q = reinterpret_cast<const __nv_bfloat162*>(&v);
    const float2 a0 = __bfloat1622float2(q[0]), a1 = __bfloat1622float2(q[1]);
    o[0] = a0.x; o[1] = a0.y; o[2] = a1.x; o[3] = a1.y;
  }
}

template <typename IO>
__global__ void __launch_bounds__(kScanThreads)
scan_bwd_tma_kernel(const __grid_constant__ BwdTma m, const BwdArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;
  constexpr int kWarps = kScanThreads / 32;
  constexpr int CB = kScanThreads / 4;  // 32 channels, 4 threads x 4 states each
  extern __shared__ __align__(128) unsigned char smem[];
  const ScanProblem& p = a.p;
  const Lane l = lane_of(a);
  const int N = p.N;  // 16
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cl = l.cl, ch = l.ch, ch0 = ch - cl;
  const int s = blockIdx.y, b = blockIdx.z;
  const int tt = m.tt;
  const int sub_per_tile = tt / kTsub;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + m.off_bar);
  float* red = reinterpret_cast<float*>(smem + m.off_red);  // [tt][warps][2N]
  const int nsub_max = a.chunk_b / kTsub;
  float4* bnd = m.bnd + ((long)(b * a.S + s) * gridDim.x + blockIdx.x) * nsub_max * kScanThreads;
  const int c_first = s * a.seg_chunks;
  const int c_last = min(a.nch_b, c_first + a.seg_chunks) - 1;

  // The tile schedule: per chunk (last to first), level-1 tiles ascending then level-2 tiles
  // descending.  Producer and consumers walk it with their own cursors.
  struct Pos { int ck, lvl, j, nt; };
  auto ntiles = [&](int ck) {
    const int t0 = ck * a.chunk_b, t1 = min(p.L, t0 + a.chunk_b);
    return (t1 - t0 + tt - 1) / tt;
  };
  auto first = [&]() { Pos q; q.ck = c_last; q.lvl = 0; q.j = 0; q.nt = ntiles(c_last); return q; };
  auto advance = [&](Pos& q) {
    if (q.lvl == 0) {
      if (++q.j == q.nt) { q.lvl = 1; q.j = q.nt - 1; }
    } else if (--q.j < 0) {
      q.ck--; q.lvl = 0; q.j = 0;
      if (q.ck >= c_first) q.nt = ntiles(q.ck);
    }
  };

  if (tid == 0) {
    for (int i = 0; i < kBwdStages; i++) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  Pos pp = first();
  int issued = 0;
  auto issue = [&]() {  // thread 0 only
    const int stg = issued % kBwdStages;
    unsigned char* base = smem + stg * m.stage_stride;
    const int t0 = pp.ck * a.chunk_b + pp.j * tt;
    if (pp.lvl == 0) {
      mbar_expect_tx(&full[stg], m.bytes_l1);
      tma_load_3d(base + m.off_x, &m.mx, ch0, t0, b, &full[stg]);
      tma_load_3d(base + m.off_dt, &m.mdt, ch0, t0, b, &full[stg]);
      tma_load_3d(base + m.off_b, &m.mb, l.g * N, t0, b, &full[stg]);
    } else {
      mbar_expect_tx(&full[stg], m.bytes_l2);
      tma_load_3d(base + m.off_x, &m.mx, ch0, t0, b, &full[stg]);
      tma_load_3d(base + m.off_dt, &m.mdt, ch0, t0, b, &full[stg]);
      tma_load_3d(base + m.off_dy, &m.mdy, ch0, t0, b, &full[stg]);
      if (p.z) tma_load_3d(base + m.off_z, &m.mz, ch0, t0, b, &full[stg]);
      tma_load_3d(base + m.off_b, &m.mb, l.g * N, t0, b, &full[stg]);
      tma_load_3d(base + m.off_c, &m.mc, l.g * N, t0, b, &full[stg]);
    }
    issued++;
    advance(pp);
  };
  if (tid == 0)
    for (int k = 0; k < kBwdStages && pp.ck >= c_first; k++) issue();

  float An[kBwdNS], A2[kBwdNS], carry[kBwdNS];
  {
    const long si = ((long)b * a.S + s) * p.HP + ch;
#pragma unroll
    for (int j = 0; j < kBwdNS; j++) {
      An[j] = __ldg(p.A + (long)ch * N + l.n0 + j);
      A2[j] = An[j] * kLog2e;
      if (a.S > 1) carry[j] = a.segend[si * N + l.n0 + j];
      else carry[j] = a.g.d_state_out ? __ldg(a.g.d_state_out + ((long)b * p.HP + ch) * N + l.n0 + j) : 0.0f;
    }
  }
  float dA_acc[kBwdNS] = {0.f, 0.f, 0.f, 0.f};
  float dD_acc = 0.0f, dtb_acc = 0.0f;
  const float Dv = p.D ? __ldg(p.D + ch) : 0.0f;
  const float bias = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + ch) : 0.0f;
  float hs[kBwdNS] = {0.f, 0.f, 0.f, 0.f};
  int n_l2 = 0;

  int q = 0;
  for (Pos cs = first(); cs.ck >= c_first; advance(cs), q++) {
    const int stg = q % kBwdStages;
    if (cs.lvl == 1 && tid == 0) tma_store_wait_read<1>();  // out buffer (n_l2 & 1) is free
    const bool ok = mbar_wait(&full[stg], (uint32_t)(q / kBwdStages) & 1u);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        record_status(p.status, SSM_ERR_TIMEOUT);
        for (int j = q; j < issued; j++) mbar_wait(&full[j % kBwdStages], (uint32_t)(j / kBwdStages) & 1u);
        tma_store_wait_all();
      }
      return;
    }
    const unsigned char* base = smem + stg * m.stage_stride;
    const IO* sx = reinterpret_cast<const IO*>(base + m.off_x);
    const IO* sdt = reinterpret_cast<const IO*>(base + m.off_dt);
    const IO* sz = reinterpret_cast<const IO*>(base + m.off_z);
    const IO* sdy = reinterpret_cast<const IO*>(base + m.off_dy);
    const IO* sB = reinterpret_cast<const IO*>(base + m.off_b);
    const IO* sC = reinterpret_cast<const IO*>(base + m.off_c);
    const int t0c = cs.ck * a.chunk_b, t1c = min(p.L, t0c + a.chunk_b);
    const int t0 = t0c + cs.j * tt;
    const int cnt = min(tt, t1c - t0);
    const int nsub = (cnt + kTsub - 1) / kTsub;

    if (cs.lvl == 0) {
      // ---- level 1: walk the tile forward, keeping every sub-chunk's start state ----------
      if (cs.j == 0) {
        const float* src = a.ckpt + (((long)b * a.nch_b + cs.ck) * p.HP + ch) * N + l.n0;
#pragma unroll
        for (int j = 0; j < kBwdNS; j++) hs[j] = src[j];
      }
      for (int k = 0; k < nsub; k++) {
        bnd[(cs.j * sub_per_tile + k) * kScanThreads + tid] = make_float4(hs[0], hs[1], hs[2], hs[3]);
        const int i1 = min(cnt, (k + 1) * kTsub);
        for (int i = k * kTsub; i < i1; i++) {
          float dl = lds_f(sdt + i * CB + cl);
          if (p.softplus) dl = softplusf_(dl + bias);
          const float dx = dl * lds_f(sx + i * CB + cl);
          float Bv[kBwdNS];
          lds4(sB + i * N + l.n0, Bv);
#pragma unroll
          for (int j = 0; j < kBwdNS; j++)
            hs[j] = decay_step<ACC>(decay_coef<ACC>(dl, A2[j]), hs[j], dx * Bv[j]);
        }
      }
      __syncthreads();  // stage fully read
      if (tid == 0 && pp.ck >= c_first) issue();
      continue;
    }

    // ---- level 2: sub-chunks last to first: recompute 8 tokens, then the adjoint over them --
    IO* out = reinterpret_cast<IO*>(smem + m.off_out + (n_l2 & 1) * m.out_stride);
    IO* odx = out;
    IO* odz = reinterpret_cast<IO*>(reinterpret_cast<unsigned char*>(out) + m.out_tile);
    IO* oddt = reinterpret_cast<IO*>(reinterpret_cast<unsigned char*>(out) + 2 * m.out_tile);
    for (int k = nsub - 1; k >= 0; k--) {
      const int i0 = k * kTsub;
      const int c8 = min(kTsub, cnt - i0);
      float hh[kTsub + 1][kBwdNS], aa[kTsub][kBwdNS], dls[kTsub], xs[kTsub], pres[kTsub];
      {
        const float4 v = bnd[(cs.j * sub_per_tile + k) * kScanThreads + tid];
        hh[0][0] = v.x; hh[0][1] = v.y; hh[0][2] = v.z; hh[0][3] = v.w;
      }
#pragma unroll
      for (int r = 0; r < kTsub; r++) {
        if (r < c8) {
          const int i = i0 + r;
          const float raw = lds_f(sdt + i * CB + cl);
          const float pre = raw + bias;
          const float dl = p.softplus ? softplusf_(pre) : raw;
          const float xv = lds_f(sx + i * CB + cl);
          float Bv[kBwdNS];
          lds4(sB + i * N + l.n0, Bv);
          const float dx = dl * xv;
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) {
            aa[r][j] = decay_coef<ACC>(dl, A2[j]);
            hh[r + 1][j] = decay_step<ACC>(aa[r][j], hh[r][j], dx * Bv[j]);
          }
          dls[r] = dl; xs[r] = xv; pres[r] = pre;
        } else {
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) { aa[r][j] = ACC ? 0.0f : 1.0f; hh[r + 1][j] = hh[r][j]; }
          dls[r] = 0.0f; xs[r] = 0.0f; pres[r] = 0.0f;
        }
      }
#pragma unroll
      for (int r = kTsub - 1; r >= 0; r--) {
        if (r < c8) {  // uniform over the block
          const int i = i0 + r;
          float Bv[kBwdNS], Cv[kBwdNS];
          lds4(sB + i * N + l.n0, Bv);
          lds4(sC + i * N + l.n0, Cv);
          const float dyv = lds_f(sdy + i * CB + cl);
          float gy = dyv, ypre = 0.0f, zv = 0.0f;
          if (p.z) {
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < kBwdNS; j++) part = fmaf(Cv[j], hh[r + 1][j], part);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            ypre = fmaf(Dv, xs[r], part);
            zv = lds_f(sz + i * CB + cl);
            gy = dyv * siluf_(zv);
          }
          const float dlx = dls[r] * xs[r];
          float sB = 0.0f, sAw = 0.0f, v8[8];
#pragma unroll
          for (int j = 0; j < kBwdNS; j++) {
            const float dh = fmaf(gy, Cv[j], carry[j]);
            v8[4 + j] = gy * hh[r + 1][j];          // dC partial
            sB = fmaf(dh, Bv[j], sB);
            v8[j] = dh * dlx;                       // dB partial
            const float cn = decay_apply<ACC>(aa[r][j], dh);
            const float w = cn * hh[r][j];
            sAw = fmaf(An[j], w, sAw);
            dA_acc[j] = fmaf(dls[r], w, dA_acc[j]);
            carry[j] = cn;
          }
          sB += __shfl_xor_sync(0xffffffffu, sB, 1);
          sAw += __shfl_xor_sync(0xffffffffu, sAw, 1);
          sB += __shfl_xor_sync(0xffffffffu, sB, 2);
          sAw += __shfl_xor_sync(0xffffffffu, sAw, 2);
          const float dxv = fmaf(gy, Dv, dls[r] * sB);
          const float ddl = fmaf(xs[r], sB, sAw);
          const float ddt = p.softplus ? ddl * softplus_gradf_(pres[r]) : ddl;
          dD_acc = fmaf(gy, xs[r], dD_acc);
          if (l.sg == 0) {
            sts_f(odx + i * CB + cl, dxv);
            if (p.z) sts_f(odz + i * CB + cl, dyv * ypre * silu_gradf_(zv));
            sts_f(oddt + i * CB + cl, ddt);
            dtb_acc += ddt;
          }
          const float tot = reduce8_transposed(v8, lane);
          const int o = (lane >> 2) & 7;  // 0..3: dB of state n0+o, 4..7: dC of state n0+o-4
          red[(i * kWarps + warp) * 2 * N + (o >> 2) * N + l.n0 + (o & 3)] = tot;
        }
      }
    }
    fence_async_shared();
    __syncthreads();  // stage read, out tiles and red complete
    for (int idx = tid; idx < cnt * 2 * N; idx += kScanThreads) {
      const int i = idx / (2 * N), r = idx - i * 2 * N;
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; w++) v += red[(i * kWarps + w) * 2 * N + r];
      const long tok = (long)b * p.L + t0 + i;
      a.part_bc[((tok * p.G + l.g) * a.bpg + l.blk) * 2 * N + r] = v;
    }
    if (tid == 0) {
      tma_store_3d(&m.mdx, odx, ch0, t0, b);
      if (p.z && a.g.d_z) tma_store_3d(&m.mdz, odz, ch0, t0, b);
      tma_store_3d(&m.mddt, oddt, ch0, t0, b);
      tma_store_commit();
      if (pp.ck >= c_first) issue();
    }
    n_l2++;
  }
  if (tid == 0) tma_store_wait_all();

  const long si = ((long)b * a.S + s) * p.HP + ch;
#pragma unroll
  for (int j = 0; j < kBwdNS; j++) {
    a.dA_part[si * N + l.n0 + j] = dA_acc[j];
    if (s == 0) a.dh0[((long)b * p.HP + ch) * N + l.n0 + j] = carry[j];
  }
  if (l.sg == 0) {
    a.dD_part[si] = dD_acc;
    a.dtb_part[si] = dtb_acc;
  }
}

// ---- host side -------------------------------------------------------------------------
struct BwdPlan {
  int tpc, gc, bpg, chunk_b, nch_b, S, seg_chunks;
  int tma_tt;  // tile tokens of the TMA-staged path; 0 when the shape does not allow it
  size_t off_fwd, fwd_bytes, off_ckpt, off_dhloc, off_segend, off_sumd, off_part_bc, off_dA,
      off_dD, off_dtb, off_ddt, off_dh0, off_bnd, bytes, smem;
};

static BwdPlan plan_bwd(const ScanProblem& p, int num_sms) {
  BwdPlan q{};
  int ns;
  state_split(p.N, kBwdNS, &ns, &q.tpc);
  q.gc = (p.H / p.G) * p.P;
  const int cpb = kScanThreads / q.tpc;
  q.bpg = (q.gc + cpb - 1) / cpb;
  q.chunk_b = p.chunk <= kMaxBwdChunk ? p.chunk : kDefaultChunk;
  q.nch_b = (p.L + q.chunk_b - 1) / q.chunk_b;
  const long base_threads = (long)p.ns * p.G * q.bpg * kScanThreads;
  const long target = (long)num_sms * kBwdTargetThreadsPerSM;
  long S = (target + base_threads - 1) / base_threads;
  if (S > q.nch_b) S = q.nch_b;
  if (S < 1) S = 1;
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
  const int io = p.io == SSM_BF16 ? 2 : 4;
  if (p.P == 1 && p.a_per_state && p.N == 16 && q.tpc == 4 && (p.HP * io) % 16 == 0 &&
      q.gc % (kScanThreads / 4) == 0 && q.chunk_b % kTsub == 0)
    q.tma_tt = q.chunk_b % 32 == 0 ? 32 : (q.chunk_b % 16 == 0 ? 16 : 8);
  if (q.tma_tt) {
    const size_t blocks = (size_t)p.G * q.bpg * q.S * p.ns;
    q.off_bnd = take(sizeof(float4) * blocks * (q.chunk_b / kTsub) * kScanThreads);
  }
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
static cudaError_t launch_bwd_t(const BwdArgs& a, size_t smem, const BwdTma* m, size_t tma_smem,
                                cudaStream_t st) {
  const ScanProblem& p = a.p;
  if (a.S > 1) {
    dim3 g1(p.G * a.bpg, a.S - 1, p.ns);
    scan_bwd_local_kernel<IO, SCALAR_A, FULL><<<g1, kScanThreads, 0, st>>>(a), count_launches(1);
    scan_bwd_carry_kernel<<<blocks_for((long)p.ns * p.HP * p.N), 256, 0, st>>>(a), count_launches(1);
  }
  dim3 g2(p.G * a.bpg, a.S, p.ns);
  if (m) {
    auto kt = scan_bwd_tma_kernel<IO>;
    cudaError_t e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tma_smem);
    if (e != cudaSuccess) return e;
    kt<<<g2, kScanThreads, tma_smem, st>>>(*m, a), count_launches(1);
  } else {
    auto kern = scan_bwd_kernel<IO, SCALAR_A, FULL>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
    }
    kern<<<g2, kScanThreads, smem, st>>>(a), count_launches(1);
  }
  reduce_bc_kernel<IO><<<blocks_for((long)p.ns * p.L * p.G * 2 * p.N), 256, 0, st>>>(a), count_launches(1);
  const long nparams = (long)(p.a_per_state ? p.H * p.N : p.H) + p.HP + p.H;
  reduce_params_kernel<<<blocks_for(nparams), 256, 0, st>>>(a), count_launches(1);
  if (p.P > 1) {
    reduce_ddt_kernel<IO><<<blocks_for((long)p.ns * p.L * p.H), 256, 0, st>>>(a), count_launches(1);
    if (p.softplus && a.g.d_dt_bias) reduce_dtb_kernel<IO><<<blocks_for(p.H), 256, 0, st>>>(a), count_launches(1);
  }
  if (a.g.d_s0)
    reduce_ds0_kernel<<<blocks_for((long)p.state_rows * p.HP * p.N), 256, 0, st>>>(a), count_launches(1);
  return cudaGetLastError();
}

template <typename IO>
static cudaError_t launch_bwd_io(const BwdArgs& a, size_t smem, bool full, const BwdTma* m,
                                 size_t tma_smem, cudaStream_t st) {
  if (!a.p.a_per_state)
    return full ? launch_bwd_t<IO, true, true>(a, smem, nullptr, 0, st)
                : launch_bwd_t<IO, true, false>(a, smem, nullptr, 0, st);
  return full ? launch_bwd_t<IO, false, true>(a, smem, m, tma_smem, st)
              : launch_bwd_t<IO, false, false>(a, smem, nullptr, 0, st);
}

static bool al16(const void* v) { return ((uintptr_t)v & 15) == 0; }

// Tensor maps and shared-memory layout of the TMA-staged backward; false if not applicable.
static bool setup_bwd_tma(const ScanProblem& p, const ScanGrads& g, const BwdPlan& q, char* w,
                          BwdTma* m, size_t* smem) {
  if (!q.tma_tt) return false;
  if (!al16(p.x) || !al16(p.dt) || !al16(p.B) || !al16(p.C) || !al16(g.dy) || !al16(g.d_x) ||
      !al16(g.d_dt) || (p.z && !al16(p.z)) || (g.d_z && !al16(g.d_z)))
    return false;
  const int io = p.io == SSM_BF16 ? 2 : 4;
  const int tt = q.tma_tt, cb = kScanThreads / 4;
  const uint64_t C = p.HP, L = p.L, NSq = p.ns, GN = (uint64_t)p.G * p.N;
  memset(m, 0, sizeof(*m));
  bool ok = encode_tmap_3d(&m->mx, p.x, io, C, L, NSq, C, C * L, cb, tt, 1) &&
            encode_tmap_3d(&m->mdt, p.dt, io, C, L, NSq, C, C * L, cb, tt, 1) &&
            encode_tmap_3d(&m->mdy, g.dy, io, C, L, NSq, C, C * L, cb, tt, 1) &&
            encode_tmap_3d(&m->mb, p.B, io, GN, L, NSq, GN, GN * L, p.N, tt, 1) &&
            encode_tmap_3d(&m->mc, p.C, io, GN, L, NSq, GN, GN * L, p.N, tt, 1) &&
            encode_tmap_3d(&m->mdx, g.d_x, io, C, L, NSq, C, C * L, cb, tt, 1) &&
            encode_tmap_3d(&m->mddt, g.d_dt, io, C, L, NSq, C, C * L, cb, tt, 1);
  if (ok && p.z) ok = encode_tmap_3d(&m->mz, p.z, io, C, L, NSq, C, C * L, cb, tt, 1);
  if (ok && g.d_z) ok = encode_tmap_3d(&m->mdz, g.d_z, io, C, L, NSq, C, C * L, cb, tt, 1);
  if (!ok) return false;
  auto al = [](uint32_t v) { return (v + 127u) & ~127u; };
  const uint32_t tile = (uint32_t)(tt * cb * io), row = (uint32_t)(tt * p.N * io);
  m->tt = tt;
  m->off_x = 0;
  m->off_dt = al(tile);
  m->off_z = m->off_dt + al(tile);
  m->off_dy = m->off_z + al(tile);
  m->off_b = m->off_dy + al(tile);
  m->off_c = m->off_b + al(row);
  m->stage_stride = m->off_c + al(row);
  m->off_out = kBwdStages * m->stage_stride;
  m->out_tile = al(tile);
  m->out_stride = 3 * m->out_tile;
  m->off_red = m->off_out + 2 * m->out_stride;
  m->off_bar = m->off_red + al((uint32_t)(sizeof(float) * tt * (kScanThreads / 32) * 2 * p.N));
  m->bytes_l1 = 2 * tile + row;
  m->bytes_l2 = (3 + (p.z ? 1 : 0)) * tile + 2 * row;
  m->bnd = reinterpret_cast<float4*>(w + q.off_bnd);
  *smem = m->off_bar + 64;
  return true;
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
  a.dh0 = (float*)(w + q.off_dh0);
  const bool full = rows_vectorizable(p, kBwdNS, q.tpc);
  BwdTma m;
  size_t tma_smem = 0;
  const bool tma = setup_bwd_tma(p, g, q, w, &m, &tma_smem);
  return p.io == SSM_BF16
             ? launch_bwd_io<__nv_bfloat16>(a, q.smem, full, tma ? &m : nullptr, tma_smem, st)
             : launch_bwd_io<float>(a, q.smem, full, tma ? &m : nullptr, tma_smem, st);
}

}  // namespace ssm

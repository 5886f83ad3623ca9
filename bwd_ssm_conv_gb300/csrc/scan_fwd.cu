// scan_fwd.cu -- selective scan forward with per-chunk state checkpoints.
//
// Recurrence (infotheory mamba1/model.rs, selective_scan_state16 / forward_impl):
//   a = exp(delta A),  h_t = a h_{t-1} + (delta x_t) B_t,  y_t = (C_t . h_t + D x_t) silu(z_t)
//
// Parallel layout.  A thread owns one channel (b, h, p) and NS consecutive states; TPC =
// N_pad / NS threads share a channel and sum their parts of C . h with xor-shuffles.  Time
// is split into S segments processed by independent blocks.  Because h_end = P h_start +
// h_local with P = exp(A sum(delta)) (the affine composition that associative_scan_backward
// of kizzasi-model backprop_ssm.rs scans), the true start state of every segment is found
// in three launches that never wait on each other:
//   1. local:  each segment but the last runs from a zero state -> (h_local, sum delta);
//   2. carry:  one thread per (b, channel, n) composes the segments in order;
//   3. main:   each segment runs from its true start, writing y, the checkpoints every
//              `chunk` tokens (state at the START of the chunk) and the final state.
// With S = 1 only the main launch runs.
#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"

namespace ssm {

struct FwdArgs {
  ScanProblem p;
  int S, seg_len, tpc;
  void* y;
  float* state_out;
  float* ckpt;
  float* segstart;  // [ns][S][HP][N]
  float* hloc;      // [ns][S][HP][N]
  float* sumdelta;  // [ns][S][HP]
};

// FULL: N == tpc * NS (no padded states) and B/C rows are 16-byte aligned (vector loads).
template <typename IO, int NS, bool SCALAR_A, bool LOCAL, bool FULL>
__global__ void __launch_bounds__(kScanThreads)
scan_fwd_kernel(const FwdArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;  // accurate decay form for fp32 I/O
  const ScanProblem& p = a.p;
  const int tpc = a.tpc;
  const int tid = threadIdx.x;
  const int cl = tid / tpc, sg = tid - cl * tpc;
  const int ch = blockIdx.x * (kScanThreads / tpc) + cl;
  const int s = blockIdx.y, b = blockIdx.z;
  if (ch >= p.HP) return;  // the whole tpc-lane group of this channel leaves together
  const int h = ch / p.P, g = h / (p.H / p.G);
  const int N = p.N, n0 = sg * NS;
  const int t_begin = s * a.seg_len;
  const int t_end = min(p.L, t_begin + a.seg_len);
  const unsigned gmask = group_mask(tpc);

  float A2[SCALAR_A ? 1 : NS];
  if (SCALAR_A) {
    A2[0] = __ldg(p.A + h) * kLog2e;
  } else {
#pragma unroll
    for (int j = 0; j < NS; j++)
      A2[j] = (FULL || n0 + j < N) ? __ldg(p.A + (long)h * N + n0 + j) * kLog2e : 0.0f;
  }

  float hs[NS];
  if (LOCAL) {
#pragma unroll
    for (int j = 0; j < NS; j++) hs[j] = 0.0f;
  } else if (s == 0) {
    const float* row = start_row(p, b);
#pragma unroll
    for (int j = 0; j < NS; j++)
      hs[j] = (row && (FULL || n0 + j < N)) ? __ldg(row + (long)ch * N + n0 + j) : 0.0f;
  } else {
    const float* src = a.segstart + (((long)b * a.S + s) * p.HP + ch) * N + n0;
#pragma unroll
    for (int j = 0; j < NS; j++) hs[j] = (FULL || n0 + j < N) ? src[j] : 0.0f;
  }

  const IO* x = (const IO*)p.x;
  const IO* dt = (const IO*)p.dt;
  const IO* Bm = (const IO*)p.B;
  const IO* Cm = (const IO*)p.C;
  const IO* z = (const IO*)p.z;
  IO* y = (IO*)a.y;
  const float Dv = p.D ? __ldg(p.D + ch) : 0.0f;
  const float bias = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + h) : 0.0f;
  float sumd = 0.0f;

  for (int t = t_begin; t < t_end; t++) {
    if (!LOCAL && a.ckpt && (t % p.chunk) == 0) {
      float* dst = a.ckpt + (((long)b * p.n_chunks + t / p.chunk) * p.HP + ch) * N + n0;
#pragma unroll
      for (int j = 0; j < NS; j++)
        if (FULL || n0 + j < N) dst[j] = hs[j];
    }
    const long tok = (long)b * p.L + t;
    float dl = ld(dt + tok * p.H + h);
    if (p.softplus) dl = softplusf_(dl + bias);
    const float xv = ld(x + tok * p.HP + ch);
    const float dx = dl * xv;
    float Bv[NS], Cv[NS];
    load_row<IO, NS, FULL>(Bm + (tok * p.G + g) * N + n0, N - n0, Bv);
    if (!LOCAL) load_row<IO, NS, FULL>(Cm + (tok * p.G + g) * N + n0, N - n0, Cv);
    float acc = 0.0f;
    const DecayCoef as = SCALAR_A ? decay_coef<ACC>(dl, A2[0]) : DecayCoef{0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < NS; j++) {
      const DecayCoef av = SCALAR_A ? as : decay_coef<ACC>(dl, A2[j]);
      hs[j] = decay_step<ACC>(av, hs[j], dx * Bv[j]);
      if (!LOCAL) acc = fmaf(Cv[j], hs[j], acc);
    }
    if (LOCAL) {
      sumd += dl;
    } else {
      for (int off = tpc >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(gmask, acc, off);
      if (sg == 0 && y) {
        float yv = fmaf(Dv, xv, acc);
        if (z) yv *= siluf_(ld(z + tok * p.HP + ch));
        if (p.check_finite && !isfinite(yv)) record_status(p.status, SSM_ERR_NONFINITE);
        st(y + tok * p.HP + ch, yv);
      }
    }
  }

  if (LOCAL) {
    float* dst = a.hloc + (((long)b * a.S + s) * p.HP + ch) * N + n0;
#pragma unroll
    for (int j = 0; j < NS; j++)
      if (FULL || n0 + j < N) dst[j] = hs[j];
    if (sg == 0) a.sumdelta[((long)b * a.S + s) * p.HP + ch] = sumd;
  } else if (s == a.S - 1 && a.state_out) {
    float* dst = a.state_out + ((long)b * p.HP + ch) * N + n0;
#pragma unroll
    for (int j = 0; j < NS; j++)
      if (FULL || n0 + j < N) dst[j] = hs[j];
  }
}

// Composes the segments in order: start[s+1] = exp(A sum_delta[s]) start[s] + h_local[s].
__global__ void scan_fwd_carry_kernel(const FwdArgs a) {
  const ScanProblem& p = a.p;
  const long total = (long)p.ns * p.HP * p.N;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i % p.N);
    const long bc = i / p.N;
    const int ch = (int)(bc % p.HP), b = (int)(bc / p.HP);
    const int h = ch / p.P;
    const float A2 = (p.a_per_state ? __ldg(p.A + (long)h * p.N + n) : __ldg(p.A + h)) * kLog2e;
    const float* row = start_row(p, b);
    float hv = row ? __ldg(row + (long)ch * p.N + n) : 0.0f;
    for (int s = 0; s < a.S; s++) {
      const long si = ((long)b * a.S + s) * p.HP + ch;
      a.segstart[si * p.N + n] = hv;
      if (s + 1 < a.S) hv = fmaf(ex2(A2 * a.sumdelta[si]), hv, a.hloc[si * p.N + n]);
    }
  }
}

// ---- host side -------------------------------------------------------------------------
struct FwdPlan {
  int ns_state, tpc, S, seg_len;
  size_t off_segstart, off_hloc, off_sumdelta, bytes;
};

static FwdPlan plan_fwd(const ScanProblem& p, int num_sms) {
  FwdPlan q{};
  state_split(p.N, /*max_ns=*/16, &q.ns_state, &q.tpc);
  const long base_threads = (long)p.ns * p.HP * q.tpc;
  const long target = (long)num_sms * kFwdTargetThreadsPerSM;
  long S = (target + base_threads - 1) / base_threads;
  const long max_s = (p.L + kMinSegment - 1) / kMinSegment;
  if (S > max_s) S = max_s;
  if (S < 1) S = 1;
  q.seg_len = (int)((p.L + S - 1) / S);
  q.S = (p.L + q.seg_len - 1) / q.seg_len;
  size_t off = kStatusBytes;
  const size_t st_bytes = sizeof(float) * (size_t)p.ns * q.S * p.HP * p.N;
  if (q.S > 1) {
    q.off_segstart = off; off = align_up(off + st_bytes, 256);
    q.off_hloc = off; off = align_up(off + st_bytes, 256);
    q.off_sumdelta = off; off = align_up(off + sizeof(float) * (size_t)p.ns * q.S * p.HP, 256);
  }
  q.bytes = off;
  return q;
}

size_t scan_fwd_ws_bytes(const ScanProblem& p, int num_sms) {
  size_t a = plan_fwd(p, num_sms).bytes;
  const size_t b = scan_fwd_tma_ws_bytes(p, num_sms), c = scan_fwd_heads_ws_bytes(p, num_sms),
               d = scan_fwd_ssd_ws_bytes(p);
  if (b > a) a = b;
  if (d > a) a = d;
  return c > a ? c : a;
}

template <typename IO, int NS, bool SCALAR_A, bool FULL>
static void launch_fwd_t(const FwdArgs& a, int blocks_x, cudaStream_t st) {
  if (a.S > 1) {
    dim3 g1(blocks_x, a.S - 1, a.p.ns);
    scan_fwd_kernel<IO, NS, SCALAR_A, true, FULL><<<g1, kScanThreads, 0, st>>>(a), count_launches(1);
    const long total = (long)a.p.ns * a.p.HP * a.p.N;
    int nb = (int)((total + 255) / 256);
    scan_fwd_carry_kernel<<<nb, 256, 0, st>>>(a), count_launches(1);
  }
  dim3 g2(blocks_x, a.S, a.p.ns);
  scan_fwd_kernel<IO, NS, SCALAR_A, false, FULL><<<g2, kScanThreads, 0, st>>>(a), count_launches(1);
}

template <typename IO, int NS>
static void launch_fwd_ns(const FwdArgs& a, int blocks_x, bool full, cudaStream_t st) {
  const bool sa = !a.p.a_per_state;
  if (sa) {
    if (full) launch_fwd_t<IO, NS, true, true>(a, blocks_x, st);
    else launch_fwd_t<IO, NS, true, false>(a, blocks_x, st);
  } else {
    if (full) launch_fwd_t<IO, NS, false, true>(a, blocks_x, st);
    else launch_fwd_t<IO, NS, false, false>(a, blocks_x, st);
  }
}

template <typename IO>
static void launch_fwd_io(const FwdArgs& a, int ns_state, int blocks_x, bool full,
                          cudaStream_t st) {
  switch (ns_state) {
    case 4: launch_fwd_ns<IO, 4>(a, blocks_x, full, st); break;
    case 8: launch_fwd_ns<IO, 8>(a, blocks_x, full, st); break;
    default: launch_fwd_ns<IO, 16>(a, blocks_x, full, st); break;
  }
}

cudaError_t launch_scan_fwd(const ScanProblem& p, void* y, float* state_out, float* ckpt, void* ws,
                            int num_sms, cudaStream_t st) {
  cudaError_t e = launch_scan_fwd_tma(p, y, state_out, ckpt, ws, num_sms, st);
  if (e != cudaErrorNotSupported) return e;
  e = launch_scan_fwd_ssd(p, y, state_out, ckpt, ws, st);
  if (e != cudaErrorNotSupported) return e;
  e = launch_scan_fwd_heads(p, y, state_out, ckpt, ws, num_sms, st);
  if (e != cudaErrorNotSupported) return e;
  const FwdPlan q = plan_fwd(p, num_sms);
  FwdArgs a{};
  a.p = p;
  a.S = q.S;
  a.seg_len = q.seg_len;
  a.tpc = q.tpc;
  a.y = y;
  a.state_out = state_out;
  a.ckpt = ckpt;
  char* w = (char*)ws;
  if (q.S > 1) {
    a.segstart = (float*)(w + q.off_segstart);
    a.hloc = (float*)(w + q.off_hloc);
    a.sumdelta = (float*)(w + q.off_sumdelta);
  }
  const int cpb = kScanThreads / q.tpc;
  const int blocks_x = (p.HP + cpb - 1) / cpb;
  const bool full = rows_vectorizable(p, q.ns_state, q.tpc);
  if (p.io == SSM_BF16) launch_fwd_io<__nv_bfloat16>(a, q.ns_state, blocks_x, full, st);
  else launch_fwd_io<float>(a, q.ns_state, blocks_x, full, st);
  return cudaGetLastError();
}

}  // namespace ssm

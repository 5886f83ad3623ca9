// scan_fwd_tma.cuh -- forward scan with TMA-staged tiles: the fast path for head_dim 1 (the
// Mamba-1 layout), channel rows 16-byte aligned, d_state a multiple of 4 and a checkpoint
// interval that is a multiple of the 16-token tile; A per state or one A per channel; bf16 or
// fp32 I/O.  The Mamba-2 form (head_dim > 1) uses scan_fwd_heads.cu where it applies, other
// shapes scan_fwd.cu.
//
// Same arithmetic and segment decomposition as scan_fwd.cu (local aggregate, carry, main),
// but every block streams its inputs as [tile tokens][block channels] tiles of x, dt, z and
// [tile tokens][N] tiles of B, C into a ring of shared-memory stages: one elected thread
// issues 3-D cp.async.bulk.tensor loads that complete on an mbarrier per stage, so the loads
// of the next tiles overlap the arithmetic of this one.
// y leaves the same way, one tile per TMA store.  Segments are whole tiles long, so no tile
// straddles two segments; the sequence end is clipped by the tensor bounds (loads fill zeros,
// stores skip).
//
// Per tile a prepass does the per-(token, channel) work once -- delta (softplus when asked),
// delta x -- and lays B and C out as one record per 4 states (B then C: 16 bytes for bf16,
// 32 for fp32), so the recurrence reads a thread's states with one or two 16-byte loads.
// With one A per channel the decay is one exponential per (token, channel) for all states.
// fp32 I/O uses the accurate decay form h <- h + (expm1(delta A) h + u) (scan_common.cuh).
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"
#include "tma.cuh"

namespace ssm {

constexpr int kFwdStages = 3;
constexpr int kFwdTile = 16;  // tokens per staged tile
// Time segments: none when the (sequence, channel block) grid alone has kFwdNoSplitBlocksPerSM
// blocks per SM; otherwise enough for kFwdTargetBlocksPerSM (each extra segment costs a
// local-aggregate pass over its tokens; measured on GB300 with one long sequence).
constexpr long kFwdNoSplitBlocksPerSM = 4;
constexpr long kFwdTargetBlocksPerSM = 8;

struct FwdTmaArgs {
  CUtensorMap mx, mdt, mz, my, mb, mc;
  ScanProblem p;
  int S, seg_len, tpc, cb, tt;
  float* state_out;
  float* ckpt;
  float* segstart;
  float* hloc;
  float* sumdelta;
  int has_y;
  uint32_t bytes_main, bytes_local;        // expected transaction bytes per stage
  uint32_t off_x, off_dt, off_z, off_b, off_c, stage_stride;  // inside a stage
  uint32_t off_dd, off_bc, off_acc, off_par, off_y, y_stride, off_bar;
};

template <typename IO>
__device__ __forceinline__ float lds1(const IO* p) {
  if constexpr (sizeof(IO) == 4) return *reinterpret_cast<const float*>(p);
  else return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// A bf16 pair (one 32-bit word, low half first) as a packed fp32 pair; exact.
__device__ __forceinline__ f2_t fwd_bf2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// B and C of 4 states (n0 .. n0+3, n0 % 4 == 0) of token i from the record array.
template <typename IO>
__device__ __forceinline__ void ld_bc4(const unsigned char* rec, int i, int N, int n0,
                                      f2_t (&B2)[2], f2_t (&C2)[2]) {
  if constexpr (sizeof(IO) == 2) {
    const uint4 v = reinterpret_cast<const uint4*>(rec)[(i * N + n0) / 4];
    B2[0] = fwd_bf2_to_f2(v.x);
    B2[1] = fwd_bf2_to_f2(v.y);
    C2[0] = fwd_bf2_to_f2(v.z);
    C2[1] = fwd_bf2_to_f2(v.w);
  } else {
    const float4* r = reinterpret_cast<const float4*>(rec) + 2 * ((i * N + n0) / 4);
    const float4 vb = r[0], vc = r[1];
    B2[0] = f2_pack(vb.x, vb.y);
    B2[1] = f2_pack(vb.z, vb.w);
    C2[0] = f2_pack(vc.x, vc.y);
    C2[1] = f2_pack(vc.z, vc.w);
  }
}

// A block = 128 threads = (128 / TPC) channels x N states, NS = N / TPC states per thread, one
// sequence, one time segment.  SCALAR_A: one A per channel (the head of head_dim 1).
template <typename IO, int NS, int TPC, bool LOCAL, bool SCALAR_A>
__global__ void __launch_bounds__(kScanThreads)
scan_fwd_tma_kernel(const __grid_constant__ FwdTmaArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;  // accurate decay form for fp32 I/O
  constexpr int TT = kFwdTile;
  constexpr int tpc = TPC, cb = kScanThreads / TPC;  // compile-time: index math is shifts
  static_assert(NS % 4 == 0, "states per thread come in records of 4");
  extern __shared__ __align__(128) unsigned char smem[];
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x;
  const int cl = tid / tpc, sg = tid - cl * tpc;
  const int ch0 = blockIdx.x * cb, ch = ch0 + cl;
  const int s = blockIdx.y, b = blockIdx.z;
  const int N = p.N, n0 = sg * NS;
  const int g = ch0 / (p.H / p.G);
  const int t_begin = s * a.seg_len, t_end = min(p.L, t_begin + a.seg_len);
  const int ntiles = (t_end - t_begin + TT - 1) / TT;
  const uint32_t bytes = LOCAL ? a.bytes_local : a.bytes_main;
  const bool want_y = !LOCAL && a.has_y;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.off_bar);
  float2* sDD = reinterpret_cast<float2*>(smem + a.off_dd);  // [TT][cb] (delta, delta x)
  unsigned char* sBC = smem + a.off_bc;                       // [TT][N/4] records of B, C
  float* sACC = reinterpret_cast<float*>(smem + a.off_acc);  // [TT][cb * tpc] partial C . h
  float* sPar = reinterpret_cast<float*>(smem + a.off_par);  // [cb] D, [cb] dt_bias

  if (tid == 0) {
    for (int i = 0; i < kFwdStages; i++) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  for (int c = tid; c < cb; c += kScanThreads) {
    sPar[c] = p.D ? __ldg(p.D + ch0 + c) : 0.0f;
    sPar[cb + c] = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + ch0 + c) : 0.0f;
  }
  __syncthreads();
  auto issue = [&](int k) {  // tile k -> stage k % kFwdStages (thread 0 only)
    const int stg = k % kFwdStages;
    unsigned char* base = smem + stg * a.stage_stride;
    const int t0 = t_begin + k * TT;
    mbar_expect_tx(&full[stg], bytes);
    tma_load_3d(base + a.off_x, &a.mx, ch0, t0, b, &full[stg]);
    tma_load_3d(base + a.off_dt, &a.mdt, ch0, t0, b, &full[stg]);
    tma_load_3d(base + a.off_b, &a.mb, g * N, t0, b, &full[stg]);
    if (!LOCAL) {
      if (p.z) tma_load_3d(base + a.off_z, &a.mz, ch0, t0, b, &full[stg]);
      tma_load_3d(base + a.off_c, &a.mc, g * N, t0, b, &full[stg]);
    }
  };
  if (tid == 0)
    for (int k = 0; k < kFwdStages && k < ntiles; k++) issue(k);

  f2_t A2p[SCALAR_A ? 1 : NS / 2], hp[NS / 2];
  float A2s = 0.0f;
  {
    const float* row = nullptr;
    if (!LOCAL) row = s == 0 ? start_row(p, b) : a.segstart + (((long)b * a.S + s) * p.HP) * N;
    if constexpr (SCALAR_A) {
      A2s = __ldg(p.A + ch) * kLog2e;
    } else {
#pragma unroll
      for (int j = 0; j < NS / 2; j++)
        A2p[j] = f2_pack(__ldg(p.A + (long)ch * N + n0 + 2 * j) * kLog2e,
                         __ldg(p.A + (long)ch * N + n0 + 2 * j + 1) * kLog2e);
    }
#pragma unroll
    for (int j = 0; j < NS / 2; j++) {
      const float h0 = row ? row[(long)ch * N + n0 + 2 * j] : 0.0f;
      const float h1 = row ? row[(long)ch * N + n0 + 2 * j + 1] : 0.0f;
      hp[j] = f2_pack(h0, h1);
    }
  }
  float sumd = 0.0f;

  for (int k = 0; k < ntiles; k++) {
    const int stg = k % kFwdStages;
    if (want_y && tid == 0) tma_store_wait_read<1>();  // store k-2 has read its y buffer
    const bool ok = mbar_wait(&full[stg], (uint32_t)(k / kFwdStages) & 1u);
    if (__syncthreads_or(!ok)) {  // a tile never arrived: report, drain, leave
      if (tid == 0) {
        record_status(p.status, SSM_ERR_TIMEOUT);
        for (int j = k; j < ntiles && j < k + kFwdStages; j++)
          mbar_wait(&full[j % kFwdStages], (uint32_t)(j / kFwdStages) & 1u);
        tma_store_wait_all();
      }
      return;
    }
    unsigned char* base = smem + stg * a.stage_stride;
    const IO* sx = reinterpret_cast<const IO*>(base + a.off_x);
    const IO* sdt = reinterpret_cast<const IO*>(base + a.off_dt);
    const IO* sz = reinterpret_cast<const IO*>(base + a.off_z);
    const int t0 = t_begin + k * TT;
    const int cnt = min(TT, t_end - t0);

    // ---- prepass, once per (token, channel): delta, delta x; B, C records -------------------
    for (int idx = tid; idx < TT * cb; idx += kScanThreads) {
      const int i = idx / cb, c = idx - i * cb;
      float dl = lds1(sdt + idx);
      if (p.softplus) dl = softplusf_(dl + sPar[cb + c]);
      sDD[idx] = make_float2(dl, dl * lds1(sx + idx));
    }
    for (int idx = tid; idx < TT * N / 4; idx += kScanThreads) {
      if constexpr (sizeof(IO) == 2) {
        const uint2 vb = reinterpret_cast<const uint2*>(base + a.off_b)[idx];
        const uint2 vc = LOCAL ? make_uint2(0u, 0u) : reinterpret_cast<const uint2*>(base + a.off_c)[idx];
        reinterpret_cast<uint4*>(sBC)[idx] = make_uint4(vb.x, vb.y, vc.x, vc.y);
      } else {
        const float4 vb = reinterpret_cast<const float4*>(base + a.off_b)[idx];
        const float4 vc = LOCAL ? make_float4(0.f, 0.f, 0.f, 0.f)
                                : reinterpret_cast<const float4*>(base + a.off_c)[idx];
        reinterpret_cast<float4*>(sBC)[2 * idx] = vb;
        reinterpret_cast<float4*>(sBC)[2 * idx + 1] = vc;
      }
    }
    __syncthreads();

    // ---- the recurrence: per thread, its channel's NS states over the tile ------------------
    if (!LOCAL && a.ckpt && t0 % p.chunk == 0) {  // checkpoints fall on tile starts
      float* dst = a.ckpt + (((long)b * p.n_chunks + t0 / p.chunk) * p.HP + ch) * N + n0;
#pragma unroll
      for (int j = 0; j < NS / 2; j += 2) {
        float x0, x1, x2, x3;
        f2_unpack(hp[j], x0, x1);
        f2_unpack(hp[j + 1], x2, x3);
        *reinterpret_cast<float4*>(dst + 2 * j) = make_float4(x0, x1, x2, x3);
      }
    }
    auto token = [&](int i) {
      const float2 dd = sDD[i * cb + cl];
      const f2_t dx2 = f2_pack(dd.y, dd.y);
      f2_t dl2 = 0ull, cs2 = 0ull;
      if constexpr (SCALAR_A) {
        const float cf = decay_coef<ACC>(dd.x, A2s);  // one decay for all the thread's states
        cs2 = f2_pack(cf, cf);
      } else {
        dl2 = f2_pack(dd.x, dd.x);
      }
      f2_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
      for (int j = 0; j < NS; j += 4) {
        f2_t B2[2], C2[2];
        ld_bc4<IO>(sBC, i, N, n0 + j, B2, C2);
        const int q = j / 2;
#pragma unroll
        for (int e = 0; e < 2; e++) {
          const f2_t cf2 = SCALAR_A ? cs2 : decay2<ACC>(dl2, A2p[SCALAR_A ? 0 : q + e]);
          hp[q + e] = step2<ACC>(cf2, hp[q + e], f2_mul(dx2, B2[e]));
        }
        if (!LOCAL) {
          acc0 = f2_fma(C2[0], hp[q], acc0);
          acc1 = f2_fma(C2[1], hp[q + 1], acc1);
        }
      }
      if (LOCAL) {
        sumd += dd.x;
      } else {
        float lo, hi;
        f2_unpack(f2_add(acc0, acc1), lo, hi);
        sACC[i * cb * tpc + tid] = lo + hi;
      }
    };
    if (cnt == TT) {  // full tile: no per-token branch, so tokens can interleave
#pragma unroll
      for (int i = 0; i < TT; i++) token(i);
    } else {
#pragma unroll
      for (int i = 0; i < TT; i++)
        if (i < cnt) token(i);
    }
    __syncthreads();

    // ---- epilogue, once per (token, channel): y = (C . h + D x) silu(z) -> TMA store -----------
    if (want_y) {
      IO* sy = reinterpret_cast<IO*>(smem + a.off_y + (k & 1) * a.y_stride);
      for (int idx = tid; idx < cnt * cb; idx += kScanThreads) {
        const int i = idx / cb, c = idx - i * cb;
        const float* pa = sACC + (i * cb + c) * tpc;  // the channel's tpc partials, contiguous
        float acc;
        if constexpr (tpc == 8) {
          const float4 v = *reinterpret_cast<const float4*>(pa);
          const float4 w = *reinterpret_cast<const float4*>(pa + 4);
          acc = ((v.x + v.y) + (v.z + v.w)) + ((w.x + w.y) + (w.z + w.w));
        } else if constexpr (tpc == 4) {
          const float4 v = *reinterpret_cast<const float4*>(pa);
          acc = (v.x + v.y) + (v.z + v.w);
        } else if constexpr (tpc == 2) {
          const float2 v = *reinterpret_cast<const float2*>(pa);
          acc = v.x + v.y;
        } else {
          acc = pa[0];
        }
        float yv = fmaf(sPar[c], lds1(sx + idx), acc);
        if (p.z) yv *= siluf_(lds1(sz + idx));
        if (p.check_finite && !isfinite(yv)) record_status(p.status, SSM_ERR_NONFINITE);
        if constexpr (sizeof(IO) == 4) sy[idx] = yv;
        else sy[idx] = __float2bfloat16_rn(yv);
      }
      fence_async_shared();
      __syncthreads();  // y tile complete; stage stg fully read
      if (tid == 0) {
        tma_store_3d(&a.my, sy, ch0, t0, b);
        tma_store_commit();
      }
    }
    if (tid == 0 && k + kFwdStages < ntiles) issue(k + kFwdStages);
  }
  if (want_y && tid == 0) tma_store_wait_all();

  float* dst = nullptr;
  if (LOCAL) {
    dst = a.hloc + (((long)b * a.S + s) * p.HP + ch) * N + n0;
    if (sg == 0) a.sumdelta[((long)b * a.S + s) * p.HP + ch] = sumd;
  } else if (s == a.S - 1 && a.state_out) {
    dst = a.state_out + ((long)b * p.HP + ch) * N + n0;
  }
  if (dst) {
#pragma unroll
    for (int j = 0; j < NS / 2; j++) f2_unpack(hp[j], dst[2 * j], dst[2 * j + 1]);
  }
}

// Composes the segments in order, as scan_fwd.cu's carry kernel: start[s+1] =
// exp(A sum_delta[s]) start[s] + h_local[s].  (A template so that each translation unit that
// launches it holds its own instance.)
template <typename IO>
__global__ void scan_fwd_tma_carry_kernel(const __grid_constant__ FwdTmaArgs a) {
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

template <typename IO, int NS, int TPC, bool SCALAR_A>
cudaError_t launch_fwd_tma_t(FwdTmaArgs& a, size_t smem, cudaStream_t st) {
  auto km = scan_fwd_tma_kernel<IO, NS, TPC, false, SCALAR_A>;
  auto kl = scan_fwd_tma_kernel<IO, NS, TPC, true, SCALAR_A>;
  cudaError_t e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kl, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int bx = a.p.HP / a.cb;
  if (a.S > 1) {
    kl<<<dim3(bx, a.S - 1, a.p.ns), kScanThreads, smem, st>>>(a), count_launches(1);
    const long total = (long)a.p.ns * a.p.HP * a.p.N;
    scan_fwd_tma_carry_kernel<IO><<<(int)((total + 255) / 256), 256, 0, st>>>(a), count_launches(1);
  }
  km<<<dim3(bx, a.S, a.p.ns), kScanThreads, smem, st>>>(a), count_launches(1);
  return cudaGetLastError();
}

// The (states per thread, threads per channel, A form) combinations instantiated for each I/O
// type; X(NS, TPC, SCALAR_A).
#define SSM_FWD_TMA_VARIANTS(X) \
  X(16, 1, false) X(8, 2, false) X(4, 4, false) X(16, 2, false) X(8, 4, false) X(16, 4, false) \
  X(16, 8, true) X(8, 4, true) X(16, 4, true) X(4, 4, true)

}  // namespace ssm

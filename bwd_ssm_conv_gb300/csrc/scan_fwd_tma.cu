// scan_fwd_tma.cu -- forward scan with TMA-staged tiles: the fast path for the Mamba-1
// layout with bf16 I/O (head_dim 1; channel rows 16-byte aligned; checkpoint interval a
// multiple of the 16-token tile).  Other shapes and fp32 I/O use scan_fwd.cu.
//
// Same arithmetic and segment decomposition as scan_fwd.cu (local aggregate, carry, main),
// but every block streams its inputs as [tile tokens][block channels] tiles of x, dt, z and
// [tile tokens][N] tiles of B, C into a ring of shared-memory stages: one elected thread
// issues 3-D cp.async.bulk.tensor loads that complete on an mbarrier per stage, so the
// loads of the next tiles overlap the arithmetic of this one.  y leaves the same way, one
// tile per TMA store.  Segments are whole tiles long, so no tile straddles two segments;
// the sequence end is clipped by the tensor bounds (loads fill zeros, stores skip).
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
  uint32_t off_dl, off_dx, off_bf, off_cf, off_acc, off_par, off_y, y_stride, off_bar;
};

template <typename IO>
__device__ __forceinline__ float lds1(const IO* p) {
  if constexpr (sizeof(IO) == 4) return *reinterpret_cast<const float*>(p);
  else return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// NS consecutive values of a shared-memory row (16-byte aligned when NS*sizeof(IO) >= 16).
template <typename IO, int NS>
__device__ __forceinline__ void lds_row(const IO* ptr, float (&out)[NS]) {
  if constexpr (sizeof(IO) == 4) {
#pragma unroll
    for (int j = 0; j < NS; j += 4) {
      const float4 v = *reinterpret_cast<const float4*>(ptr + j);
      out[j] = v.x; out[j + 1] = v.y; out[j + 2] = v.z; out[j + 3] = v.w;
    }
  } else if constexpr (NS >= 8) {
#pragma unroll
    for (int j = 0; j < NS; j += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(ptr + j);
      const __nv_bfloat162* q = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const float2 f = __bfloat1622float2(q[k]);
        out[j + 2 * k] = f.x; out[j + 2 * k + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < NS; j += 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(ptr + j);
      const __nv_bfloat162* q = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int k = 0; k < 2; k++) {
        const float2 f = __bfloat1622float2(q[k]);
        out[j + 2 * k] = f.x; out[j + 2 * k + 1] = f.y;
      }
    }
  }
}

// A bf16 pair (one 32-bit word, low half first) as a packed fp32 pair; exact.
__device__ __forceinline__ f2_t bf2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <typename IO, int NS, int TPC, bool LOCAL>
__global__ void __launch_bounds__(kScanThreads)
scan_fwd_tma_kernel(const __grid_constant__ FwdTmaArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;
  constexpr int TT = kFwdTile;
  extern __shared__ __align__(128) unsigned char smem[];
  const ScanProblem& p = a.p;
  constexpr int tpc = TPC, cb = kScanThreads / TPC;  // compile-time: index math is shifts
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
  float2* sDD = reinterpret_cast<float2*>(smem + a.off_dl);  // [TT][cb] (delta, delta x)
  // [TT][N/4]: per token and group of 4 states, B then C as 8 bf16 (one 16-byte load per lane)
  uint4* sBC = reinterpret_cast<uint4*>(smem + a.off_bf);
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

  static_assert(!ACC, "the TMA forward path runs the fast decay form (bf16 I/O)");
  f2_t A2p[NS / 2], hp[NS / 2];
  {
    const float* row = nullptr;
    if (!LOCAL) row = s == 0 ? start_row(p, b) : a.segstart + (((long)b * a.S + s) * p.HP) * N;
#pragma unroll
    for (int j = 0; j < NS / 2; j++) {
      A2p[j] = f2_pack(__ldg(p.A + (long)ch * N + n0 + 2 * j) * kLog2e,
                       __ldg(p.A + (long)ch * N + n0 + 2 * j + 1) * kLog2e);
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

    // ---- prepass, once per (token, channel): delta, delta x; B, C to fp32 --------------------
    for (int idx = tid; idx < TT * cb; idx += kScanThreads) {
      const int i = idx / cb, c = idx - i * cb;
      float dl = lds1(sdt + idx);
      if (p.softplus) dl = softplusf_(dl + sPar[cb + c]);
      const float dx = dl * lds1(sx + idx);
      sDD[idx] = make_float2(dl, dx);
      (void)i;
    }
    {
      const uint2* rB = reinterpret_cast<const uint2*>(base + a.off_b);
      const uint2* rC = reinterpret_cast<const uint2*>(base + a.off_c);
      for (int idx = tid; idx < TT * N / 4; idx += kScanThreads) {
        const uint2 vb = rB[idx], vc = LOCAL ? make_uint2(0u, 0u) : rC[idx];
        sBC[idx] = make_uint4(vb.x, vb.y, vc.x, vc.y);
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
      const f2_t dl2 = f2_pack(dd.x, dd.x), dx2 = f2_pack(dd.y, dd.y);
      f2_t B2[NS / 2], C2[NS / 2];
#pragma unroll
      for (int j = 0; j < NS; j += 4) {
        const uint4 v = sBC[(i * N + n0 + j) / 4];
        B2[j / 2] = bf2_to_f2(v.x);
        B2[j / 2 + 1] = bf2_to_f2(v.y);
        C2[j / 2] = bf2_to_f2(v.z);
        C2[j / 2 + 1] = bf2_to_f2(v.w);
      }
      if (LOCAL) {
        (void)C2;
#pragma unroll
        for (int j = 0; j < NS / 2; j++)
          hp[j] = f2_fma(f2_ex2(f2_mul(dl2, A2p[j])), hp[j], f2_mul(dx2, B2[j]));
        sumd += dd.x;
      } else {
        f2_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int j = 0; j < NS; j += 4) {
          const int q = j / 2;
          hp[q] = f2_fma(f2_ex2(f2_mul(dl2, A2p[q])), hp[q], f2_mul(dx2, B2[q]));
          hp[q + 1] = f2_fma(f2_ex2(f2_mul(dl2, A2p[q + 1])), hp[q + 1], f2_mul(dx2, B2[q + 1]));
          acc0 = f2_fma(C2[q], hp[q], acc0);
          acc1 = f2_fma(C2[q + 1], hp[q + 1], acc1);
        }
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
        if (tpc == 4) {
          const float4 v = *reinterpret_cast<const float4*>(pa);
          acc = (v.x + v.y) + (v.z + v.w);
        } else if (tpc == 2) {
          const float2 v = *reinterpret_cast<const float2*>(pa);
          acc = v.x + v.y;
        } else {
          acc = 0.0f;
          for (int q = 0; q < tpc; q++) acc += pa[q];
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

// Same composition as scan_fwd.cu's carry kernel (kept separate to keep that file unchanged).
__global__ void scan_fwd_tma_carry_kernel(const __grid_constant__ FwdTmaArgs a) {
  const ScanProblem& p = a.p;
  const long total = (long)p.ns * p.HP * p.N;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i % p.N);
    const long bc = i / p.N;
    const int ch = (int)(bc % p.HP), b = (int)(bc / p.HP);
    const float A2 = __ldg(p.A + (long)ch * p.N + n) * kLog2e;
    const float* row = start_row(p, b);
    float hv = row ? __ldg(row + (long)ch * p.N + n) : 0.0f;
    for (int s = 0; s < a.S; s++) {
      const long si = ((long)b * a.S + s) * p.HP + ch;
      a.segstart[si * p.N + n] = hv;
      if (s + 1 < a.S) hv = fmaf(ex2(A2 * a.sumdelta[si]), hv, a.hloc[si * p.N + n]);
    }
  }
}

// ---- host ------------------------------------------------------------------------------
struct FwdTmaPlan {
  bool ok;
  int ns_state, tpc, cb, tt, S, seg_len;
  size_t smem, off_segstart, off_hloc, off_sumdelta, bytes;
};

static bool aligned16(const void* q) { return ((uintptr_t)q & 15) == 0; }

static FwdTmaPlan plan_fwd_tma(const ScanProblem& p, int num_sms) {
  FwdTmaPlan q{};
  const int io = p.io == SSM_BF16 ? 2 : 4;
  if (p.io != SSM_BF16 || p.P != 1 || !p.a_per_state || p.N > 256 || (p.N * io) % 16 != 0 ||
      (p.HP * io) % 16 != 0 || p.chunk % kFwdTile != 0)
    return q;
  // largest states-per-thread that still gives four blocks per SM without time segments
  // (the recurrence is latency-bound: more warps per SM beat fewer instructions per state)
  int ns = 0;
  for (int cand = 16; cand >= 4; cand >>= 1) {
    if (p.N % cand != 0) continue;
    ns = cand;
    const int cb = kScanThreads / (p.N / cand);
    if (cb > 0 && (long)p.ns * ((p.HP + cb - 1) / cb) >= 4L * num_sms) break;
  }
  if (ns < 4 || p.N / ns > 4) return q;  // instantiated: 1, 2 or 4 threads per channel
  q.ns_state = ns;
  q.tpc = p.N / ns;
  if (q.tpc > 32) return q;
  q.cb = kScanThreads / q.tpc;
  if ((p.H / p.G) % q.cb != 0 || p.HP % q.cb != 0 || q.cb * io < 16) return q;
  const int zt = p.z ? 1 : 0;
  const int per_tok = q.cb * io * (2 + zt) + 2 * p.N * io;
  (void)per_tok;
  q.tt = kFwdTile;
  const long base = (long)p.ns * (p.HP / q.cb);
  long S = base >= kFwdNoSplitBlocksPerSM * num_sms
               ? 1 : (kFwdTargetBlocksPerSM * num_sms + base - 1) / base;
  const long max_s = (p.L + kMinSegment - 1) / kMinSegment;
  if (S > max_s) S = max_s;
  if (S < 1) S = 1;
  int seg = (int)((p.L + S - 1) / S);
  seg = (seg + q.tt - 1) / q.tt * q.tt;
  q.seg_len = seg;
  q.S = (p.L + seg - 1) / seg;
  size_t off = kStatusBytes;
  const size_t st_bytes = sizeof(float) * (size_t)p.ns * q.S * p.HP * p.N;
  if (q.S > 1) {
    q.off_segstart = off; off = align_up(off + st_bytes, 256);
    q.off_hloc = off; off = align_up(off + st_bytes, 256);
    q.off_sumdelta = off; off = align_up(off + sizeof(float) * (size_t)p.ns * q.S * p.HP, 256);
  }
  q.bytes = off;
  q.ok = aligned16(p.x) && aligned16(p.dt) && aligned16(p.B) && aligned16(p.C) &&
         (!p.z || aligned16(p.z));
  return q;
}

size_t scan_fwd_tma_ws_bytes(const ScanProblem& p, int num_sms) {
  const FwdTmaPlan q = plan_fwd_tma(p, num_sms);
  return q.ok ? q.bytes : 0;
}

template <typename IO, int NS, int TPC>
static cudaError_t launch_fwd_tma_t(FwdTmaArgs& a, size_t smem, cudaStream_t st) {
  auto km = scan_fwd_tma_kernel<IO, NS, TPC, false>;
  auto kl = scan_fwd_tma_kernel<IO, NS, TPC, true>;
  cudaError_t e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kl, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int bx = a.p.HP / a.cb;
  if (a.S > 1) {
    kl<<<dim3(bx, a.S - 1, a.p.ns), kScanThreads, smem, st>>>(a), count_launches(1);
    const long total = (long)a.p.ns * a.p.HP * a.p.N;
    scan_fwd_tma_carry_kernel<<<(int)((total + 255) / 256), 256, 0, st>>>(a), count_launches(1);
  }
  km<<<dim3(bx, a.S, a.p.ns), kScanThreads, smem, st>>>(a), count_launches(1);
  return cudaGetLastError();
}

// Returns cudaErrorNotSupported (without launching anything) when the fast path does not
// apply to this problem; the caller then uses the general kernels.
cudaError_t launch_scan_fwd_tma(const ScanProblem& p, void* y, float* state_out, float* ckpt,
                                void* ws, int num_sms, cudaStream_t st) {
  const FwdTmaPlan q = plan_fwd_tma(p, num_sms);
  if (!q.ok || (y && !aligned16(y)) || (ckpt && !aligned16(ckpt))) return cudaErrorNotSupported;
  const int io = p.io == SSM_BF16 ? 2 : 4;
  FwdTmaArgs a;
  memset(&a, 0, sizeof(a));
  a.p = p;
  a.S = q.S; a.seg_len = q.seg_len; a.tpc = q.tpc; a.cb = q.cb; a.tt = q.tt;
  a.state_out = state_out; a.ckpt = ckpt; a.has_y = y != nullptr;
  char* w = (char*)ws;
  if (q.S > 1) {
    a.segstart = (float*)(w + q.off_segstart);
    a.hloc = (float*)(w + q.off_hloc);
    a.sumdelta = (float*)(w + q.off_sumdelta);
  }
  const uint64_t C = p.HP, L = p.L, NSq = p.ns, GN = (uint64_t)p.G * p.N;
  bool ok = encode_tmap_3d(&a.mx, p.x, io, C, L, NSq, C, C * L, q.cb, q.tt, 1) &&
            encode_tmap_3d(&a.mdt, p.dt, io, C, L, NSq, C, C * L, q.cb, q.tt, 1) &&
            encode_tmap_3d(&a.mb, p.B, io, GN, L, NSq, GN, GN * L, p.N, q.tt, 1) &&
            encode_tmap_3d(&a.mc, p.C, io, GN, L, NSq, GN, GN * L, p.N, q.tt, 1);
  if (ok && p.z) ok = encode_tmap_3d(&a.mz, p.z, io, C, L, NSq, C, C * L, q.cb, q.tt, 1);
  if (ok && y) ok = encode_tmap_3d(&a.my, y, io, C, L, NSq, C, C * L, q.cb, q.tt, 1);
  if (!ok) return cudaErrorNotSupported;
  const uint32_t tile = (uint32_t)(q.tt * q.cb * io), row = (uint32_t)(q.tt * p.N * io);
  auto al = [](uint32_t v) { return (v + 127u) & ~127u; };
  a.off_x = 0;
  a.off_dt = al(tile);
  a.off_z = a.off_dt + al(tile);
  a.off_b = a.off_z + (p.z ? al(tile) : 0);
  a.off_c = a.off_b + al(row);
  a.stage_stride = a.off_c + al(row);
  const uint32_t f_tile = (uint32_t)(q.tt * q.cb * 4), f_row = (uint32_t)(q.tt * p.N * 4);
  a.off_dl = kFwdStages * a.stage_stride;         // float2 (delta, delta x) per item
  a.off_dx = a.off_dl + al(2 * f_tile);
  a.off_bf = a.off_dx;                            // interleaved bf16 B, C: TT x N x 2 x 2 bytes
  a.off_cf = a.off_bf;
  a.off_acc = a.off_bf + al(f_row);
  a.off_par = a.off_acc + al((uint32_t)(q.tt * kScanThreads * 4));
  a.off_y = a.off_par + al((uint32_t)(2 * q.cb * 4));
  a.y_stride = al(tile);
  a.off_bar = a.off_y + 2 * a.y_stride;
  const size_t smem = a.off_bar + 64;
  a.bytes_local = 2 * tile + row;
  a.bytes_main = (2 + (p.z ? 1 : 0)) * tile + 2 * row;
  // (states per thread, threads per channel) pairs for d_state 16, 32, 64 (others: general path)
  const int key = q.ns_state * 100 + q.tpc;
  switch (key) {
    case 1601: return launch_fwd_tma_t<__nv_bfloat16, 16, 1>(a, smem, st);
    case 802: return launch_fwd_tma_t<__nv_bfloat16, 8, 2>(a, smem, st);
    case 404: return launch_fwd_tma_t<__nv_bfloat16, 4, 4>(a, smem, st);
    case 1602: return launch_fwd_tma_t<__nv_bfloat16, 16, 2>(a, smem, st);
    case 804: return launch_fwd_tma_t<__nv_bfloat16, 8, 4>(a, smem, st);
    case 1604: return launch_fwd_tma_t<__nv_bfloat16, 16, 4>(a, smem, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace ssm

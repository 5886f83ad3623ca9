// scan_fwd_heads.cu -- forward scan for the Mamba-2 form: one A per head, head_dim P a multiple
// of 64, d_state 128 (ggmlR's ssm_scan with a [1, n_head] A; the recurrence of infotheory's
// mamba1/model.rs with the decay shared by all states of a head).
//
// A block = 256 threads = one head's 64 channels x 128 states, one sequence, one time segment.
// A thread holds a 4-channel x 8-state tile of the state: per token it needs 4 values of
// delta x, 8 of B and 8 of C (0.6 loads per state), and the decay exp(delta A) is one value per
// (token, head), computed once per tile.  A warp = 2 channel groups x 16 state groups, so the
// sum over states for y closes inside the warp (a transposed shuffle reduction).  Tiles of x,
// z, dt, B, C arrive by cp.async.bulk.tensor into a 2-stage mbarrier ring; y leaves by TMA
// store.  Time segments compose exactly as in scan_fwd.cu (local aggregate, carry, main).
#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"
#include "tma.cuh"

namespace ssm {

namespace {

constexpr int kMhThreads = 256;
constexpr int kMhStages = 2;
constexpr int kMhTile = 16;     // tokens per staged tile
constexpr int kMhP = 64;        // channels per block
constexpr int kMhN = 128;       // d_state
constexpr int kMhTP = 4;        // channels per thread
constexpr int kMhTN = 8;        // states per thread

struct MhArgs {
  CUtensorMap mx, mdt, mz, my, mb, mc;
  ScanProblem p;
  int S, seg_len, dt_box;
  float* state_out;
  float* ckpt;
  float* segstart;  // [ns][S][HP][N]
  float* hloc;      // [ns][S][HP][N]
  float* sumdelta;  // [ns][S][HP]
  int has_y;
  uint32_t bytes_main, bytes_local;
  uint32_t off_x, off_dt, off_z, off_b, off_c, stage_stride;
  uint32_t off_dx, off_t, off_bf, off_cf, off_yp, off_y, y_stride, off_bar;
};

template <typename IO>
__device__ __forceinline__ float mh_lds(const IO* p) {
  if constexpr (sizeof(IO) == 4) return *reinterpret_cast<const float*>(p);
  else return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

template <typename IO, bool LOCAL>
__global__ void __launch_bounds__(kMhThreads)
scan_fwd_heads_kernel(const __grid_constant__ MhArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;  // accurate decay form for fp32 I/O
  constexpr int TT = kMhTile, N = kMhN;
  extern __shared__ __align__(128) unsigned char smem[];
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ng = lane & 15, pgl = lane >> 4;
  const int pl0 = warp * 8 + pgl * kMhTP;  // first of this thread's 4 channels, within the block
  const int n0 = ng * kMhTN;               // first of its 8 states
  const int blocks_per_head = p.P / kMhP;
  const int h = blockIdx.x / blocks_per_head;
  const int ch0 = h * p.P + (blockIdx.x - h * blocks_per_head) * kMhP;
  const int g = h / (p.H / p.G);
  const int h_lo = h / a.dt_box * a.dt_box;
  const int s = blockIdx.y, b = blockIdx.z;
  const int t_begin = s * a.seg_len, t_end = min(p.L, t_begin + a.seg_len);
  const int ntiles = (t_end - t_begin + TT - 1) / TT;
  const uint32_t bytes = LOCAL ? a.bytes_local : a.bytes_main;
  const bool want_y = !LOCAL && a.has_y;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.off_bar);
  float* sDX = reinterpret_cast<float*>(smem + a.off_dx);   // [TT][64] delta x
  float2* sT = reinterpret_cast<float2*>(smem + a.off_t);   // [TT] (decay coefficient, delta)
  float* sYP = reinterpret_cast<float*>(smem + a.off_yp);   // [TT][64] C . h

  if (tid == 0) {
    for (int i = 0; i < kMhStages; i++) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int k) {  // tile k -> stage k % kMhStages (thread 0 only)
    const int stg = k % kMhStages;
    unsigned char* base = smem + stg * a.stage_stride;
    const int t0 = t_begin + k * TT;
    mbar_expect_tx(&full[stg], bytes);
    tma_load_3d(base + a.off_x, &a.mx, ch0, t0, b, &full[stg]);
    tma_load_3d(base + a.off_dt, &a.mdt, h_lo, t0, b, &full[stg]);
    tma_load_3d(base + a.off_b, &a.mb, g * N, t0, b, &full[stg]);
    if (!LOCAL) {
      if (p.z) tma_load_3d(base + a.off_z, &a.mz, ch0, t0, b, &full[stg]);
      tma_load_3d(base + a.off_c, &a.mc, g * N, t0, b, &full[stg]);
    }
  };
  if (tid == 0)
    for (int k = 0; k < kMhStages && k < ntiles; k++) issue(k);

  const float A2 = __ldg(p.A + h) * kLog2e;
  const float bias = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + h) : 0.0f;
  f2_t hs[kMhTP][kMhTN / 2];  // [channel][state pair]
  {
    const float* row = nullptr;
    if (!LOCAL) row = s == 0 ? start_row(p, b) : a.segstart + (((long)b * a.S + s) * p.HP) * N;
#pragma unroll
    for (int c = 0; c < kMhTP; c++) {
      const float* r = row ? row + (long)(ch0 + pl0 + c) * N + n0 : nullptr;
#pragma unroll
      for (int q = 0; q < kMhTN / 2; q++)
        hs[c][q] = r ? f2_pack(r[2 * q], r[2 * q + 1]) : 0ull;
    }
  }
  float sumd = 0.0f;

  for (int k = 0; k < ntiles; k++) {
    const int stg = k % kMhStages;
    if (want_y && tid == 0) tma_store_wait_read<1>();  // store k-2 has read its y buffer
    const bool ok = mbar_wait(&full[stg], (uint32_t)(k / kMhStages) & 1u);
    if (__syncthreads_or(!ok)) {  // a tile never arrived: report, drain, leave
      if (tid == 0) {
        record_status(p.status, SSM_ERR_TIMEOUT);
        for (int j = k; j < ntiles && j < k + kMhStages; j++)
          mbar_wait(&full[j % kMhStages], (uint32_t)(j / kMhStages) & 1u);
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

    // ---- prepass: per token delta and the decay; per (token, channel) delta x; B, C fp32 -----
    if (tid < TT) {
      float dl = mh_lds(sdt + tid * a.dt_box + (h - h_lo));
      if (p.softplus) dl = softplusf_(dl + bias);
      sT[tid] = make_float2(decay_coef<ACC>(dl, A2).c, dl);  // s is the form's constant
    }
    __syncthreads();
    for (int idx = tid; idx < TT * kMhP; idx += kMhThreads)
      sDX[idx] = sT[idx / kMhP].y * mh_lds(sx + idx);
    const float* sBf;
    const float* sCf;
    if constexpr (sizeof(IO) == 4) {
      sBf = reinterpret_cast<const float*>(base + a.off_b);
      sCf = reinterpret_cast<const float*>(base + a.off_c);
    } else {
      float* wB = reinterpret_cast<float*>(smem + a.off_bf);
      float* wC = reinterpret_cast<float*>(smem + a.off_cf);
      const IO* rB = reinterpret_cast<const IO*>(base + a.off_b);
      const IO* rC = reinterpret_cast<const IO*>(base + a.off_c);
      for (int idx = tid; idx < TT * N; idx += kMhThreads) {
        wB[idx] = mh_lds(rB + idx);
        if (!LOCAL) wC[idx] = mh_lds(rC + idx);
      }
      sBf = wB;
      sCf = wC;
    }
    __syncthreads();

    if (!LOCAL && a.ckpt && t0 % p.chunk == 0) {  // checkpoints fall on tile starts
#pragma unroll
      for (int c = 0; c < kMhTP; c++) {
        float* dst = a.ckpt + (((long)b * p.n_chunks + t0 / p.chunk) * p.HP + ch0 + pl0 + c) * N + n0;
#pragma unroll
        for (int q = 0; q < kMhTN / 2; q += 2) {
          float x0, x1, x2, x3;
          f2_unpack(hs[c][q], x0, x1);
          f2_unpack(hs[c][q + 1], x2, x3);
          *reinterpret_cast<float4*>(dst + 2 * q) = make_float4(x0, x1, x2, x3);
        }
      }
    }

    // ---- the recurrence: rank-1 update of the thread's 4 x 8 tile, then C . h ---------------
    auto token = [&](int i) {
      const float2 tc = sT[i];
      const DecayCoef2 cf2 = decay_pair(DecayCoef{tc.x, ACC ? 1.0f : 0.0f});
      const float4 dxv = *reinterpret_cast<const float4*>(sDX + i * kMhP + pl0);
      const float dxs[kMhTP] = {dxv.x, dxv.y, dxv.z, dxv.w};
      f2_t B2[kMhTN / 2], C2[kMhTN / 2];
#pragma unroll
      for (int q = 0; q < kMhTN / 2; q += 2) {
        const float4 vb = *reinterpret_cast<const float4*>(sBf + i * N + n0 + 2 * q);
        B2[q] = f2_pack(vb.x, vb.y);
        B2[q + 1] = f2_pack(vb.z, vb.w);
        if (!LOCAL) {
          const float4 vc = *reinterpret_cast<const float4*>(sCf + i * N + n0 + 2 * q);
          C2[q] = f2_pack(vc.x, vc.y);
          C2[q + 1] = f2_pack(vc.z, vc.w);
        }
      }
      float part[kMhTP];
#pragma unroll
      for (int c = 0; c < kMhTP; c++) {
        const f2_t dx2 = f2_pack(dxs[c], dxs[c]);
        f2_t acc = 0ull;
#pragma unroll
        for (int q = 0; q < kMhTN / 2; q++) {
          hs[c][q] = step2<ACC>(cf2, hs[c][q], f2_mul(dx2, B2[q]));
          if (!LOCAL) acc = f2_fma(C2[q], hs[c][q], acc);
        }
        part[c] = LOCAL ? 0.0f : f2_sum(acc);
      }
      if (LOCAL) {
        sumd += tc.y;
        return;
      }
      // sum over the 16 state groups (lane bits 0..3), transposed over bits 3 and 2: lane ends
      // with channel slot 2 (bit 3) + (bit 2) summed over all 128 states
      const bool u3 = lane & 8, u2 = lane & 4;
      const float s0 = u3 ? part[0] : part[2], s1 = u3 ? part[1] : part[3];
      const float k0 = u3 ? part[2] : part[0], k1 = u3 ? part[3] : part[1];
      const float w0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 8);
      const float w1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 8);
      float v = (u2 ? w1 : w0) + __shfl_xor_sync(0xffffffffu, u2 ? w0 : w1, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if ((lane & 3) == 0) sYP[i * kMhP + pl0 + (u3 ? 2 : 0) + (u2 ? 1 : 0)] = v;
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
      for (int idx = tid; idx < cnt * kMhP; idx += kMhThreads) {
        const int c = idx % kMhP;
        float yv = sYP[idx];
        if (p.D) yv = fmaf(__ldg(p.D + ch0 + c), mh_lds(sx + idx), yv);
        if (p.z) yv *= siluf_(mh_lds(sz + idx));
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
    if (tid == 0 && k + kMhStages < ntiles) issue(k + kMhStages);
  }
  if (want_y && tid == 0) tma_store_wait_all();

  float* dst = nullptr;
  if (LOCAL) {
    dst = a.hloc + (((long)b * a.S + s) * p.HP + ch0) * N;
    if (ng == 0)
      for (int c = 0; c < kMhTP; c++) a.sumdelta[((long)b * a.S + s) * p.HP + ch0 + pl0 + c] = sumd;
  } else if (s == a.S - 1 && a.state_out) {
    dst = a.state_out + ((long)b * p.HP + ch0) * N;
  }
  if (dst) {
#pragma unroll
    for (int c = 0; c < kMhTP; c++)
#pragma unroll
      for (int q = 0; q < kMhTN / 2; q++)
        f2_unpack(hs[c][q], dst[(pl0 + c) * N + n0 + 2 * q], dst[(pl0 + c) * N + n0 + 2 * q + 1]);
  }
}

// Composes the segments in order: start[s+1] = exp(A sum_delta[s]) start[s] + h_local[s].
__global__ void scan_fwd_heads_carry_kernel(const __grid_constant__ MhArgs a) {
  const ScanProblem& p = a.p;
  const long total = (long)p.ns * p.HP * p.N;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i % p.N);
    const long bc = i / p.N;
    const int ch = (int)(bc % p.HP), b = (int)(bc / p.HP);
    const float A2 = __ldg(p.A + ch / p.P) * kLog2e;
    const float* row = start_row(p, b);
    float hv = row ? __ldg(row + (long)ch * p.N + n) : 0.0f;
    for (int s = 0; s < a.S; s++) {
      const long si = ((long)b * a.S + s) * p.HP + ch;
      a.segstart[si * p.N + n] = hv;
      if (s + 1 < a.S) hv = fmaf(ex2(A2 * a.sumdelta[si]), hv, a.hloc[si * p.N + n]);
    }
  }
}

// Time segments: none when (sequence, head, 64-channel block) alone gives this many blocks per
// SM, else enough segments to reach it (each extra segment costs a local pass over its tokens).
constexpr long kMhTargetBlocksPerSM = 2;

struct MhPlan {
  bool ok;
  int S, seg_len, dt_box;
  size_t off_segstart, off_hloc, off_sumdelta, bytes;
};

bool al16(const void* q) { return ((uintptr_t)q & 15) == 0; }

MhPlan plan_heads(const ScanProblem& p, int num_sms) {
  MhPlan q{};
  const int io = p.io == SSM_BF16 ? 2 : 4;
  if (p.a_per_state || p.P % kMhP != 0 || p.N != kMhN || (p.H * io) % 16 != 0 ||
      p.chunk % kMhTile != 0)
    return q;
  q.dt_box = 16 / io;
  const long base = (long)p.ns * p.H * (p.P / kMhP);
  long S = base >= kMhTargetBlocksPerSM * num_sms
               ? 1 : (kMhTargetBlocksPerSM * num_sms + base - 1) / base;
  const long max_s = (p.L + kMinSegment - 1) / kMinSegment;
  if (S > max_s) S = max_s;
  if (S < 1) S = 1;
  int seg = (int)((p.L + S - 1) / S);
  seg = (seg + kMhTile - 1) / kMhTile * kMhTile;
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
  q.ok = al16(p.x) && al16(p.dt) && al16(p.B) && al16(p.C) && (!p.z || al16(p.z));
  return q;
}

template <typename IO>
cudaError_t launch_heads_t(MhArgs& a, size_t smem, cudaStream_t st) {
  auto km = scan_fwd_heads_kernel<IO, false>;
  auto kl = scan_fwd_heads_kernel<IO, true>;
  cudaError_t e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kl, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int bx = a.p.H * (a.p.P / kMhP);
  if (a.S > 1) {
    kl<<<dim3(bx, a.S - 1, a.p.ns), kMhThreads, smem, st>>>(a), count_launches(1);
    const long total = (long)a.p.ns * a.p.HP * a.p.N;
    scan_fwd_heads_carry_kernel<<<(int)((total + 255) / 256), 256, 0, st>>>(a), count_launches(1);
  }
  km<<<dim3(bx, a.S, a.p.ns), kMhThreads, smem, st>>>(a), count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t scan_fwd_heads_ws_bytes(const ScanProblem& p, int num_sms) {
  const MhPlan q = plan_heads(p, num_sms);
  return q.ok ? q.bytes : 0;
}

// Returns cudaErrorNotSupported (without launching anything) when this path does not apply.
cudaError_t launch_scan_fwd_heads(const ScanProblem& p, void* y, float* state_out, float* ckpt,
                                  void* ws, int num_sms, cudaStream_t st) {
  const MhPlan q = plan_heads(p, num_sms);
  if (!q.ok || (y && !al16(y)) || (ckpt && !al16(ckpt))) return cudaErrorNotSupported;
  const int io = p.io == SSM_BF16 ? 2 : 4;
  MhArgs a;
  memset(&a, 0, sizeof(a));
  a.p = p;
  a.S = q.S; a.seg_len = q.seg_len; a.dt_box = q.dt_box;
  a.state_out = state_out; a.ckpt = ckpt; a.has_y = y != nullptr;
  char* w = (char*)ws;
  if (q.S > 1) {
    a.segstart = (float*)(w + q.off_segstart);
    a.hloc = (float*)(w + q.off_hloc);
    a.sumdelta = (float*)(w + q.off_sumdelta);
  }
  const uint64_t C = p.HP, L = p.L, NSq = p.ns, GN = (uint64_t)p.G * p.N, H = p.H;
  bool ok = encode_tmap_3d(&a.mx, p.x, io, C, L, NSq, C, C * L, kMhP, kMhTile, 1) &&
            encode_tmap_3d(&a.mdt, p.dt, io, H, L, NSq, H, H * L, q.dt_box, kMhTile, 1) &&
            encode_tmap_3d(&a.mb, p.B, io, GN, L, NSq, GN, GN * L, kMhN, kMhTile, 1) &&
            encode_tmap_3d(&a.mc, p.C, io, GN, L, NSq, GN, GN * L, kMhN, kMhTile, 1);
  if (ok && p.z) ok = encode_tmap_3d(&a.mz, p.z, io, C, L, NSq, C, C * L, kMhP, kMhTile, 1);
  if (ok && y) ok = encode_tmap_3d(&a.my, y, io, C, L, NSq, C, C * L, kMhP, kMhTile, 1);
  if (!ok) return cudaErrorNotSupported;
  auto al = [](uint32_t v) { return (v + 127u) & ~127u; };
  const uint32_t tile = kMhTile * kMhP * io, row = kMhTile * kMhN * io, dtt = kMhTile * q.dt_box * io;
  a.off_x = 0;
  a.off_dt = al(tile);
  a.off_z = a.off_dt + al(dtt);
  a.off_b = a.off_z + (p.z ? al(tile) : 0);
  a.off_c = a.off_b + al(row);
  a.stage_stride = a.off_c + al(row);
  a.off_dx = kMhStages * a.stage_stride;
  a.off_t = a.off_dx + al(kMhTile * kMhP * 4);
  a.off_bf = a.off_t + al(kMhTile * 8);
  const uint32_t conv = io == 2 ? al(kMhTile * kMhN * 4) : 0;  // fp32 copies of bf16 B, C
  a.off_cf = a.off_bf + conv;
  a.off_yp = a.off_cf + conv;
  a.off_y = a.off_yp + al(kMhTile * kMhP * 4);
  a.y_stride = al(tile);
  a.off_bar = a.off_y + 2 * a.y_stride;
  const size_t smem = a.off_bar + 64;
  if (smem > 227u * 1024u) return cudaErrorNotSupported;
  a.bytes_local = tile + dtt + row;
  a.bytes_main = (1 + (p.z ? 1 : 0)) * tile + dtt + 2 * row;
  return io == 2 ? launch_heads_t<__nv_bfloat16>(a, smem, st) : launch_heads_t<float>(a, smem, st);
}

}  // namespace ssm

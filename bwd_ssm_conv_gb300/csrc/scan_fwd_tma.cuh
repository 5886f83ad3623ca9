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
// delta x -- and converts bf16 B and C rows to fp32 once, so the recurrence reads 4 states of
// B or C with one 16-byte shared load and no per-thread conversion.  The lanes of a channel
// finish C . h with a shuffle reduce-scatter over groups of tokens and each writes the y of
// one token, so no partial sums go through shared memory and no separate epilogue pass runs.
// With one A per channel the decay is one exponential per (token, channel) for all states.
// fp32 I/O uses the accurate decay form h <- h + (expm1(delta A) h + u) (scan_common.cuh).
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"
#include "tma.cuh"

#include <type_traits>

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
  // shared-memory layouts: [0] the main pass, [1] the local pass (no z, C, y: a smaller block)
  struct Layout {
    uint32_t off_x, off_dt, off_z, off_b, off_c, stage_stride;  // inside a stage
    uint32_t off_dd, off_bf, off_cf, off_par, off_y, y_stride, off_bar;
    uint32_t off_sxs;  // fused conv: [cb][odd pitch] fp32 sx columns of a tile
  } lay[2];
};

// Columns of sx a tile of the fused conv reads (TT tokens and the K-1 before the first) and
// the odd row pitch of their fp32 staging buffer (a warp reading 32 channels at one column
// then touches 32 different banks).
template <int CK>
__host__ __device__ constexpr int conv_cols() { return 16 + CK - 1; }
template <int CK>
__host__ __device__ constexpr int conv_pitch() { return conv_cols<CK>() | 1; }

// The TMA swizzle of the x, z and y tiles ([TT][cb], one tile row per token): the span of a
// tile row when that is 32, 64 or 128 bytes (as a log2 of 16-byte chunks), else none.  The
// epilogue's warp reads 4 token rows of 8 channels; unswizzled, rows 128 bytes apart share
// banks (2-way for bf16 rows of 32 channels, 4-way for fp32).
template <typename IO, int CB>
__host__ __device__ constexpr int fwd_tile_swizzle() {
  return CB * (int)sizeof(IO) == 32 ? 1 : CB * (int)sizeof(IO) == 64 ? 2
                                        : CB * (int)sizeof(IO) == 128 ? 3 : 0;
}

template <typename IO>
__device__ __forceinline__ float lds1(const IO* p) {
  if constexpr (sizeof(IO) == 4) return *reinterpret_cast<const float*>(p);
  else return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// Sum over the TPC lanes of a channel group of v[0..TPC-1] (one value per token of a group of
// TPC consecutive tokens), scattered: lane sg of the group ends with the total of token sg in
// v[0].  Recursive halving: at distance d the lane keeps the half of its range that its bit d
// selects and sends the other half to the partner, which keeps it.  TPC - 1 shuffles.
template <int TPC>
__device__ __forceinline__ float group_reduce_scatter(float (&v)[TPC], int sg) {
#pragma unroll
  for (int d = TPC / 2; d >= 1; d >>= 1) {
    const bool up = (sg & d) != 0;
#pragma unroll
    for (int j = 0; j < d; j++) {
      const float keep = up ? v[j + d] : v[j];
      const float send = up ? v[j] : v[j + d];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, d);
    }
  }
  return v[0];
}

// A block = THR threads = (THR / TPC) channels x N states, NS = N / TPC states per thread, one
// sequence, one time segment.  SCALAR_A: one A per channel (the head of head_dim 1).
//
// CK > 0 (the fused conv1d of width CK): x is not copied from memory but computed in the
// prepass from sx, x = act(sum_k sx[t+k] w[k] + bias), rounded to the io type as ssm_conv_fwd
// stores it, and written into the stage's x slot, so that everything after the prepass reads
// it as it would read a copied tile.  A tile's sx columns are loaded into registers one tile
// ahead with plain loads (a row of L + CK - 1 elements starts at any alignment, which TMA
// cannot copy) and stored to shared memory once the prepass has read the previous ones.
//
// Per tile: a prepass writes (delta, delta x) once per (token, channel) and, for bf16 I/O, B and
// C as fp32 rows (fp32 I/O reads the staged rows as they are).  The recurrence then runs over
// groups of TPC tokens; after each group the lanes of a channel reduce-scatter their partial
// C . h sums so that lane sg holds token sg's total and writes that token's
// y = (C . h + D x) silu(z) into the output tile itself.
//
// Registers: without the conv the compiler's own choice is kept (a minimum of 0 blocks per SM
// states none: under 64 for the d_state 16 layout, where a minimum of one block would let it
// spend 120 and the grid would no longer fit in one wave).  The fused conv's staging would take that
// layout past 64; its bound keeps the 8 blocks per SM that time segments aim for.  The 8 states
// x 2 threads layout, which bf16 takes when it needs time segments, would spend 124 (4 blocks
// per SM); a bound of 6 blocks (80 registers) measured 4 % faster on one 16384-token sequence
// of d_inner 2048, a bound of 8 (64 registers) 2 % slower.
template <int NS, int TPC, int CK>
constexpr int fwd_min_blocks() {
  return CK > 0 ? (int)kFwdTargetBlocksPerSM : (NS == 8 && TPC == 2 ? 6 : 0);
}

template <typename IO, int NS, int TPC, int THR, bool LOCAL, bool SCALAR_A, int CK>
__global__ void __launch_bounds__(THR, fwd_min_blocks<NS, TPC, CK>())
scan_fwd_tma_kernel(const __grid_constant__ FwdTmaArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;  // accurate decay form for fp32 I/O
  constexpr int TT = kFwdTile;
  constexpr int cb = THR / TPC;  // compile-time: index math is shifts
  static_assert(NS % 4 == 0, "states per thread come in groups of 4");
  static_assert(TT % TPC == 0, "token groups tile the staged tile");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // the swizzled tiles want 1024-byte alignment: the host adds 1024 bytes for this shift
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr int SWZ = fwd_tile_swizzle<IO, cb>();
  auto xi = [](int idx) { return swizzled_index<SWZ, (int)sizeof(IO)>(idx); };  // x, z, y tiles
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x;
  const int cl = tid / TPC, sg = tid - cl * TPC;
  const int ch0 = blockIdx.x * cb, ch = ch0 + cl;
  const int s = blockIdx.y, b = blockIdx.z;
  const int N = p.N, n0 = sg * NS;
  const int g = ch0 / (p.H / p.G);
  const int t_begin = s * a.seg_len, t_end = min(p.L, t_begin + a.seg_len);
  const int ntiles = (t_end - t_begin + TT - 1) / TT;
  const uint32_t bytes = LOCAL ? a.bytes_local : a.bytes_main;
  const bool want_y = !LOCAL && a.has_y;
  const FwdTmaArgs::Layout& Y = a.lay[LOCAL ? 1 : 0];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Y.off_bar);
  float2* sDD = reinterpret_cast<float2*>(smem + Y.off_dd);  // [TT][cb] (delta, delta x)
  float* sBf = reinterpret_cast<float*>(smem + Y.off_bf);     // [TT][N] B as fp32 (bf16 I/O)
  float* sCf = reinterpret_cast<float*>(smem + Y.off_cf);     // [TT][N] C as fp32 (bf16 I/O)
  float* sPar = reinterpret_cast<float*>(smem + Y.off_par);  // [cb] D, [cb] dt_bias

  if (tid == 0) {
    for (int i = 0; i < kFwdStages; i++) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  for (int c = tid; c < cb; c += THR) {
    sPar[c] = p.D ? __ldg(p.D + ch0 + c) : 0.0f;
    sPar[cb + c] = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + ch0 + c) : 0.0f;
    if constexpr (CK > 0) {  // conv bias, then weights [cb][CK]
      sPar[2 * cb + c] = p.conv_b ? __ldg(p.conv_b + ch0 + c) : 0.0f;
#pragma unroll
      for (int k = 0; k < CK; k++)
        sPar[3 * cb + c * CK + k] = __ldg(p.conv_w + (long)(ch0 + c) * CK + k);
    }
  }
  // ---- fused conv: a tile's sx columns, loaded into registers one tile ahead ---------------
  // Thread tid stages row tid / 4 of the block's cb = THR / 4 rows, columns tid % 4 + 4u.
  constexpr int SXW = CK > 0 ? conv_cols<CK>() : 1, SXP = CK > 0 ? conv_pitch<CK>() : 1;
  constexpr int SXU = (SXW + 3) / 4;  // staged elements per thread
  static_assert(CK == 0 || (cb * 4 == THR && TT == 16 && THR == 128), "fused conv layout");
  const long sx_row = (long)p.L + CK - 1;
  const int sx_r = tid >> 2, sx_q = tid & 3;
  const IO* sx_rowp = CK > 0 ? reinterpret_cast<const IO*>(p.sx) +
                                   ((long)b * p.HP + ch0 + sx_r) * sx_row + sx_q
                             : nullptr;
  float* sxs = reinterpret_cast<float*>(smem + Y.off_sxs);
  IO sxv[SXU];
  auto sx_load = [&](int t0) {
    const IO* q = sx_rowp + t0;
    if (t0 + SXW <= sx_row) {  // every column of the tile exists
#pragma unroll
      for (int u = 0; u < SXU; u++)
        if (SXW % 4 == 0 || 4 * u + sx_q < SXW) sxv[u] = q[4 * u];
    } else {
#pragma unroll
      for (int u = 0; u < SXU; u++)
        sxv[u] = (4 * u + sx_q < SXW && t0 + 4 * u + sx_q < sx_row) ? q[4 * u] : IO(0.0f);
    }
  };
  auto sx_store = [&]() {
#pragma unroll
    for (int u = 0; u < SXU; u++)
      if (SXW % 4 == 0 || 4 * u + sx_q < SXW)
        sxs[sx_r * SXP + 4 * u + sx_q] = static_cast<float>(sxv[u]);
  };
  if constexpr (CK > 0) {
    sx_load(t_begin);
    sx_store();
  }
  __syncthreads();
  auto issue = [&](int k) {  // tile k -> stage k % kFwdStages (thread 0 only)
    const int stg = k % kFwdStages;
    unsigned char* base = smem + stg * Y.stage_stride;
    const int t0 = t_begin + k * TT;
    mbar_expect_tx(&full[stg], bytes);
    if constexpr (CK == 0) tma_load_3d(base + Y.off_x, &a.mx, ch0, t0, b, &full[stg]);
    tma_load_3d(base + Y.off_dt, &a.mdt, ch0, t0, b, &full[stg]);
    tma_load_3d(base + Y.off_b, &a.mb, g * N, t0, b, &full[stg]);
    if (!LOCAL) {
      if (p.z) tma_load_3d(base + Y.off_z, &a.mz, ch0, t0, b, &full[stg]);
      tma_load_3d(base + Y.off_c, &a.mc, g * N, t0, b, &full[stg]);
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
  const float Dc = sPar[cl];
  float sumd = 0.0f;

  for (int k = 0; k < ntiles; k++) {
    const int stg = k % kFwdStages;
    if (want_y && tid == 0) tma_store_wait_read<1>();  // store k-2 has read its y buffer
    if constexpr (CK > 0)
      if (k + 1 < ntiles) sx_load(t_begin + (k + 1) * TT);  // lands while this tile runs
    const bool ok = mbar_wait(&full[stg], (uint32_t)(k / kFwdStages) & 1u);
    unsigned char* base = smem + stg * Y.stage_stride;
    const IO* sx = reinterpret_cast<const IO*>(base + Y.off_x);
    const IO* sdt = reinterpret_cast<const IO*>(base + Y.off_dt);
    const IO* sz = reinterpret_cast<const IO*>(base + Y.off_z);
    const int t0 = t_begin + k * TT;
    const int cnt = min(TT, t_end - t0);

    // ---- prepass (a tile that never arrived leaves stale but in-bounds shared memory); a
    // compile-time item count lets the items' shared loads be in flight together ------------
    static_assert(TT * cb % THR == 0, "prepass items per thread");
    if constexpr (CK == 0) {
#pragma unroll
      for (int u = 0; u < TT * cb / THR; u++) {
        const int idx = tid + u * THR;
        const int c = idx % cb;
        float dl = lds1(sdt + idx);
        if (p.softplus) dl = softplusf_(dl + sPar[cb + c]);
        sDD[idx] = make_float2(dl, dl * lds1(sx + xi(idx)));
      }
    } else {
      // the conv: warp w takes tokens 4w .. 4w+3 of channel `lane`, a sliding window over
      // its sx columns; x goes into the stage's x slot (rounded to the io type, as
      // ssm_conv_fwd stores it) for the epilogue
      const int c = tid & 31, i0 = (tid >> 5) * 4;
      float wk[CK], win[4 + CK - 1];
#pragma unroll
      for (int kk = 0; kk < CK; kk++) wk[kk] = sPar[3 * cb + c * CK + kk];
#pragma unroll
      for (int m = 0; m < 4 + CK - 1; m++) win[m] = sxs[c * SXP + i0 + m];
      const float cbias = sPar[2 * cb + c], dtb = sPar[cb + c];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int idx = (i0 + u) * cb + c;
        float dl = lds1(sdt + idx);
        if (p.softplus) dl = softplusf_(dl + dtb);
        float acc = cbias;
#pragma unroll
        for (int kk = 0; kk < CK; kk++) acc = fmaf(win[u + kk], wk[kk], acc);
        if (p.conv_silu) acc = siluf_(acc);
        const IO xr = static_cast<IO>(acc);
        const_cast<IO*>(sx)[xi(idx)] = xr;
        sDD[idx] = make_float2(dl, dl * static_cast<float>(xr));
      }
    }
    if constexpr (sizeof(IO) == 2) {
      const uint2* rb = reinterpret_cast<const uint2*>(base + Y.off_b);
      const uint2* rc = reinterpret_cast<const uint2*>(base + Y.off_c);
      for (int idx = tid; idx < TT * N / 4; idx += THR) {
        const uint2 vb = rb[idx];
        reinterpret_cast<float4*>(sBf)[idx] =
            make_float4(__uint_as_float(vb.x << 16), __uint_as_float(vb.x & 0xffff0000u),
                        __uint_as_float(vb.y << 16), __uint_as_float(vb.y & 0xffff0000u));
        if (!LOCAL) {
          const uint2 vc = rc[idx];
          reinterpret_cast<float4*>(sCf)[idx] =
              make_float4(__uint_as_float(vc.x << 16), __uint_as_float(vc.x & 0xffff0000u),
                          __uint_as_float(vc.y << 16), __uint_as_float(vc.y & 0xffff0000u));
        }
      }
    }
    if (__syncthreads_or(!ok)) {  // a tile never arrived: report, drain, leave
      if (tid == 0) {
        record_status(p.status, SSM_ERR_TIMEOUT);
        for (int j = k; j < ntiles && j < k + kFwdStages; j++)
          mbar_wait(&full[j % kFwdStages], (uint32_t)(j / kFwdStages) & 1u);
        tma_store_wait_all();
      }
      return;
    }
    const float* Bf = sizeof(IO) == 4 ? reinterpret_cast<const float*>(base + Y.off_b) : sBf;
    const float* Cf = sizeof(IO) == 4 ? reinterpret_cast<const float*>(base + Y.off_c) : sCf;
    // the next tile's sx columns: the prepass above has read these (barrier), and the next
    // prepass reads them after the barrier that ends this tile
    if constexpr (CK > 0)
      if (k + 1 < ntiles) sx_store();

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
    // the decay coefficients of one token (one per state pair, or one for all states)
    auto decays = [&](float dl, DecayCoef2 (&cf)[NS / 2]) {
      if constexpr (SCALAR_A) {
        const DecayCoef2 c = decay_pair(decay_coef<ACC>(dl, A2s));
#pragma unroll
        for (int q = 0; q < NS / 2; q++) cf[q] = c;
      } else {
        const f2_t dl2 = f2_pack(dl, dl);
#pragma unroll
        for (int q = 0; q < NS / 2; q++) cf[q] = decay2<ACC>(dl2, A2p[q]);
      }
    };
    // one token: advance the states with its decays; returns this thread's part of C . h
    auto token = [&](int i, float2 dd, const DecayCoef2 (&cf)[NS / 2]) -> float {
      const f2_t dx2 = f2_pack(dd.y, dd.y);
      f2_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
      for (int j = 0; j < NS; j += 4) {
        const float4 vb = *reinterpret_cast<const float4*>(Bf + i * N + n0 + j);
        const f2_t B2[2] = {f2_pack(vb.x, vb.y), f2_pack(vb.z, vb.w)};
        const int q = j / 2;
#pragma unroll
        for (int e = 0; e < 2; e++) hp[q + e] = step2<ACC>(cf[q + e], hp[q + e], f2_mul(dx2, B2[e]));
        if (!LOCAL) {
          const float4 vc = *reinterpret_cast<const float4*>(Cf + i * N + n0 + j);
          acc0 = f2_fma(f2_pack(vc.x, vc.y), hp[q], acc0);
          acc1 = f2_fma(f2_pack(vc.z, vc.w), hp[q + 1], acc1);
        }
      }
      if (LOCAL) {
        sumd += dd.x;
        return 0.0f;
      }
      return f2_sum(f2_add(acc0, acc1));
    };
    IO* sy = reinterpret_cast<IO*>(smem + Y.off_y + (k & 1) * Y.y_stride);
    // fp32 I/O with one A per state: the decays of a whole group (the long accurate expm1 form)
    // are computed before its state updates, which do not feed them, so their latency overlaps
    // the update chain (measured faster).  bf16 I/O makes them token by token: batched there,
    // the one-instruction SFU decays measured 45 % slower.  Large groups would not fit in
    // registers, and the one-A-per-channel form has a single decay per token.
    constexpr bool BATCH = ACC && !SCALAR_A && TPC * NS <= 32;
    // one group of TPC tokens; FULL: every token of the group is inside the sequence
    auto group = [&](int i0, auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
      float acc[TPC];
      if constexpr (BATCH) {
        float2 dd[TPC];
        DecayCoef2 cf[TPC][NS / 2];
#pragma unroll
        for (int u = 0; u < TPC; u++) {
          dd[u] = sDD[(i0 + u) * cb + cl];
          decays(dd[u].x, cf[u]);
        }
#pragma unroll
        for (int u = 0; u < TPC; u++)
          acc[u] = (FULL || i0 + u < cnt) ? token(i0 + u, dd[u], cf[u]) : 0.0f;
      } else {
#pragma unroll
        for (int u = 0; u < TPC; u++) {
          acc[u] = 0.0f;
          if (FULL || i0 + u < cnt) {
            const float2 dd = sDD[(i0 + u) * cb + cl];
            DecayCoef2 cf[NS / 2];
            decays(dd.x, cf);
            acc[u] = token(i0 + u, dd, cf);
          }
        }
      }
      if (LOCAL) return;
      const float tot = group_reduce_scatter<TPC>(acc, sg);
      if (want_y) {  // token i0 + sg of channel cl (rows past the sequence end are not stored)
        const int idx = xi((i0 + sg) * cb + cl);
        float yv = fmaf(Dc, lds1(sx + idx), tot);
        if (p.z) yv *= siluf_(lds1(sz + idx));
        if (p.check_finite && (FULL || i0 + sg < cnt) && !isfinite(yv))
          record_status(p.status, SSM_ERR_NONFINITE);
        if constexpr (sizeof(IO) == 4) sy[idx] = yv;
        else sy[idx] = __float2bfloat16_rn(yv);
      }
    };
    if (cnt == TT) {  // full tile: no per-token branch, so tokens can interleave
#pragma unroll
      for (int i0 = 0; i0 < TT; i0 += TPC) group(i0, std::true_type{});
    } else {
#pragma unroll
      for (int i0 = 0; i0 < TT; i0 += TPC) group(i0, std::false_type{});
    }
    if (want_y) fence_async_shared();
    __syncthreads();  // y tile complete; stage stg and the prepass buffers fully read
    if (tid == 0) {
      if (want_y) {
        tma_store_3d(&a.my, sy, ch0, t0, b);
        tma_store_commit();
      }
      if (k + kFwdStages < ntiles) issue(k + kFwdStages);
    }
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
    // segments 0 .. S-1, 8 at a time: their decays and local aggregates do not depend on hv,
    // so their loads go out together ahead of the composition
    constexpr int kBatch = 8;
    for (int s0 = 0; s0 < a.S; s0 += kBatch) {
      float dk[kBatch], lv[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; j++) {
        const int s = s0 + j;
        const long si = ((long)b * a.S + s) * p.HP + ch;
        dk[j] = s + 1 < a.S ? ex2(A2 * a.sumdelta[si]) : 0.0f;
        lv[j] = s + 1 < a.S ? a.hloc[si * p.N + n] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kBatch; j++) {
        const int s = s0 + j;
        if (s >= a.S) break;
        a.segstart[(((long)b * a.S + s) * p.HP + ch) * p.N + n] = hv;
        if (s + 1 < a.S) hv = fmaf(dk[j], hv, lv[j]);
      }
    }
  }
}

template <typename IO, int NS, int TPC, bool SCALAR_A, int THR, int CK>
cudaError_t launch_fwd_tma_t(FwdTmaArgs& a, size_t smem, size_t smem_loc, cudaStream_t st) {
  auto km = scan_fwd_tma_kernel<IO, NS, TPC, THR, false, SCALAR_A, CK>;
  auto kl = scan_fwd_tma_kernel<IO, NS, TPC, THR, true, SCALAR_A, CK>;
  cudaError_t e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kl, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_loc);
  if (e != cudaSuccess) return e;
  const int bx = a.p.HP / a.cb;
  if (a.S > 1) {
    kl<<<dim3(bx, a.S - 1, a.p.ns), THR, smem_loc, st>>>(a), count_launches(1);
    const long total = (long)a.p.ns * a.p.HP * a.p.N;
    scan_fwd_tma_carry_kernel<IO><<<(int)((total + 255) / 256), 256, 0, st>>>(a), count_launches(1);
  }
  km<<<dim3(bx, a.S, a.p.ns), THR, smem, st>>>(a), count_launches(1);
  return cudaGetLastError();
}

// The (states per thread, threads per channel, A form, block threads, fused conv width)
// combinations instantiated for each I/O type; X(NS, TPC, SCALAR_A, THR, CK).  The fused conv
// (CK > 0) comes with the layout d_state 16 takes (4 states x 4 threads per channel).
#define SSM_FWD_TMA_VARIANTS(X) \
  X(16, 1, false, 128, 0) X(8, 2, false, 128, 0) X(4, 4, false, 128, 0) X(16, 2, false, 128, 0) \
  X(8, 4, false, 128, 0) X(16, 4, false, 128, 0) X(16, 8, true, 128, 0) X(8, 4, true, 128, 0) \
  X(16, 4, true, 128, 0) X(4, 4, true, 128, 0) \
  X(4, 4, false, 128, 1) X(4, 4, false, 128, 2) X(4, 4, false, 128, 3) X(4, 4, false, 128, 4)

}  // namespace ssm

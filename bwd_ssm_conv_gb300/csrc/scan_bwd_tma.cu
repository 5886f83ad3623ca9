// scan_bwd_tma.cu -- TMA-staged backward scan for the Mamba-1 layout with d_state 16
// (head_dim 1, rows 16-byte aligned, checkpoint interval a multiple of 16).
//
// Same arithmetic and workspace outputs as the general kernels in scan_bwd.cu.  A block =
// 128 threads = 32 channels x 16 states (4 threads of 4 states per channel), one sequence,
// one (chain, chunk) unit at a time when persistent, else one time segment.  Inputs arrive as
// [16 tokens][32 channels] tiles (x, dt, z, dy) and [16 tokens][16] tiles (B, C) through a
// 2-stage ring filled by cp.async.bulk.tensor; dx, dz, ddt leave as TMA-stored tiles.  Per
// tile, work that depends only on (token, channel) -- delta, the gate, dy silu'(z),
// softplus' -- is done once by the whole block in a prepass, so the per-state loops carry only
// the recurrence (packed f32x2 arithmetic); the per-channel sums over states are added across
// lane pairs and go through shared memory to an epilogue that writes dx, dz and ddt, and the
// dB/dC sums over channels use a warp butterfly whose exchanges need no lane-dependent selects
// (each thread's states sit in registers in a lane-permuted order).  Four blocks fit an SM
// (at most 128 registers, about 54 KB of shared memory).
//
// Per chunk (last to first): level 1 walks the chunk's tiles forward from the checkpoint,
// saving each tile's start state in tensor memory; level 2 walks the tiles in reverse,
// recomputes the tile's 16 states into tensor memory and runs the adjoint over them in reverse,
// reading them back four tokens at a time and recomputing each token's decays.  The state
// history never leaves the SM.
#include <type_traits>

#include "scan_bwd.cuh"
#include "tma.cuh"
#include "tmem.cuh"

namespace ssm {

constexpr int kBwdStages = 2;
constexpr int kBwdTile = 16;                  // tokens per staged tile
constexpr int kCB = kScanThreads / 4;         // channels per block
constexpr int kWarps = kScanThreads / 32;
// Tensor memory of a block: 128 columns (a quarter of the SM's; shared memory keeps a block's
// SM to 4 blocks).  Per thread (lane), 4 columns per state record of its 4 states:
// columns [0, 64): the recomputed states of the current level-2 tile, record k = the state
// before token k; columns [64, 128): level 1's tile start states, record j = tile j of the chunk.
constexpr uint32_t kTmCols = 128;
constexpr uint32_t kTmHist = 0, kTmStart = 64;
constexpr int kTmChunkTiles = 16;             // tile starts that fit: chunks of <= 256 tokens

struct BwdTma {
  CUtensorMap mx, mdt, mz, mdy, mb, mc, mdx, mdz, mddt;
  uint32_t bytes_l1, bytes_l2, bytes_loc;
  uint32_t off_x, off_dt, off_z, off_dy, off_b, off_c, stage_stride;
  uint32_t off_p, off_spg, off_e, off_bf, off_cf, off_part, off_red, off_out, out_tile, out_stride;
  uint32_t off_par, off_acc, off_bar, smem;
  // the local-adjoint kernel's own, smaller layout: the same tile stages, then its (delta, gy)
  // records, C as fp32 rows, dt_bias and the barriers
  uint32_t loc_off_p, loc_off_cf, loc_off_par, loc_off_bar, loc_smem;
  // persistent mode: queue counter, per-unit ready flags, units, chains, chain stride; the
  // dB/dC reduction items that share the queue: per-(sequence, group, chunk) counts of finished
  // units, items per chunk, 32-token slices per chunk, and the queue's length (units + items)
  int* counter;
  int* flags;
  int units, chains, gx;
  int* done;
  int red_per_chunk, red_slices, queue_len;
  uint32_t flag_spin;  // polls of a unit flag before the wait gives up
};

constexpr uint32_t kFlagSpin = 1u << 22;
// Chunks (the last to finish) whose dB/dC reduction items wait for the end of the persistent
// queue.  On 16 x 2048 tokens x 1536 channels in chunks of 256: 1 -> 780 MB of DRAM traffic per
// call and 1.231 ms, 3 -> 822 MB and 1.227 ms, all 8 -> 1094 MB and 1.224 ms.
constexpr int kRedTail = 3;

// Waits (bounded) until another block has published *flag; gives up at once when any block has
// recorded an error in the status word, so that one failure cannot chain into long waits.
__device__ __forceinline__ bool wait_unit_flag(const int* flag, const int* status, uint32_t spin) {
  for (uint32_t i = 0; i < spin; i++) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v) return true;
    if (status && *reinterpret_cast<const volatile int*>(status)) return false;
    __nanosleep(64);
  }
  return false;
}
// Waits (bounded, as wait_unit_flag) until *count reaches `target`.
__device__ __forceinline__ bool wait_count(const int* count, int target, const int* status,
                                           uint32_t spin) {
  for (uint32_t i = 0; i < spin; i++) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
    if (v >= target) return true;
    if (status && *reinterpret_cast<const volatile int*>(status)) return false;
    __nanosleep(64);
  }
  return false;
}
__device__ __forceinline__ void publish_unit_flag(int* flag) {
  __threadfence();
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

int bwd_tma_tile(const ScanProblem& p, int chunk_b, int gc) {
  const int io = p.io == SSM_BF16 ? 2 : 4;
  if (p.P == 1 && p.a_per_state && p.N == 16 && (p.HP * io) % 16 == 0 && gc % kCB == 0 &&
      chunk_b % kBwdTile == 0 && chunk_b <= kTmChunkTiles * kBwdTile)
    return kBwdTile;
  return 0;
}
int bwd_tma_channels_per_block() { return kCB; }
int bwd_tma_queue_ints(const ScanProblem& p, int nch, long chains) {
  // queue counter, unit flags, per-(sequence, group, chunk) counts of finished units
  return (int)(1 + chains * nch + (long)p.ns * p.G * nch);
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

// B (and C) of a tile as fp32: the staged tile itself for fp32 I/O, else converted once.
template <typename IO>
__device__ __forceinline__ const float* tile_rows_f32(const unsigned char* stage_rows, float* conv,
                                                      int count) {
  if constexpr (sizeof(IO) == 4) {
    (void)conv; (void)count;
    return reinterpret_cast<const float*>(stage_rows);
  } else {
    const IO* src = reinterpret_cast<const IO*>(stage_rows);
    for (int idx = threadIdx.x; idx < count; idx += kScanThreads) conv[idx] = lds_f(src + idx);
    return conv;
  }
}

// Register slot j of a thread holds state n0 + (j ^ p), p = lane bits 3..4 (see the dB/dC sums
// below).  B and C of a tile are kept as fp32 in 4 copies, copy p holding within every group of 4
// states the order (j ^ p), so that each lane reads its slots with one 16-byte load.
// Consecutive copies lie kPermPadF floats (64 bytes) more than a copy apart.  A warp reads 4
// state groups from each of the 4 copies; unpadded (1024-byte copies) all four copies fall on
// the same banks, and a 16-byte read took 4 shared-memory wavefronts instead of 2.
constexpr int kPermPadF = 16;
template <typename IO>
__device__ __forceinline__ void tile_rows_perm(const unsigned char* stage_rows, float* dst, int count) {
  const IO* src = reinterpret_cast<const IO*>(stage_rows);
  for (int idx = threadIdx.x; idx < count; idx += kScanThreads) {
    const float v = lds_f(src + idx);
    const int base = idx & ~3, j = idx & 3;
#pragma unroll
    for (int pc = 0; pc < 4; pc++) dst[pc * (count + kPermPadF) + base + (j ^ pc)] = v;
  }
}

// A bf16 pair (one 32-bit word, low half first) as a packed fp32 pair; exact.
__device__ __forceinline__ f2_t bf2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// Four bf16 (two words) with their order permuted by j -> j ^ pc.
__device__ __forceinline__ uint2 perm4_bf16(uint2 v, int pc) {
  if (pc & 1) {
    v.x = __byte_perm(v.x, 0u, 0x1032);
    v.y = __byte_perm(v.y, 0u, 0x1032);
  }
  return (pc & 2) ? make_uint2(v.y, v.x) : v;
}
// bf16 I/O: B and C of a tile as [4 copies][TT][N/4] records of 8 bf16 (B of 4 states, then C
// of the same 4 states), copy pc in the order (j ^ pc), copies kPermPadF / 4 records apart
// beyond their size; C is left out on level-1 tiles.
__device__ __forceinline__ void tile_bc_perm_bf16(const unsigned char* rb, const unsigned char* rc,
                                                  uint4* dst, int groups, bool with_c) {
  const uint2* b2 = reinterpret_cast<const uint2*>(rb);
  const uint2* c2 = reinterpret_cast<const uint2*>(rc);
  for (int idx = threadIdx.x; idx < groups; idx += kScanThreads) {
    const uint2 vb = b2[idx], vc = with_c ? c2[idx] : make_uint2(0u, 0u);
#pragma unroll
    for (int pc = 0; pc < 4; pc++) {
      const uint2 pb = perm4_bf16(vb, pc), pcv = perm4_bf16(vc, pc);
      dst[pc * (groups + kPermPadF / 4) + idx] = make_uint4(pb.x, pb.y, pcv.x, pcv.y);
    }
  }
}

// Sums the dB and dC products of a token over the 8 channels of a warp (lane bits 2..4).  Slot j
// holds state n0 + (j ^ p) with p = lane bits 3..4, so at the exchanges over bit 4 (slots 2,3 go
// out, 0,1 stay) and bit 3 (slot 1 out, slot 0 stays) the partner always sends the states this lane
// keeps: no lane-dependent selects.  The last exchange (bit 2) is a plain sum.  Returns the totals
// (dB, dC) of state n0 + p, identical on the lane pair that differs in bit 2.
__device__ __forceinline__ f2_t reduce_bc_warp(f2_t dB01, f2_t dB23, f2_t dC01, f2_t dC23) {
  float b2, b3, c2, c3;
  f2_unpack(dB23, b2, b3);
  f2_unpack(dC23, c2, c3);
  const f2_t rb = f2_pack(__shfl_xor_sync(0xffffffffu, b2, 16), __shfl_xor_sync(0xffffffffu, b3, 16));
  const f2_t rc = f2_pack(__shfl_xor_sync(0xffffffffu, c2, 16), __shfl_xor_sync(0xffffffffu, c3, 16));
  float wb0, wb1, wc0, wc1;
  f2_unpack(f2_add(dB01, rb), wb0, wb1);
  f2_unpack(f2_add(dC01, rc), wc0, wc1);
  const f2_t x = f2_add(f2_pack(wb0, wc0), f2_pack(__shfl_xor_sync(0xffffffffu, wb1, 8),
                                                   __shfl_xor_sync(0xffffffffu, wc1, 8)));
  float xb, xc;
  f2_unpack(x, xb, xc);
  return f2_add(x, f2_pack(__shfl_xor_sync(0xffffffffu, xb, 4), __shfl_xor_sync(0xffffffffu, xc, 4)));
}

// One dB/dC reduction item of the persistent path: for (sequence, group) bg = j / slices and the
// 32-token slice j % slices of chunk cc, the sums over the a.bpg channel blocks' partials, taken
// in block order 0..bpg-1 (the separate reduction kernel's order, so the results are the same
// bits), once that chunk's units of bg are all counted.  A wait that gives up records a time-out
// and returns.  Entered and left by the whole block.
template <typename IO>
__device__ __forceinline__ void reduce_item(const BwdTma& m, const BwdArgs& a, int cc, int j) {
  constexpr int N = 16, R2 = 2 * N;
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x;
  const int bg = j / m.red_slices, slice = j - bg * m.red_slices;
  const int rb = bg / p.G, rg = bg - rb * p.G;
  bool ok = true;
  if (tid == 0) {
    ok = wait_count(m.done + (long)bg * a.nch_b + cc, a.bpg, p.status, m.flag_spin);
    if (!ok) record_status(p.status, SSM_ERR_TIMEOUT);
  }
  if (__syncthreads_or(!ok)) return;
  const int t0 = cc * a.chunk_b + slice * 32;
  const int tn = min(32, min(p.L, (cc + 1) * a.chunk_b) - t0);
  // 8 threads share a token's partial line (one per block index k: 2N floats, 128 bytes), each
  // holding 4 entries (one 16-byte load per line); thread tid sums the quad q of tokens
  // i0 + kRowsQ u.  kK block indices x kOutQ tokens of loads are in flight together, and each sum
  // still adds its partials in the order k = 0, 1, ... (paired adds round as scalar ones).
  constexpr int kQ = R2 / 4, kRowsQ = kScanThreads / kQ, kOutQ = 32 / kRowsQ, kK = 4;
  static_assert(kScanThreads % kQ == 0 && 32 % kRowsQ == 0 && 32 % kQ == 0, "item layout");
  const int q = tid % kQ, i0 = tid / kQ;
  const long tg0 = ((long)rb * p.L + t0 + i0) * p.G + rg;
  const long tstep = (long)kRowsQ * p.G;                 // token rows between passes
  const float* line0 = a.part_bc + tg0 * a.bpg * R2;     // token i0's line of block 0
  const long sstep = tstep * a.bpg * R2;
  f2_t v[kOutQ][2];
#pragma unroll
  for (int u = 0; u < kOutQ; u++) v[u][0] = v[u][1] = 0ull;
  auto acc = [&](int u, float4 t) {
    v[u][0] = f2_add(v[u][0], f2_pack(t.x, t.y));
    v[u][1] = f2_add(v[u][1], f2_pack(t.z, t.w));
  };
  auto ld4 = [&](int u, int k) {
    return __ldcg(reinterpret_cast<const float4*>(line0 + u * sstep + (long)k * R2) + q);
  };
  int k = 0;
  for (; k + kK <= a.bpg; k += kK) {
    float4 t[kK][kOutQ];
#pragma unroll
    for (int d = 0; d < kK; d++)
#pragma unroll
      for (int u = 0; u < kOutQ; u++)
        t[d][u] = i0 + u * kRowsQ < tn ? ld4(u, k + d) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int d = 0; d < kK; d++)
#pragma unroll
      for (int u = 0; u < kOutQ; u++) acc(u, t[d][u]);
  }
  for (; k < a.bpg; k++) {
#pragma unroll
    for (int u = 0; u < kOutQ; u++)
      if (i0 + u * kRowsQ < tn) acc(u, ld4(u, k));
  }
  const int r = 4 * q;  // entries r .. r+3: dB (r < N) or dC, never both
  IO* dst = (IO*)(r < N ? a.g.d_B : a.g.d_C) + (r < N ? r : r - N);
#pragma unroll
  for (int u = 0; u < kOutQ; u++) {
    if (i0 + u * kRowsQ >= tn) continue;
    float e[4];
    f2_unpack(v[u][0], e[0], e[1]);
    f2_unpack(v[u][1], e[2], e[3]);
    IO* o = dst + (tg0 + u * tstep) * N;
#pragma unroll
    for (int c = 0; c < 4; c++) sts_f(o + c, e[c]);
  }
  // the lines are read (their values are in the sums; a line's 8 readers share a warp): drop
  // them from L2 unwritten
  __syncwarp();
  for (int kk = q; kk < a.bpg; kk += kQ) {
#pragma unroll
    for (int u = 0; u < kOutQ; u++)
      if (i0 + u * kRowsQ < tn) discard_l2_line(line0 + u * sstep + (long)kk * R2);
  }
  __syncthreads();
}

// PERSIST: the grid is a set of resident blocks that take work from one queue.  The queue holds
// the (chain, chunk) units chunk-major, last chunk first (unit u: chain u % chains, chunk
// nch - 1 - u / chains), so the unit that produces a chunk's end adjoint (the start adjoint of
// the chunk after it) was taken `chains` positions earlier by a running block.  The dB/dC
// reduction items of chunk c follow the units of chunk c - 1, whose units were all taken before
// them, except for the last kRedTail chunks to finish (c < kRedTail), whose items close the
// queue (nch = 8, kRedTail = 3):
//   [units 7] [units 6][items 7] [units 5][items 6] ... [units 2][items 3] [units 1] [units 0]
//   [items 2] [items 1] [items 0]
// Every wait is on work taken earlier.  A chunk's partials are summed about one chunk of units
// after they are stored, while they are still in L2; the items at the end run in the slots
// that the last units leave idle, on partials recent enough to be in L2 too.  Otherwise one
// block = one (sequence, channel block, segment) of whole chunks, as given by the grid.
template <typename IO, bool PERSIST>
__global__ void __launch_bounds__(kScanThreads, kBwdTmaBlocksPerSM)
scan_bwd_tma_kernel(const __grid_constant__ BwdTma m, const BwdArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;
  constexpr int TT = kBwdTile, CB = kCB, N = 16;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int sUnit;
  const ScanProblem& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pm = (lane >> 3) & 3;  // slot j holds state n0 + (j ^ pm)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + m.off_bar);
  // L2 policy of the tiles read or written for the last time: first out
  const uint64_t pol_first = l2_policy_evict_first();
  __shared__ uint32_t sTmem;
  if (tid == 0) {
    for (int i = 0; i < kBwdStages; i++) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(&sTmem, kTmCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tm = sTmem + ((uint32_t)(warp * 32) << 16);  // this warp's lanes
  // ring cursors run on across units: a stage's barrier phase follows the count of its uses
  int issued = 0, qpos = 0, n_l2 = 0;
  // the units; every way out (done, or a wait that gave up) returns from here to the release
  // of the tensor memory below
  [&]() {
  for (int round = 0;; round++) {
  int ux, s, b;
  if constexpr (PERSIST) {
    if (tid == 0) {
      const bool failed = p.status && *reinterpret_cast<const volatile int*>(p.status) != 0;
      sUnit = failed ? m.queue_len : atomicAdd(m.counter, 1);
    }
    __syncthreads();
    const int q = sUnit;
    if (q >= m.queue_len) break;
    // position -> unit u, or reduction item j of chunk cc
    int u = q, cc = -1, j = 0;
    if (q >= m.chains) {
      const int C = m.chains, R = m.red_per_chunk, per = C + R;
      const int k1 = max(0, a.nch_b - kRedTail);  // unit blocks 1..k1 carry items
      const int q2 = q - C;
      if (q2 < k1 * per) {
        const int k = 1 + q2 / per, r = q2 - (k - 1) * per;
        if (r < C) u = k * C + r;
        else { cc = a.nch_b - k; j = r - C; }
      } else {
        const int q3 = q2 - k1 * per, nb = a.nch_b - 1 - k1;
        if (q3 < nb * C) {
          u = (1 + k1) * C + q3;
        } else {
          const int q4 = q3 - nb * C, t = min(kRedTail, a.nch_b);
          cc = t - 1 - q4 / R;
          j = q4 - (t - 1 - cc) * R;
        }
      }
    }
    if (cc >= 0) {
      reduce_item<IO>(m, a, cc, j);
      continue;
    }
    const int chain = u % m.chains;
    s = a.nch_b - 1 - u / m.chains;
    ux = chain % m.gx;
    b = chain / m.gx;
  } else {
    if (round > 0) break;
    ux = blockIdx.x; s = blockIdx.y; b = blockIdx.z;
  }
  const Lane l = lane_of(a, ux);
  const int cl = l.cl, ch = l.ch, ch0 = ch - cl, n0 = l.n0;
  float2* sD2 = reinterpret_cast<float2*>(smem + m.off_p);       // [TT][CB] (delta, delta x)
  float* sGy = reinterpret_cast<float*>(smem + m.off_spg);       // [TT][CB] gy = dy silu(z)
  float4* sE = reinterpret_cast<float4*>(smem + m.off_e);        // [TT][CB] (x, gy, dyg, softplus')
  // per-channel state sums of lane pairs (4 lanes hold a channel's 16 states): [TT][threads / 2]
  float* sPB = reinterpret_cast<float*>(smem + m.off_part);      // sum_n dh B
  float* sPA = sPB + TT * kScanThreads / 2;                       // sum_n A w
  float* sPY = sPA + TT * kScanThreads / 2;                       // sum_n C h
  float* red = reinterpret_cast<float*>(smem + m.off_red);       // [TT][warps][2N]
  float* sPar = reinterpret_cast<float*>(smem + m.off_par);      // D[CB], dt_bias[CB]
  float* sAcc = reinterpret_cast<float*>(smem + m.off_acc);      // [warps][CB][2]
  const int c_first = s * a.seg_chunks;
  const int c_last = min(a.nch_b, c_first + a.seg_chunks) - 1;

  // Tile schedule: per chunk (last to first), level-1 tiles ascending then level-2 tiles
  // descending.  Thread 0 (producer) and every thread (consumer) walk it with own cursors.
  struct Pos { int ck, lvl, j, nt; };
  auto ntiles = [&](int ck) {
    const int t0 = ck * a.chunk_b, t1 = min(p.L, t0 + a.chunk_b);
    return (t1 - t0 + TT - 1) / TT;
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

  for (int c = tid; c < CB; c += kScanThreads) {
    sPar[c] = p.D ? __ldg(p.D + ch0 + c) : 0.0f;
    sPar[CB + c] = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + ch0 + c) : 0.0f;
  }
  __syncthreads();
  Pos pp = first();
  auto issue = [&]() {  // thread 0 only
    const int stg = issued % kBwdStages;
    unsigned char* base = smem + stg * m.stage_stride;
    const int t0 = pp.ck * a.chunk_b + pp.j * TT;
    if (pp.lvl == 0) {
      mbar_expect_tx(&full[stg], m.bytes_l1);
      tma_load_3d(base + m.off_x, &m.mx, ch0, t0, b, &full[stg]);
      tma_load_3d(base + m.off_dt, &m.mdt, ch0, t0, b, &full[stg]);
      tma_load_3d(base + m.off_b, &m.mb, l.g * N, t0, b, &full[stg]);
    } else {  // the last read of these tiles: first out of L2, ahead of the state scratch
      mbar_expect_tx(&full[stg], m.bytes_l2);
      tma_load_3d_hint(base + m.off_x, &m.mx, ch0, t0, b, &full[stg], pol_first);
      tma_load_3d_hint(base + m.off_dt, &m.mdt, ch0, t0, b, &full[stg], pol_first);
      tma_load_3d_hint(base + m.off_dy, &m.mdy, ch0, t0, b, &full[stg], pol_first);
      if (p.z) tma_load_3d_hint(base + m.off_z, &m.mz, ch0, t0, b, &full[stg], pol_first);
      tma_load_3d_hint(base + m.off_b, &m.mb, l.g * N, t0, b, &full[stg], pol_first);
      tma_load_3d_hint(base + m.off_c, &m.mc, l.g * N, t0, b, &full[stg], pol_first);
    }
    issued++;
    advance(pp);
  };
  if (tid == 0)
    for (int k = 0; k < kBwdStages && pp.ck >= c_first; k++) issue();

  f2_t A2p[2], Anp[2], carry2[2], dA2[2] = {0ull, 0ull}, hp[2] = {0ull, 0ull};
  {
    const long si = ((long)b * a.S + s) * p.HP + ch;
    // the adjoint at the segment's end: given by the caller for the last one; else from the
    // carry pass, or (persistent) from the unit of the next chunk once it has published it
    const bool from_next = a.S > 1 && s < a.S - 1;
    if (PERSIST && from_next) {
      bool ok = true;
      if (tid == 0) {
        ok = wait_unit_flag(m.flags + (long)(b * m.gx + ux) * a.nch_b + s, p.status, m.flag_spin);
        if (!ok) record_status(p.status, SSM_ERR_TIMEOUT);
      }
      // the flag's outcome reaches every thread; on a give-up the block waits (bounded) for its
      // tile copies in flight and skips the rest of its work
      if (__syncthreads_or(!ok)) {
        if (tid == 0) {
          for (int j = qpos; j < issued; j++)
            mbar_wait(&full[j % kBwdStages], (uint32_t)(j / kBwdStages) & 1u);
          tma_store_wait_all();
        }
        return;
      }
    }
    float cv[4], av[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int n = n0 + (j ^ pm);
      if (from_next) cv[j] = __ldcg(a.segend + si * N + n);
      else cv[j] = a.g.d_state_out ? __ldg(a.g.d_state_out + ((long)b * p.HP + ch) * N + n) : 0.0f;
      av[j] = __ldg(p.A + (long)ch * N + n);
    }
#pragma unroll
    for (int q = 0; q < 2; q++) {
      const float a0 = av[2 * q], a1 = av[2 * q + 1];
      Anp[q] = f2_pack(a0, a1);
      A2p[q] = f2_pack(a0 * kLog2e, a1 * kLog2e);
      carry2[q] = f2_pack(cv[2 * q], cv[2 * q + 1]);
    }
  }
  float dD_acc = 0.0f, dtb_acc = 0.0f;  // of channel tid % CB, over this thread's epilogue items

  for (Pos cs = first(); cs.ck >= c_first; advance(cs), qpos++) {
    const int stg = qpos % kBwdStages;
    // a tile that never arrived leaves stale but in-bounds shared memory: the prepass reads it,
    // and the barrier after the prepass sends the whole block out
    const bool ok = mbar_wait(&full[stg], (uint32_t)(qpos / kBwdStages) & 1u);
    const unsigned char* base = smem + stg * m.stage_stride;
    const IO* sx = reinterpret_cast<const IO*>(base + m.off_x);
    const IO* sdt = reinterpret_cast<const IO*>(base + m.off_dt);
    const IO* sz = reinterpret_cast<const IO*>(base + m.off_z);
    const IO* sdy = reinterpret_cast<const IO*>(base + m.off_dy);
    const int t0c = cs.ck * a.chunk_b, t1c = min(p.L, t0c + a.chunk_b);
    const int t0 = t0c + cs.j * TT;
    const int cnt = min(TT, t1c - t0);

    // ---- prepass, once per (token, channel); a compile-time item count lets the items'
    // shared loads be in flight together -------------------------------------------------------
    static_assert(TT * CB % kScanThreads == 0, "prepass items per thread");
#pragma unroll
    for (int u = 0; u < TT * CB / kScanThreads; u++) {
      const int idx = tid + u * kScanThreads;
      const int c = idx % CB;
      const float raw = lds_f(sdt + idx);
      const float pre = raw + sPar[CB + c];
      const float dl = p.softplus ? softplusf_(pre) : raw;
      const float xv = lds_f(sx + idx);
      if (cs.lvl == 1) {
        const float dyv = lds_f(sdy + idx);
        float gy = dyv, dyg = 0.0f;
        if (p.z) {
          const float zv = lds_f(sz + idx), sgm = sigmoidf_(zv);
          gy = dyv * zv * sgm;
          dyg = dyv * sgm * (1.0f + zv * (1.0f - sgm));
        }
        sGy[idx] = gy;
        sE[idx] = make_float4(xv, gy, dyg, p.softplus ? softplus_gradf_(pre) : 1.0f);
      }
      sD2[idx] = make_float2(dl, dl * xv);
    }
    // B and C: this lane's permuted copy (bf16 records for bf16 I/O, fp32 rows otherwise)
    const uint4* sBCq = reinterpret_cast<const uint4*>(smem + m.off_bf) + pm * (TT * N / 4 + kPermPadF / 4);
    const float* sBf = reinterpret_cast<const float*>(smem + m.off_bf) + pm * (TT * N + kPermPadF);
    const float* sCf = reinterpret_cast<const float*>(smem + m.off_cf) + pm * (TT * N + kPermPadF);
    if constexpr (sizeof(IO) == 2) {
      tile_bc_perm_bf16(base + m.off_b, base + m.off_c, reinterpret_cast<uint4*>(smem + m.off_bf),
                        TT * N / 4, cs.lvl == 1);
    } else {
      tile_rows_perm<IO>(base + m.off_b, reinterpret_cast<float*>(smem + m.off_bf), TT * N);
      if (cs.lvl == 1) tile_rows_perm<IO>(base + m.off_c, reinterpret_cast<float*>(smem + m.off_cf), TT * N);
    }
    auto ld_b = [&](int i, f2_t (&B2)[2]) {
      if constexpr (sizeof(IO) == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(sBCq + i * (N / 4) + (n0 >> 2));
        B2[0] = bf2_to_f2(v.x);
        B2[1] = bf2_to_f2(v.y);
      } else {
        const float4 v = *reinterpret_cast<const float4*>(sBf + i * N + n0);
        B2[0] = f2_pack(v.x, v.y);
        B2[1] = f2_pack(v.z, v.w);
      }
    };
    auto ld_bc = [&](int i, f2_t (&B2)[2], f2_t (&C2)[2]) {
      if constexpr (sizeof(IO) == 2) {
        const uint4 v = sBCq[i * (N / 4) + (n0 >> 2)];
        B2[0] = bf2_to_f2(v.x);
        B2[1] = bf2_to_f2(v.y);
        C2[0] = bf2_to_f2(v.z);
        C2[1] = bf2_to_f2(v.w);
      } else {
        const float4 v = *reinterpret_cast<const float4*>(sBf + i * N + n0);
        const float4 w = *reinterpret_cast<const float4*>(sCf + i * N + n0);
        B2[0] = f2_pack(v.x, v.y);
        B2[1] = f2_pack(v.z, v.w);
        C2[0] = f2_pack(w.x, w.y);
        C2[1] = f2_pack(w.z, w.w);
      }
    };
    if (__syncthreads_or(!ok)) {  // the prepass and the B/C copies are complete
      if (tid == 0) {
        record_status(p.status, SSM_ERR_TIMEOUT);
        for (int j = qpos; j < issued; j++) mbar_wait(&full[j % kBwdStages], (uint32_t)(j / kBwdStages) & 1u);
        tma_store_wait_all();
      }
      return;
    }

    if (cs.lvl == 0) {
      // ---- level 1: walk the tile forward from its start state, which goes to tensor memory
      if (cs.j == 0) {
        const float* src = a.ckpt + (((long)b * a.nch_b + cs.ck) * p.HP + ch) * N + n0;
        hp[0] = f2_pack(src[0 ^ pm], src[1 ^ pm]);
        hp[1] = f2_pack(src[2 ^ pm], src[3 ^ pm]);
      }
      {
        float h0, h1, h2, h3;
        f2_unpack(hp[0], h0, h1);
        f2_unpack(hp[1], h2, h3);
        tmem_st4(tm + kTmStart + 4 * cs.j, h0, h1, h2, h3);
      }
      auto token = [&](int i) {
        const float2 d2 = sD2[i * CB + cl];
        const f2_t dl2 = f2_pack(d2.x, d2.x), dx2 = f2_pack(d2.y, d2.y);
        f2_t B2[2];
        ld_b(i, B2);
        hp[0] = step2<ACC>(decay2<ACC, true>(dl2, A2p[0]), hp[0], f2_mul(dx2, B2[0]));
        hp[1] = step2<ACC>(decay2<ACC, true>(dl2, A2p[1]), hp[1], f2_mul(dx2, B2[1]));
      };
      if (cnt == TT) {  // full tile: no per-token branch, so tokens can interleave
#pragma unroll
        for (int i = 0; i < TT; i++) token(i);
      } else {
#pragma unroll
        for (int i = 0; i < TT; i++)
          if (i < cnt) token(i);
      }
      __syncthreads();  // stage fully read
      if (tid == 0 && pp.ck >= c_first) issue();
      continue;
    }

    // ---- level 2: recompute the tile's states into tensor memory, then the adjoint in reverse
    tmem_wait_st();  // the tile start states of level 1 have landed
    f2_t hcur[2];
    {
      float v[4];
      tmem_ld4(tm + kTmStart + 4 * cs.j, v);
      hcur[0] = f2_pack(v[0], v[1]);
      hcur[1] = f2_pack(v[2], v[3]);
    }
    // One token of the adjoint: hcur = the state after token i, hprev = the state before it;
    // the decays are recomputed (a second copy of the history would not fit tensor memory).
    auto adjoint = [&](int i, const f2_t (&hcur)[2], const f2_t (&hprev)[2]) {
        const float2 d2 = sD2[i * CB + cl];
        const float gyv = sGy[i * CB + cl];
        const f2_t dl2 = f2_pack(d2.x, d2.x), gy2 = f2_pack(gyv, gyv);
        const f2_t dlx2 = f2_pack(d2.y, d2.y);
        f2_t B2[2], C2[2];
        ld_bc(i, B2, C2);
        f2_t sB2 = 0ull, sAw2 = 0ull, yp2 = 0ull, dB2[2], dC2[2];
#pragma unroll
        for (int q = 0; q < 2; q++) {
          const f2_t dh2 = f2_fma(gy2, C2[q], carry2[q]);
          dC2[q] = f2_mul(gy2, hcur[q]);
          sB2 = f2_fma(dh2, B2[q], sB2);
          dB2[q] = f2_mul(dh2, dlx2);
          const f2_t cn2 = apply2<ACC>(decay2<ACC, true>(dl2, A2p[q]), dh2);
          const f2_t w2 = f2_mul(cn2, hprev[q]);
          sAw2 = f2_fma(Anp[q], w2, sAw2);
          dA2[q] = f2_fma(dl2, w2, dA2[q]);
          yp2 = f2_fma(C2[q], hcur[q], yp2);
          carry2[q] = cn2;
        }
        {  // sum the lane pair (states n0 .. n0+3 and the neighbour's 4), one store per sum
          float vb = f2_sum(sB2), va = f2_sum(sAw2), vy = f2_sum(yp2);
          vb += __shfl_xor_sync(0xffffffffu, vb, 1);
          va += __shfl_xor_sync(0xffffffffu, va, 1);
          vy += __shfl_xor_sync(0xffffffffu, vy, 1);
          const int q = i * (kScanThreads / 2) + (tid >> 1);
          if (tid & 1) {
            sPY[q] = vy;
          } else {
            sPB[q] = vb;
            sPA[q] = va;
          }
        }
        float tb, tc;
        f2_unpack(reduce_bc_warp(dB2[0], dB2[1], dC2[0], dC2[1]), tb, tc);
        const int hi = (lane >> 2) & 1;  // of the lane pair: 0 writes dB, 1 writes dC
        red[(i * kWarps + warp) * 2 * N + hi * N + n0 + pm] = hi ? tc : tb;
    };
    // FULL (all TT tokens present) drops the per-token branches
    auto level2 = [&](auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
      // records 4g .. 4g+3 (the states before tokens 4g .. 4g+3) go out in one store; one
      // group at a time (unrolled, the groups' registers would overlap)
#pragma unroll 1
      for (int g = 0; g < TT / 4; g++) {
        if (!FULL && 4 * g >= cnt) break;
        float rec[16];
#pragma unroll
        for (int u = 0; u < 4; u++) {
          f2_unpack(hcur[0], rec[4 * u], rec[4 * u + 1]);
          f2_unpack(hcur[1], rec[4 * u + 2], rec[4 * u + 3]);
          const int i = 4 * g + u;
          if (FULL || i < cnt) {
            const float2 d2 = sD2[i * CB + cl];
            const f2_t dl2 = f2_pack(d2.x, d2.x), dx2 = f2_pack(d2.y, d2.y);
            f2_t B2[2];
            ld_b(i, B2);
            hcur[0] = step2<ACC>(decay2<ACC, true>(dl2, A2p[0]), hcur[0], f2_mul(dx2, B2[0]));
            hcur[1] = step2<ACC>(decay2<ACC, true>(dl2, A2p[1]), hcur[1], f2_mul(dx2, B2[1]));
          }
        }
        tmem_st16(tm + kTmHist + 16 * g, rec);
      }
      tmem_wait_st();
      // hcur: the state after the tile's last token
#pragma unroll 1
      for (int g = TT / 4 - 1; g >= 0; g--) {
        if (!FULL && 4 * g >= cnt) continue;
        float rec[16];
        tmem_ld16(tm + kTmHist + 16 * g, rec);
#pragma unroll
        for (int u = 3; u >= 0; u--) {
          const int i = 4 * g + u;
          if (FULL || i < cnt) {  // uniform over the block
            const f2_t hprev[2] = {f2_pack(rec[4 * u], rec[4 * u + 1]),
                                   f2_pack(rec[4 * u + 2], rec[4 * u + 3])};
            adjoint(i, hcur, hprev);
            hcur[0] = hprev[0];
            hcur[1] = hprev[1];
          }
        }
      }
    };
    if (cnt == TT) level2(std::true_type{});
    else level2(std::false_type{});
    if (tid == 0) tma_store_wait_read<0>();  // the previous tile's stores have read `out`
    __syncthreads();  // sPart and red complete; `out` free

    // ---- epilogue, once per (token, channel): dx, dz, ddt; dD and d dt_bias partials --------
    IO* out = reinterpret_cast<IO*>(smem + m.off_out);
    IO* odx = out;
    IO* odz = reinterpret_cast<IO*>(reinterpret_cast<unsigned char*>(out) + m.out_tile);
    IO* oddt = reinterpret_cast<IO*>(reinterpret_cast<unsigned char*>(out) + 2 * m.out_tile);
    auto epi = [&](int idx) {
      const int i = idx / CB, c = idx - i * CB;  // c == tid % CB for every item of this thread
      const int pi = i * (kScanThreads / 2) + c * 2;  // the 2 lane pairs of channel c
      const float2 vb = *reinterpret_cast<const float2*>(sPB + pi);
      const float2 va = *reinterpret_cast<const float2*>(sPA + pi);
      const float2 vy = *reinterpret_cast<const float2*>(sPY + pi);
      const float sBt = vb.x + vb.y;
      const float sAwt = va.x + va.y;
      const float ypt = vy.x + vy.y;
      const float4 e4 = sE[idx];                  // (x, gy, dyg, softplus')
      const float dl = sD2[idx].x;
      const float D = sPar[c];
      const float ddl = fmaf(e4.x, sBt, sAwt);
      const float ddt = p.softplus ? ddl * e4.w : ddl;
      const float dxv = fmaf(e4.y, D, dl * sBt), dzv = e4.z * fmaf(D, e4.x, ypt);
      if (p.check_finite && !(isfinite(dxv) && isfinite(dzv) && isfinite(ddt)))
        record_status(p.status, SSM_ERR_NONFINITE);
      sts_f(odx + idx, dxv);
      sts_f(odz + idx, dzv);
      sts_f(oddt + idx, ddt);
      dD_acc = fmaf(e4.y, e4.x, dD_acc);
      dtb_acc += ddt;
    };
    // dB and dC of the tile's tokens: this block's sum over its warps, one partial per block
    auto red_item = [&](int idx) {
      const int i = idx / (2 * N), r = idx - i * 2 * N;
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; w++) v += red[(i * kWarps + w) * 2 * N + r];
      const long tok = (long)b * p.L + t0 + i;
      float* dst = a.part_bc + ((tok * p.G + l.g) * a.bpg + l.blk) * 2 * N + r;
      if constexpr (PERSIST) *dst = v;  // summed from L2 by a reduction item a chunk later
      else st_global_hint(dst, v, pol_first);
    };
    if (cnt == TT) {  // full tile: a compile-time item count, so the items interleave
#pragma unroll
      for (int u = 0; u < TT * CB / kScanThreads; u++) epi(tid + u * kScanThreads);
#pragma unroll
      for (int u = 0; u < TT * 2 * N / kScanThreads; u++) red_item(tid + u * kScanThreads);
    } else {
      for (int idx = tid; idx < cnt * CB; idx += kScanThreads) epi(idx);
      for (int idx = tid; idx < cnt * 2 * N; idx += kScanThreads) red_item(idx);
    }
    fence_async_shared();
    __syncthreads();  // out tiles complete; stage fully read
    if (tid == 0) {
      tma_store_3d_hint(&m.mdx, odx, ch0, t0, b, pol_first);
      if (p.z && a.g.d_z) tma_store_3d_hint(&m.mdz, odz, ch0, t0, b, pol_first);
      tma_store_3d_hint(&m.mddt, oddt, ch0, t0, b, pol_first);
      tma_store_commit();
      if (pp.ck >= c_first) issue();
    }
    n_l2++;
  }
  if (tid == 0) tma_store_wait_all();

  const long si = ((long)b * a.S + s) * p.HP + ch;
#pragma unroll
  for (int q = 0; q < 2; q++) {
    const int n_lo = n0 + ((2 * q) ^ pm), n_hi = n0 + ((2 * q + 1) ^ pm);
    f2_unpack(dA2[q], a.dA_part[si * N + n_lo], a.dA_part[si * N + n_hi]);
    if (s == 0)
      f2_unpack(carry2[q], a.dh0[((long)b * p.HP + ch) * N + n_lo],
                a.dh0[((long)b * p.HP + ch) * N + n_hi]);
  }
  sAcc[(warp * CB + (tid % CB)) * 2] = dD_acc;
  sAcc[(warp * CB + (tid % CB)) * 2 + 1] = dtb_acc;
  __syncthreads();
  if (tid < CB) {
    float vD = 0.0f, vT = 0.0f;
    for (int w = 0; w < kWarps; w++) {
      vD += sAcc[(w * CB + tid) * 2];
      vT += sAcc[(w * CB + tid) * 2 + 1];
    }
    const long sc = ((long)b * a.S + s) * p.HP + ch0 + tid;
    a.dD_part[sc] = vD;
    a.dtb_part[sc] = vT;
  }
  if (PERSIST && s > 0) {  // this chunk's start adjoint ends chunk s - 1: hand it over
    const long se = ((long)b * a.S + s - 1) * p.HP + ch;
#pragma unroll
    for (int q = 0; q < 2; q++)
      f2_unpack(carry2[q], a.segend[se * N + n0 + ((2 * q) ^ pm)],
                a.segend[se * N + n0 + ((2 * q + 1) ^ pm)]);
    __syncthreads();
    if (tid == 0) publish_unit_flag(m.flags + (long)(b * m.gx + ux) * a.nch_b + s - 1);
  }
  if constexpr (PERSIST) {  // the unit's dB/dC partials are all stored: count it
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(m.done + ((long)b * p.G + l.g) * a.nch_b + s, 1);
    }
  }
  }  // units
  }();
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(sTmem, kTmCols);
}

// Local adjoint of segments 1..S-1 (zero adjoint at the segment end), tiles in reverse.
template <typename IO>
__global__ void __launch_bounds__(kScanThreads)
scan_bwd_tma_local_kernel(const __grid_constant__ BwdTma m, const BwdArgs a) {
  constexpr bool ACC = sizeof(IO) == 4;
  constexpr int TT = kBwdTile, CB = kCB, N = 16;
  extern __shared__ __align__(128) unsigned char smem[];
  const ScanProblem& p = a.p;
  const Lane l = lane_of(a);
  const int tid = threadIdx.x;
  const int cl = l.cl, ch = l.ch, ch0 = ch - cl, n0 = l.n0;
  const int s = blockIdx.y + 1, b = blockIdx.z;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + m.loc_off_bar);
  float2* sP = reinterpret_cast<float2*>(smem + m.loc_off_p);  // [TT][CB] (delta, gy)
  float* sPar = reinterpret_cast<float*>(smem + m.loc_off_par);
  const int t_begin = s * a.seg_chunks * a.chunk_b;
  const int t_end = min(p.L, t_begin + a.seg_chunks * a.chunk_b);
  const int nt = (t_end - t_begin + TT - 1) / TT;

  if (tid == 0) {
    for (int i = 0; i < kBwdStages; i++) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  for (int c = tid; c < CB; c += kScanThreads)
    sPar[CB + c] = (p.softplus && p.dt_bias) ? __ldg(p.dt_bias + ch0 + c) : 0.0f;
  __syncthreads();
  auto issue = [&](int k) {  // tile nt-1-k (reverse order) -> stage k % stages
    const int stg = k % kBwdStages;
    unsigned char* base = smem + stg * m.stage_stride;
    const int t0 = t_begin + (nt - 1 - k) * TT;
    mbar_expect_tx(&full[stg], m.bytes_loc);
    tma_load_3d(base + m.off_dt, &m.mdt, ch0, t0, b, &full[stg]);
    tma_load_3d(base + m.off_dy, &m.mdy, ch0, t0, b, &full[stg]);
    if (p.z) tma_load_3d(base + m.off_z, &m.mz, ch0, t0, b, &full[stg]);
    tma_load_3d(base + m.off_c, &m.mc, l.g * N, t0, b, &full[stg]);
  };
  if (tid == 0)
    for (int k = 0; k < kBwdStages && k < nt; k++) issue(k);

  f2_t A2p[2], c2[2] = {0ull, 0ull};
#pragma unroll
  for (int q = 0; q < 2; q++)
    A2p[q] = f2_pack(__ldg(p.A + (long)ch * N + n0 + 2 * q) * kLog2e,
                     __ldg(p.A + (long)ch * N + n0 + 2 * q + 1) * kLog2e);
  float sumd = 0.0f;
  for (int k = 0; k < nt; k++) {
    const int stg = k % kBwdStages;
    const bool ok = mbar_wait(&full[stg], (uint32_t)(k / kBwdStages) & 1u);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        record_status(p.status, SSM_ERR_TIMEOUT);
        for (int j = k; j < nt && j < k + kBwdStages; j++)
          mbar_wait(&full[j % kBwdStages], (uint32_t)(j / kBwdStages) & 1u);
      }
      return;
    }
    const unsigned char* base = smem + stg * m.stage_stride;
    const IO* sdt = reinterpret_cast<const IO*>(base + m.off_dt);
    const IO* sz = reinterpret_cast<const IO*>(base + m.off_z);
    const IO* sdy = reinterpret_cast<const IO*>(base + m.off_dy);
    const int t0 = t_begin + (nt - 1 - k) * TT;
    const int cnt = min(TT, t_end - t0);
    for (int idx = tid; idx < TT * CB; idx += kScanThreads) {
      const int c = idx % CB;
      const float raw = lds_f(sdt + idx);
      const float dl = p.softplus ? softplusf_(raw + sPar[CB + c]) : raw;
      float gy = lds_f(sdy + idx);
      if (p.z) gy *= siluf_(lds_f(sz + idx));
      sP[idx] = make_float2(dl, gy);
    }
    const float* sCf = tile_rows_f32<IO>(base + m.off_c, reinterpret_cast<float*>(smem + m.loc_off_cf), TT * N);
    __syncthreads();
#pragma unroll
    for (int r = TT - 1; r >= 0; r--) {
      if (r < cnt) {
        const float2 p4 = sP[r * CB + cl];
        const f2_t dl2 = f2_pack(p4.x, p4.x), gy2 = f2_pack(p4.y, p4.y);
        const float4 cv = *reinterpret_cast<const float4*>(sCf + r * N + n0);
        c2[0] = apply2<ACC>(decay2<ACC, true>(dl2, A2p[0]), f2_fma(gy2, f2_pack(cv.x, cv.y), c2[0]));
        c2[1] = apply2<ACC>(decay2<ACC, true>(dl2, A2p[1]), f2_fma(gy2, f2_pack(cv.z, cv.w), c2[1]));
        sumd += p4.x;
      }
    }
    __syncthreads();
    if (tid == 0 && k + kBwdStages < nt) issue(k + kBwdStages);
  }
  const long si = ((long)b * a.S + s) * p.HP + ch;
#pragma unroll
  for (int q = 0; q < 2; q++)
    f2_unpack(c2[q], a.dhloc[si * N + n0 + 2 * q], a.dhloc[si * N + n0 + 2 * q + 1]);
  if (l.sg == 0) a.sumd[si] = sumd;
}

// ---- host --------------------------------------------------------------------------------
static bool al16(const void* v) { return ((uintptr_t)v & 15) == 0; }

static bool setup_bwd_tma(const BwdArgs& a, const BwdPlan& q, char* w, BwdTma* m) {
  const ScanProblem& p = a.p;
  const ScanGrads& g = a.g;
  if (!q.tma_tt) return false;
  if (!al16(p.x) || !al16(p.dt) || !al16(p.B) || !al16(p.C) || !al16(g.dy) || !al16(g.d_x) ||
      !al16(g.d_dt) || (p.z && !al16(p.z)) || (g.d_z && !al16(g.d_z)))
    return false;
  const int io = p.io == SSM_BF16 ? 2 : 4;
  const int TT = kBwdTile, cb = kCB;
  const uint64_t C = p.HP, L = p.L, NSq = p.ns, GN = (uint64_t)p.G * p.N;
  memset(m, 0, sizeof(*m));
  bool ok = encode_tmap_3d(&m->mx, p.x, io, C, L, NSq, C, C * L, cb, TT, 1) &&
            encode_tmap_3d(&m->mdt, p.dt, io, C, L, NSq, C, C * L, cb, TT, 1) &&
            encode_tmap_3d(&m->mdy, g.dy, io, C, L, NSq, C, C * L, cb, TT, 1) &&
            encode_tmap_3d(&m->mb, p.B, io, GN, L, NSq, GN, GN * L, p.N, TT, 1) &&
            encode_tmap_3d(&m->mc, p.C, io, GN, L, NSq, GN, GN * L, p.N, TT, 1) &&
            encode_tmap_3d(&m->mdx, g.d_x, io, C, L, NSq, C, C * L, cb, TT, 1) &&
            encode_tmap_3d(&m->mddt, g.d_dt, io, C, L, NSq, C, C * L, cb, TT, 1);
  if (ok && p.z) ok = encode_tmap_3d(&m->mz, p.z, io, C, L, NSq, C, C * L, cb, TT, 1);
  if (ok && g.d_z) ok = encode_tmap_3d(&m->mdz, g.d_z, io, C, L, NSq, C, C * L, cb, TT, 1);
  if (!ok) return false;
  auto al = [](uint32_t v) { return (v + 127u) & ~127u; };
  const uint32_t tile = (uint32_t)(TT * cb * io), row = (uint32_t)(TT * p.N * io);
  m->off_x = 0;
  m->off_dt = al(tile);
  m->off_z = m->off_dt + al(tile);
  m->off_dy = m->off_z + al(tile);
  m->off_b = m->off_dy + al(tile);
  m->off_c = m->off_b + al(row);
  m->stage_stride = m->off_c + al(row);
  uint32_t off = kBwdStages * m->stage_stride;
  auto take = [&](uint32_t bytes) { uint32_t o = off; off = al(off + bytes); return o; };
  m->off_p = take(TT * cb * 8);
  m->off_spg = take(TT * cb * 4);
  m->off_e = take(TT * cb * 16);
  // B, C in 4 permuted copies: bf16 records (B and C together) or fp32 rows; off_cf also holds
  // the local kernel's fp32 C rows
  m->off_bf = take(4 * (TT * p.N + kPermPadF) * 4);
  m->off_cf = take(io == 2 ? TT * p.N * 4 : 4 * (TT * p.N + kPermPadF) * 4);
  m->off_part = take(3 * TT * (kScanThreads / 2) * 4);
  m->off_red = take(TT * kWarps * 2 * p.N * 4);
  m->out_tile = al(tile);
  m->out_stride = 3 * m->out_tile;
  m->off_out = take(m->out_stride);
  m->off_par = take(2 * cb * 4);
  m->off_acc = take(kWarps * cb * 2 * 4);
  m->off_bar = take(64);
  m->smem = off;
  off = kBwdStages * m->stage_stride;
  m->loc_off_p = take(TT * cb * 8);
  m->loc_off_cf = take(TT * p.N * 4);
  m->loc_off_par = take(2 * cb * 4);
  m->loc_off_bar = take(64);
  m->loc_smem = off;
  m->bytes_l1 = 2 * tile + row;
  m->bytes_l2 = (3 + (p.z ? 1 : 0)) * tile + 2 * row;
  m->bytes_loc = (2 + (p.z ? 1 : 0)) * tile + row;
  m->flag_spin = (p.debug_flags & kDebugNoWait) ? 0u : kFlagSpin;
  return true;
}

bool bwd_tma_ready(const BwdArgs& a, const BwdPlan& q) {
  BwdTma m;
  return setup_bwd_tma(a, q, nullptr, &m);
}

// Zeroes the persistent path's queue counter and unit flags (the workspace holds anything).
__global__ void bwd_queue_reset_kernel(int* q, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) q[i] = 0;
}

// Blocks of a main kernel resident on an SM, from its registers and shared memory, capped at
// the 512 / kTmCols that share the SM's tensor memory (a block beyond that would wait in the
// allocation until one ends).  The runtime's occupancy query counts one block per SM for a
// kernel that allocates tensor memory, whatever it takes.
static int resident_blocks(const void* fn, size_t dyn_smem) {
  cudaFuncAttributes fa;
  int dev = 0, regs_sm = 0, smem_sm = 0, reserved = 0;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
    return 0;
  const int warps = kScanThreads / 32;
  const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp in 256s
  const int by_regs = regs_sm / (warp_regs * warps);
  const size_t block_smem = fa.sharedSizeBytes + dyn_smem + (size_t)reserved;
  const int by_smem = (int)((size_t)smem_sm / block_smem);
  int n = by_regs < by_smem ? by_regs : by_smem;
  if (n > (int)(512u / kTmCols)) n = (int)(512u / kTmCols);
  return n;
}

template <typename IO, bool PERSIST>
static cudaError_t launch_main_t(BwdTma& m, const BwdArgs& a, const BwdPlan& q, int num_sms,
                                 cudaStream_t st) {
  const ScanProblem& p = a.p;
  auto k = scan_bwd_tma_kernel<IO, PERSIST>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m.smem);
  if (e != cudaSuccess) return e;
  const int per_sm = resident_blocks(reinterpret_cast<const void*>(k), m.smem);
  if (per_sm < 1) return cudaErrorNotSupported;
  if (!PERSIST) {
    k<<<dim3(p.G * a.bpg, a.S, p.ns), kScanThreads, m.smem, st>>>(m, a), count_launches(1);
    return cudaGetLastError();
  }
  m.gx = p.G * a.bpg;
  m.chains = m.gx * p.ns;
  m.units = m.chains * a.nch_b;
  m.done = m.flags + m.units;
  m.red_slices = (a.chunk_b + 31) / 32;
  m.red_per_chunk = p.ns * p.G * m.red_slices;
  m.queue_len = m.units + a.nch_b * m.red_per_chunk;
  const int nq = bwd_tma_queue_ints(p, a.nch_b, m.chains);
  const long slots = (long)per_sm * num_sms;
  const int grid = (int)(slots < m.units ? slots : m.units);
  bwd_queue_reset_kernel<<<(nq + 255) / 256, 256, 0, st>>>(m.counter, nq), count_launches(1);
  k<<<grid, kScanThreads, m.smem, st>>>(m, a), count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_bwd_tma_main(const BwdArgs& a, const BwdPlan& q, char* ws, cudaStream_t st) {
  BwdTma m;
  if (!setup_bwd_tma(a, q, ws, &m)) return cudaErrorNotSupported;
  int dev = 0, num_sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (q.persist) {
    m.counter = reinterpret_cast<int*>(ws + q.off_queue);
    m.flags = m.counter + 1;
    return a.p.io == SSM_BF16 ? launch_main_t<__nv_bfloat16, true>(m, a, q, num_sms, st)
                              : launch_main_t<float, true>(m, a, q, num_sms, st);
  }
  return a.p.io == SSM_BF16 ? launch_main_t<__nv_bfloat16, false>(m, a, q, num_sms, st)
                            : launch_main_t<float, false>(m, a, q, num_sms, st);
}

cudaError_t launch_bwd_tma_local(const BwdArgs& a, const BwdPlan& q, char* ws, cudaStream_t st) {
  BwdTma m;
  if (!setup_bwd_tma(a, q, ws, &m)) return cudaErrorNotSupported;
  const ScanProblem& p = a.p;
  dim3 grid(p.G * a.bpg, a.S - 1, p.ns);
  cudaError_t e;
  if (p.io == SSM_BF16) {
    auto k = scan_bwd_tma_local_kernel<__nv_bfloat16>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m.loc_smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kScanThreads, m.loc_smem, st>>>(m, a), count_launches(1);
  } else {
    auto k = scan_bwd_tma_local_kernel<float>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)m.loc_smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kScanThreads, m.loc_smem, st>>>(m, a), count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace ssm

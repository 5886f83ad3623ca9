// scan_fwd_tma.cu -- host side of the TMA forward scan (kernels in scan_fwd_tma.cuh): the
// plan, the tensor maps, the shared-memory layout and the dispatch over instantiated shapes.
// bf16 instances are compiled here, fp32 ones in scan_fwd_tma_f32.cu.
#include "scan_fwd_tma.cuh"

namespace ssm {

#define SSM_EXTERN_F32(NS, TPC, SA, THR, CK) \
  extern template cudaError_t launch_fwd_tma_t<float, NS, TPC, SA, THR, CK>(FwdTmaArgs&, size_t, size_t, cudaStream_t);
SSM_FWD_TMA_VARIANTS(SSM_EXTERN_F32)
#undef SSM_EXTERN_F32

static bool instantiated(int ns, int tpc, bool scalar_a, int ck, int thr = 128) {
#define SSM_MATCH(NS, TPC, SA, THR, CK) \
  if (ns == NS && tpc == TPC && scalar_a == SA && thr == THR && ck == CK) return true;
  SSM_FWD_TMA_VARIANTS(SSM_MATCH)
#undef SSM_MATCH
  return false;
}

struct FwdTmaPlan {
  bool ok;
  int ns_state, tpc, thr, cb, tt, S, seg_len;
  size_t off_segstart, off_hloc, off_sumdelta, bytes;
};

static bool aligned16(const void* q) { return ((uintptr_t)q & 15) == 0; }

static FwdTmaPlan plan_fwd_tma(const ScanProblem& p, int num_sms) {
  FwdTmaPlan q{};
  const int io = p.io == SSM_BF16 ? 2 : 4;
  const bool sa = !p.a_per_state;
  // head_dim > 1 (the Mamba-2 form) stays on the general kernels: here every channel of a head
  // would re-read the head's B/C records from shared memory, which measured slower.
  if (p.P != 1 || p.N % 4 != 0 || p.N > 256 || (p.N * io) % 16 != 0 || (p.HP * io) % 16 != 0 ||
      p.chunk % kFwdTile != 0)
    return q;
  // the fused conv prelude comes with its own instances
  const int ck = p.sx ? p.d_conv : 0;
  if (p.sx && (ck < 1 || ck > 4)) return q;
  // largest states-per-thread that still gives four blocks per SM without time segments
  // (the recurrence is latency-bound: more warps per SM beat fewer instructions per state;
  // two states per thread, eight threads per channel, measured slower on both of d_inner 1536
  // x 16 sequences and d_inner 2048 x 1 sequence).  When none does, time segments make up the
  // blocks, and for bf16 I/O 8 states per thread (fewer shuffles per token, twice the
  // segments) beat 4: d_inner 2048 x one 16384-token sequence 0.321 -> 0.310 ms.  Not for
  // fp32, whose batched accurate decays then cost more (d_inner 512 x 8 x 1024: 0.093 ->
  // 0.103 ms); with 16 states per thread both lose (0.376 ms on the former).
  // a layout applies when it is instantiated and its channel block (128 threads / threads per
  // channel) tiles a group's channels and the rows
  auto fits = [&](int cand) {
    if (cand > p.N || p.N % cand != 0 || !instantiated(cand, p.N / cand, sa, ck)) return false;
    const int cb = kScanThreads / (p.N / cand);
    return (p.H / p.G) % cb == 0 && p.HP % cb == 0 && cb * io >= 16;
  };
  int ns = 0;
  bool fills = false;
  for (int cand = 16; cand >= 4; cand >>= 1) {
    if (!fits(cand)) continue;
    ns = cand;
    const int cb = kScanThreads / (p.N / cand);
    if ((long)p.ns * ((p.HP + cb - 1) / cb) >= 4L * num_sms) { fills = true; break; }
  }
  if (!fills && io == 2 && ns < 8 && fits(8)) ns = 8;
  if (ns == 0) return q;
  q.ns_state = ns;
  q.tpc = p.N / ns;
  q.thr = kScanThreads;
  q.cb = q.thr / q.tpc;
  if ((p.H / p.G) % q.cb != 0 || p.HP % q.cb != 0 || q.cb * io < 16) return q;
  q.tt = kFwdTile;
  // counted in 128-thread block equivalents, whatever the block size
  const long base = (long)p.ns * (p.HP / q.cb) * q.thr / kScanThreads;
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
  q.ok = (p.sx ? (uintptr_t)p.sx % io == 0 : aligned16(p.x)) && aligned16(p.dt) &&
         aligned16(p.B) && aligned16(p.C) && (!p.z || aligned16(p.z));
  return q;
}

size_t scan_fwd_tma_ws_bytes(const ScanProblem& p, int num_sms) {
  const FwdTmaPlan q = plan_fwd_tma(p, num_sms);
  return q.ok ? q.bytes : 0;
}

// Returns cudaErrorNotSupported (without launching anything) when the fast path does not
// apply to this problem; the caller then uses the general kernels.
cudaError_t launch_scan_fwd_tma(const ScanProblem& p, void* y, float* state_out, float* ckpt,
                                void* ws, int num_sms, cudaStream_t st) {
  const FwdTmaPlan q = plan_fwd_tma(p, num_sms);
  if (!q.ok || (y && !aligned16(y)) || (ckpt && !aligned16(ckpt))) return cudaErrorNotSupported;
  if (!p.sx && !p.x) return cudaErrorNotSupported;  // no tensor map over a missing input
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
  const int ck = p.sx ? p.d_conv : 0;  // the fused conv computes x: no tensor map for it
  // the x, z and y tiles are swizzled whenever a tile row (cb channels) is 32, 64 or 128 bytes,
  // the rule the kernel's fwd_tile_swizzle applies to the same cb
  const int rowb = q.cb * io, swz = (rowb == 32 || rowb == 64 || rowb == 128) ? rowb : 0;
  bool ok = (ck > 0 || encode_tmap_3d(&a.mx, p.x, io, C, L, NSq, C, C * L, q.cb, q.tt, 1, swz)) &&
            encode_tmap_3d(&a.mdt, p.dt, io, C, L, NSq, C, C * L, q.cb, q.tt, 1) &&
            encode_tmap_3d(&a.mb, p.B, io, GN, L, NSq, GN, GN * L, p.N, q.tt, 1) &&
            encode_tmap_3d(&a.mc, p.C, io, GN, L, NSq, GN, GN * L, p.N, q.tt, 1);
  if (ok && p.z) ok = encode_tmap_3d(&a.mz, p.z, io, C, L, NSq, C, C * L, q.cb, q.tt, 1, swz);
  if (ok && y) ok = encode_tmap_3d(&a.my, y, io, C, L, NSq, C, C * L, q.cb, q.tt, 1, swz);
  if (!ok) return cudaErrorNotSupported;
  const uint32_t tile = (uint32_t)(q.tt * q.cb * io), row = (uint32_t)(q.tt * p.N * io);
  // every buffer 128-byte aligned; the swizzled x, z, y tiles (and so the stages) 1024-byte
  // aligned, from a base the kernel aligns to 1024 bytes
  auto al = [](uint32_t v) { return (v + 127u) & ~127u; };
  auto alk = [](uint32_t v) { return (v + 1023u) & ~1023u; };
  FwdTmaArgs::Layout& M = a.lay[0];
  M.off_x = 0;
  M.off_dt = al(tile);
  M.off_z = alk(M.off_dt + al(tile));
  M.off_b = M.off_z + (p.z ? al(tile) : 0);
  M.off_c = M.off_b + al(row);
  M.stage_stride = alk(M.off_c + al(row));
  M.off_dd = kFwdStages * M.stage_stride;                       // float2 (delta, delta x)
  // B and C of a tile as fp32 rows (bf16 I/O only; fp32 I/O reads the staged rows)
  const uint32_t frow = io == 2 ? al((uint32_t)(q.tt * p.N * 4)) : 0u;
  M.off_bf = M.off_dd + al((uint32_t)(q.tt * q.cb * 8));
  M.off_cf = M.off_bf + frow;
  M.off_par = M.off_cf + frow;
  // D, dt_bias; with the fused conv also the conv bias and weights
  const uint32_t par = al((uint32_t)((2 + (ck ? 1 + ck : 0)) * q.cb * 4));
  M.off_y = alk(M.off_par + par);
  M.y_stride = alk(tile);
  M.off_sxs = M.off_y + 2 * M.y_stride;
  const uint32_t pitch = (uint32_t)((q.tt + ck - 1) | 1);
  const uint32_t sxs = ck > 0 ? al((uint32_t)(q.cb * pitch * 4)) : 0u;
  M.off_bar = M.off_sxs + sxs;
  const size_t smem = M.off_bar + 64 + 1024;  // + the kernel's alignment of its base
  if (smem > 227u * 1024u) return cudaErrorNotSupported;
  // the local pass reads no z or C and writes no y: stages of x, dt and B, then its records
  // (about two thirds of the main layout, so more blocks fit on an SM)
  FwdTmaArgs::Layout& Lo = a.lay[1];
  Lo = M;
  Lo.off_b = alk(Lo.off_dt + al(tile));
  Lo.off_z = Lo.off_c = Lo.off_b;  // not read
  Lo.stage_stride = alk(Lo.off_b + al(row));
  Lo.off_dd = kFwdStages * Lo.stage_stride;
  Lo.off_bf = Lo.off_dd + al((uint32_t)(q.tt * q.cb * 8));
  Lo.off_cf = Lo.off_bf;           // not written
  Lo.off_par = Lo.off_bf + frow;
  Lo.off_y = Lo.off_par;           // not written
  Lo.y_stride = 0;
  Lo.off_sxs = alk(Lo.off_par + par);
  Lo.off_bar = Lo.off_sxs + sxs;
  const size_t smem_loc = Lo.off_bar + 64 + 1024;
  // the fused conv's x slot in a stage is written by the prepass, not copied
  a.bytes_local = (ck > 0 ? 1 : 2) * tile + row;
  a.bytes_main = ((ck > 0 ? 1 : 2) + (p.z ? 1 : 0)) * tile + 2 * row;
  const bool sa = !p.a_per_state;
#define SSM_DISPATCH(NS, TPC, SA, THR, CK)                                              \
  if (q.ns_state == NS && q.tpc == TPC && sa == SA && q.thr == THR && ck == CK)         \
    return io == 2 ? launch_fwd_tma_t<__nv_bfloat16, NS, TPC, SA, THR, CK>(a, smem, smem_loc, st) \
                   : launch_fwd_tma_t<float, NS, TPC, SA, THR, CK>(a, smem, smem_loc, st);
  SSM_FWD_TMA_VARIANTS(SSM_DISPATCH)
#undef SSM_DISPATCH
  return cudaErrorNotSupported;
}

}  // namespace ssm

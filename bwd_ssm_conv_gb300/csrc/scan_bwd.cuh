// scan_bwd.cuh -- declarations shared by the backward scan's translation units.
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "scan_common.cuh"

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

// dB, dC of every (token, group) = the sum over the blocks' partials, in block order.
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

struct Lane {
  int tpc, cl, sg, g, blk, cig, ch, h, n0;
  bool valid;
};

// bx: the block's index along (group, channel block), blockIdx.x unless a persistent block
// takes its work units from a queue.
__device__ __forceinline__ Lane lane_of(const BwdArgs& a, int bx) {
  Lane l;
  l.tpc = a.tpc;
  l.cl = threadIdx.x / l.tpc;
  l.sg = threadIdx.x - l.cl * l.tpc;
  l.g = bx / a.bpg;
  l.blk = bx - l.g * a.bpg;
  l.cig = l.blk * (kScanThreads / l.tpc) + l.cl;
  l.valid = l.cig < a.gc;
  l.ch = l.g * a.gc + (l.valid ? l.cig : 0);
  l.h = l.ch / a.p.P;
  l.n0 = l.sg * kBwdNS;
  return l;
}
__device__ __forceinline__ Lane lane_of(const BwdArgs& a) { return lane_of(a, blockIdx.x); }

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

struct BwdPlan {
  int tpc, gc, bpg, chunk_b, nch_b, S, seg_chunks;
  int tma_tt;  // tile tokens of the TMA-staged path; 0 when the shape does not allow it
  bool heads;  // the Mamba-2-form path (scan_bwd_heads.cu) applies
  // Persistent TMA path: every chunk is a segment (S == nch_b), resident blocks take (chain,
  // chunk) units from a queue, last chunk first, and hand each chunk's start adjoint to the unit
  // of the chunk before it (see scan_bwd_tma.cu).
  bool persist;
  size_t off_fwd, fwd_bytes, off_ckpt, off_dhloc, off_segend, off_sumd, off_part_bc, off_dA,
      off_dD, off_dtb, off_ddt, off_dh0, off_mh, off_queue, bytes, smem;
};
// Resident blocks per SM the TMA-staged backward is built for (its launch bound; each block
// also holds a quarter of the SM's tensor memory).
constexpr int kBwdTmaBlocksPerSM = 4;

// Mamba-2-form backward (scan_bwd_heads.cu): one A per head, head_dim % 32 == 0, d_state 128.
bool bwd_heads_applies(const ScanProblem& p, int chunk_b);
int bwd_heads_blocks(const ScanProblem& p);
size_t bwd_heads_scratch_floats(const ScanProblem& p, int S, int chunk_b);
cudaError_t launch_bwd_heads(const BwdArgs& a, float* scratch, cudaStream_t st);

// TMA-staged backward kernels (scan_bwd_tma.cu), Mamba-1 layout with d_state 16.
// bwd_tma_tile: the tile size this shape would use, 0 if the path cannot take it.
int bwd_tma_tile(const ScanProblem& p, int chunk_b, int gc);
// Channels per block of the TMA-staged main kernel (its per-block dB/dC partials are per
// this many channels).
int bwd_tma_channels_per_block();
// Ints of the persistent path's queue area in the workspace (counters, flags, unit counts).
int bwd_tma_queue_ints(const ScanProblem& p, int nch, long chains);
// The persistent TMA path sums the dB/dC partials itself, in reduction items of its queue.
// Both return cudaErrorNotSupported, launching nothing, when the pointers do not allow the
// path; the caller then runs the general kernels.
cudaError_t launch_bwd_tma_local(const BwdArgs& a, const BwdPlan& q, char* ws, cudaStream_t st);
cudaError_t launch_bwd_tma_main(const BwdArgs& a, const BwdPlan& q, char* ws, cudaStream_t st);
// Whether launch_bwd_tma_main will take this call (the plan allows TMA and the pointers do).
bool bwd_tma_ready(const BwdArgs& a, const BwdPlan& q);

}  // namespace ssm

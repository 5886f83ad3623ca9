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

struct BwdPlan {
  int tpc, gc, bpg, chunk_b, nch_b, S, seg_chunks;
  int tma_tt;  // tile tokens of the TMA-staged path; 0 when the shape does not allow it
  size_t off_fwd, fwd_bytes, off_ckpt, off_dhloc, off_segend, off_sumd, off_part_bc, off_dA,
      off_dD, off_dtb, off_ddt, off_dh0, off_bnd, bytes, smem;
};

// TMA-staged backward kernels (scan_bwd_tma.cu), Mamba-1 layout with d_state 16.
// bwd_tma_tile: the tile size this shape would use, 0 if the path cannot take it.
int bwd_tma_tile(const ScanProblem& p, int chunk_b, int tpc, int gc);
// Both return cudaErrorNotSupported, launching nothing, when the pointers do not allow the
// path; the caller then runs the general kernels.
cudaError_t launch_bwd_tma_local(const BwdArgs& a, const BwdPlan& q, char* ws, cudaStream_t st);
cudaError_t launch_bwd_tma_main(const BwdArgs& a, const BwdPlan& q, char* ws, cudaStream_t st);

}  // namespace ssm

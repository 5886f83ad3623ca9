// scan_common.cuh -- layout decisions and small helpers shared by the scan kernels.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace ssm {

constexpr int kScanThreads = 128;              // threads per scan block
constexpr long kFwdTargetThreadsPerSM = 768;   // below this, time segments add parallelism
// Backward time segments: none when the (sequence, channel block) grid alone has
// kBwdNoSplitThreadsPerSM threads per SM; otherwise enough segments for kBwdTargetThreadsPerSM
// (each extra segment costs a local adjoint pass; measured on GB300 with one long sequence).
constexpr long kBwdNoSplitThreadsPerSM = 512;
constexpr long kBwdTargetThreadsPerSM = 4096;
constexpr int kMinSegment = 64;                // shortest time segment worth a block

__host__ inline int pow2_ceil(int v) {
  int r = 1;
  while (r < v) r <<= 1;
  return r;
}

// States per thread (ns, a power of two in {4, 8, 16}) and threads per channel (tpc, a
// power of two <= 32) so that ns * tpc >= N; states beyond N are padding and stay zero.
__host__ inline void state_split(int N, int pref_ns, int* ns, int* tpc) {
  int n = pow2_ceil(N);
  if (n < 4) n = 4;
  *ns = n < pref_ns ? n : pref_ns;
  *tpc = pow2_ceil((N + *ns - 1) / *ns);
}

// ---- the per-step decay ---------------------------------------------------------------
// Fast form (bf16 I/O): a = 2^(delta A log2 e) by the SFU, h <- a h + u.
// Accurate form (fp32 I/O): when delta |A| is small, a sits just below 1 and fp32 cannot hold
// 1 - a to better than ~6e-8 / (delta |A|); the SFU result is also biased there (about -0.3
// ulp), and both errors compound over the ~1 / (delta |A|) tokens a state remembers.  The step
// therefore carries e = exp(delta A) - 1 and updates h <- h + (e h + u), which keeps each
// step's error at one fp32 rounding of h.  e comes from the Taylor series x + x^2/2 + x^3/6 +
// x^4/24 (remainder below 1.3e-7 relative for |x| < 1/16) and from 2^(x log2 e) - 1 above that.
// SMALL (the backward kernels): for a small decay 1 + e keeps only ~6e-8 / a of it (a gradient
// through a decay of 1e-5 would be 1 % off), so above |delta A| = 1/16, where 1 - a > 0.06 and
// a itself is as good, the step carries a from the SFU and updates h <- a h + u.  (The forward
// keeps e up to the SFU range: its outputs need no relative precision of small decays, and its
// 1e-4 fp32 gate has little room for a change of rounding.)
// Either way the coefficient is (c, s) with a = c + s: (a, 0) for the fast form and for the
// larger SMALL steps, (e, 1) otherwise.  s is 0 or 1, so s h and s v are exact; without SMALL
// it is the constant 1 of the accurate form.
struct DecayCoef { float c, s; };
template <bool ACC, bool SMALL = false>
__device__ __forceinline__ DecayCoef decay_coef(float dl, float A2) {
  const float x2 = dl * A2;  // delta A log2(e)
  const float a = ex2(x2);
  if (!ACC) return DecayCoef{a, 0.0f};
  const float x = x2 * 0.6931471805599453f;  // delta A
  const float p = x * fmaf(x, fmaf(x, fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f), 1.0f);
  const bool near1 = fabsf(x) < 0.0625f;
  if (!SMALL) return DecayCoef{near1 ? p : a - 1.0f, 1.0f};
  return DecayCoef{near1 ? p : a, near1 ? 1.0f : 0.0f};  // selects: neighbouring states differ
}
// h <- a h + u   (fast)   or   h <- (c h + u) + s h   (accurate; (e h + u) + h near a = 1)
template <bool ACC>
__device__ __forceinline__ float decay_step(DecayCoef k, float h, float u) {
  return ACC ? fmaf(k.s, h, fmaf(k.c, h, u)) : fmaf(k.c, h, u);
}
// a * v   (fast)   or   c v + s v   (accurate; v + e v near a = 1)
template <bool ACC>
__device__ __forceinline__ float decay_apply(DecayCoef k, float v) {
  return ACC ? fmaf(k.c, v, k.s * v) : k.c * v;
}

// Packed versions for a pair of states (f32x2): the coefficients and their two uses.
struct DecayCoef2 { f2_t c, s; };
__device__ __forceinline__ DecayCoef2 decay_pair(DecayCoef k) {
  return DecayCoef2{f2_pack(k.c, k.c), f2_pack(k.s, k.s)};
}
template <bool ACC, bool SMALL = false>
__device__ __forceinline__ DecayCoef2 decay2(f2_t dl2, f2_t A2p) {
  if constexpr (!ACC) return DecayCoef2{f2_ex2(f2_mul(dl2, A2p)), 0ull};
  float dl, d2, a0, a1;
  f2_unpack(dl2, dl, d2);
  f2_unpack(A2p, a0, a1);
  const DecayCoef k0 = decay_coef<true, SMALL>(dl, a0), k1 = decay_coef<true, SMALL>(dl, a1);
  return DecayCoef2{f2_pack(k0.c, k1.c), f2_pack(k0.s, k1.s)};
}
template <bool ACC>
__device__ __forceinline__ f2_t step2(const DecayCoef2& k, f2_t h, f2_t u) {
  return ACC ? f2_fma(k.s, h, f2_fma(k.c, h, u)) : f2_fma(k.c, h, u);
}
template <bool ACC>
__device__ __forceinline__ f2_t apply2(const DecayCoef2& k, f2_t v) {
  return ACC ? f2_fma(k.c, v, f2_mul(k.s, v)) : f2_mul(k.c, v);
}
__device__ __forceinline__ float f2_sum(f2_t v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  return lo + hi;
}

// Lanes of the tpc-lane group this lane belongs to (xor-shuffles stay inside it).
__device__ __forceinline__ unsigned group_mask(int tpc) {
  if (tpc >= 32) return 0xffffffffu;
  const int lane = threadIdx.x & 31;
  return ((1u << tpc) - 1u) << (lane & ~(tpc - 1));
}

// Row of s0 that sequence b starts from, or NULL for a zero state.  An id outside
// [0, state_rows) is recorded in the status word and read as a zero state.
__device__ __forceinline__ const float* start_row(const ScanProblem& p, int b) {
  if (!p.s0) return nullptr;
  int row = p.ids ? __ldg(p.ids + b) : b;
  if (row < 0 || row >= p.state_rows) {
    record_status(p.status, SSM_ERR_INVALID_ARG);
    return nullptr;
  }
  return p.s0 + (long)row * p.HP * p.N;
}

// NS consecutive values of a B or C row.  FULL: all NS are in range and the address is
// aligned to min(16, NS * sizeof(IO)) bytes, so vector loads are used.
template <typename IO, int NS, bool FULL>
__device__ __forceinline__ void load_row(const IO* ptr, int nvalid, float (&out)[NS]) {
  if (FULL) {
    if (sizeof(IO) == 4) {
#pragma unroll
      for (int j = 0; j < NS; j += 4) {
        float4 v = __ldg(reinterpret_cast<const float4*>(ptr + j));
        out[j] = v.x; out[j + 1] = v.y; out[j + 2] = v.z; out[j + 3] = v.w;
      }
    } else if (NS >= 8) {
#pragma unroll
      for (int j = 0; j < NS; j += 8) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(ptr + j));
        const __nv_bfloat162* q = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int k = 0; k < 4; k++) {
          float2 f = __bfloat1622float2(q[k]);
          out[j + 2 * k] = f.x;
          out[j + 2 * k + 1] = f.y;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < NS; j += 4) {
        uint2 v = __ldg(reinterpret_cast<const uint2*>(ptr + j));
        const __nv_bfloat162* q = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int k = 0; k < 2; k++) {
          float2 f = __bfloat1622float2(q[k]);
          out[j + 2 * k] = f.x;
          out[j + 2 * k + 1] = f.y;
        }
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < NS; j++) out[j] = (j < nvalid) ? ld(ptr + j) : 0.0f;
  }
}

__host__ inline bool rows_vectorizable(const ScanProblem& p, int ns, int tpc) {
  if (p.N != ns * tpc) return false;
  const size_t sz = p.io == SSM_BF16 ? 2 : 4;
  const size_t vb = ns * sz < 16 ? ns * sz : 16;
  if ((p.N * sz) % vb != 0) return false;
  if (((uintptr_t)p.B % 16) != 0 || ((uintptr_t)p.C % 16) != 0) return false;
  return true;
}

}  // namespace ssm

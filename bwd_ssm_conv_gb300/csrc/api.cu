// api.cu -- the extern "C" entry points of include/ssm.h: argument validation on the host,
// workspace carving, launch.  Nothing here allocates, frees or synchronises (except
// ssm_scan_status, which by contract waits for the stream to read the status word).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.cuh"
#include "ssm.h"

#include <atomic>

namespace ssm {
static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace ssm

namespace {

using ssm::ScanGrads;
using ssm::ScanProblem;

constexpr long long kMaxPerSeq = (1LL << 31) - 1;
constexpr long long kMaxTotal = 1LL << 40;

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int io_size(int io) { return io == SSM_BF16 ? 2 : (io == SSM_F32 ? 4 : 0); }

int num_sms_current() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int conv_check(const void* sx, const float* c, const void* out, int n_s, int d_inner, int n_t,
               int d_conv, int io) {
  if (!sx || !c || !out) return SSM_ERR_INVALID_ARG;
  if (n_s <= 0 || d_inner <= 0 || n_t <= 0 || d_conv <= 0) return SSM_ERR_INVALID_ARG;
  const int sz = io_size(io);
  if (!sz) return SSM_ERR_INVALID_ARG;
  if (d_conv > SSM_MAX_D_CONV) return SSM_ERR_UNSUPPORTED;
  const long long W = (long long)n_t + d_conv - 1;
  if ((long long)d_inner * W > kMaxPerSeq || (long long)n_s * d_inner * W > kMaxTotal)
    return SSM_ERR_UNSUPPORTED;
  if (!aligned(sx, sz) || !aligned(out, sz) || !aligned(c, 4)) return SSM_ERR_INVALID_ARG;
  return SSM_OK;
}

// Fills a ScanProblem from a descriptor; returns a status.
int scan_problem(const ssm_scan_desc* d, int backward, ScanProblem* p) {
  if (!d) return SSM_ERR_INVALID_ARG;
  if (d->n_seqs <= 0 || d->n_tok <= 0 || d->n_head <= 0 || d->head_dim <= 0 || d->d_state <= 0 ||
      d->n_group <= 0 || d->state_rows < 0 || d->chunk < 0)
    return SSM_ERR_INVALID_ARG;
  if (d->n_head % d->n_group != 0) return SSM_ERR_INVALID_ARG;
  if (d->a_per_state != 0 && d->a_per_state != 1) return SSM_ERR_INVALID_ARG;
  if (!io_size(d->io)) return SSM_ERR_INVALID_ARG;
  if (d->flags & ~(unsigned)(SSM_DT_SOFTPLUS | SSM_CHECK_FINITE | SSM_A_LOG | SSM_DEBUG_NO_WAIT |
                             SSM_SCAN_CHUNKED))
    return SSM_ERR_INVALID_ARG;
  if (d->d_state > (backward ? SSM_MAX_D_STATE_BWD : SSM_MAX_D_STATE)) return SSM_ERR_UNSUPPORTED;
  const long long HP = (long long)d->n_head * d->head_dim;
  const long long per_seq = (long long)d->n_tok * HP * d->d_state;
  const long long bc = (long long)d->n_tok * d->n_group * d->d_state;
  if (per_seq > kMaxPerSeq || bc > kMaxPerSeq || HP > kMaxPerSeq) return SSM_ERR_UNSUPPORTED;
  if ((long long)d->n_seqs * per_seq > kMaxTotal) return SSM_ERR_UNSUPPORTED;
  *p = ScanProblem{};
  p->ns = d->n_seqs;
  p->L = d->n_tok;
  p->H = d->n_head;
  p->P = d->head_dim;
  p->N = d->d_state;
  p->G = d->n_group;
  p->HP = (int)HP;
  p->a_per_state = d->a_per_state;
  p->softplus = (d->flags & SSM_DT_SOFTPLUS) ? 1 : 0;
  p->check_finite = (d->flags & SSM_CHECK_FINITE) ? 1 : 0;
  p->debug_flags = (d->flags & SSM_DEBUG_NO_WAIT) ? ssm::kDebugNoWait : 0;
  p->chunked = (d->flags & SSM_SCAN_CHUNKED) ? 1 : 0;
  p->state_rows = d->state_rows > 0 ? d->state_rows : d->n_seqs;
  p->chunk = d->chunk > 0 ? d->chunk : 256;
  p->n_chunks = (p->L + p->chunk - 1) / p->chunk;
  p->io = d->io;
  return SSM_OK;
}

int check_act(const void* ptr, int io) { return aligned(ptr, io_size(io)); }

// SSM_A_LOG: elements of A and the 256-aligned scratch holding A = -exp(A_log), placed after
// the `base` bytes a call's plan needs.
bool a_log_of(const ssm_scan_desc* d) { return d && (d->flags & SSM_A_LOG); }
int a_count(const ScanProblem& p) { return p.a_per_state ? p.H * p.N : p.H; }
size_t a_bytes(const ScanProblem& p) { return ssm::align_up(sizeof(float) * (size_t)a_count(p), 256); }

// Converts A_log into the scratch after `base` and points p->A at it.
int stage_a(const ssm_scan_desc* d, ScanProblem* p, void* ws, size_t base, cudaStream_t st) {
  if (!a_log_of(d)) return SSM_OK;
  float* a = (float*)((char*)ws + ssm::align_up(base, 256));
  if (ssm::launch_a_from_log(p->A, a, a_count(*p), st) != cudaSuccess) return SSM_ERR_CUDA;
  p->A = a;
  return SSM_OK;
}

}  // namespace

extern "C" {

int ssm_abi_version(void) { return SSM_ABI_VERSION; }

unsigned long long ssm_kernel_launches(void) {
  return ssm::g_launches.load(std::memory_order_relaxed);
}

const char* ssm_status_string(int s) {
  switch (s) {
    case SSM_OK: return "ok";
    case SSM_ERR_INVALID_ARG: return "invalid argument (null pointer, size, alignment or state row id)";
    case SSM_ERR_UNSUPPORTED: return "size beyond a documented limit of this library";
    case SSM_ERR_WORKSPACE: return "workspace missing or smaller than the *_workspace_size result";
    case SSM_ERR_CUDA: return "a CUDA launch failed";
    case SSM_ERR_TIMEOUT: return "a bounded wait (for a staged tile, or for the next chunk's adjoint) gave up; that block skipped the rest of its work";
    case SSM_ERR_NONFINITE: return "a non-finite output was produced";
    default: return "unknown status";
  }
}

int ssm_conv_fwd(const void* sx, const float* c, const float* bias, void* out,
                 void* conv_state_out, int n_s, int d_inner, int n_t, int d_conv, int io,
                 unsigned flags, void* stream) {
  int rc = conv_check(sx, c, out, n_s, d_inner, n_t, d_conv, io);
  if (rc != SSM_OK) return rc;
  if (flags & ~(unsigned)SSM_CONV_SILU) return SSM_ERR_INVALID_ARG;
  if ((bias && !aligned(bias, 4)) || (conv_state_out && !check_act(conv_state_out, io)))
    return SSM_ERR_INVALID_ARG;
  cudaError_t e = ssm::launch_conv_fwd(sx, c, bias, out, conv_state_out, n_s, d_inner, n_t, d_conv,
                                       io, (flags & SSM_CONV_SILU) ? 1 : 0, (cudaStream_t)stream);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_conv_workspace_size(int n_s, int d_inner, int n_t, int d_conv) {
  if (n_s <= 0 || d_inner <= 0 || n_t <= 0 || d_conv <= 0 || d_conv > SSM_MAX_D_CONV) return 0;
  return ssm::conv_bwd_ws_bytes(n_s, d_inner, n_t, d_conv);
}

int ssm_conv_bwd(const void* sx, const float* c, const float* bias, const void* dout,
                 void* d_sx, float* d_c, float* d_bias, void* ws, size_t ws_bytes, int n_s,
                 int d_inner, int n_t, int d_conv, int io, unsigned flags, void* stream) {
  int rc = conv_check(sx, c, dout, n_s, d_inner, n_t, d_conv, io);
  if (rc != SSM_OK) return rc;
  if (!d_sx || !d_c || !check_act(d_sx, io) || !aligned(d_c, 4)) return SSM_ERR_INVALID_ARG;
  if ((bias && !aligned(bias, 4)) || (d_bias && !aligned(d_bias, 4))) return SSM_ERR_INVALID_ARG;
  if (flags & ~(unsigned)SSM_CONV_SILU) return SSM_ERR_INVALID_ARG;
  const size_t need = ssm::conv_bwd_ws_bytes(n_s, d_inner, n_t, d_conv);
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return SSM_ERR_WORKSPACE;
  cudaError_t e = ssm::launch_conv_bwd(sx, c, bias, dout, d_sx, d_c, d_bias, ws, n_s, d_inner, n_t,
                                       d_conv, io, (flags & SSM_CONV_SILU) ? 1 : 0,
                                       (cudaStream_t)stream);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_scan_workspace_size(const ssm_scan_desc* desc, int backward) {
  ScanProblem p;
  if (scan_problem(desc, backward, &p) != SSM_OK) return 0;
  const int sms = num_sms_current();
  if (sms <= 0) return 0;
  const size_t base = backward ? ssm::scan_bwd_ws_bytes(p, sms) : ssm::scan_fwd_ws_bytes(p, sms);
  return a_log_of(desc) ? ssm::align_up(base, 256) + a_bytes(p) : base;
}

int ssm_scan_fwd(const ssm_scan_desc* desc, const float* s0, const int32_t* ids, const void* x,
                 const void* dt, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, void* y, float* state_out, float* ckpt,
                 void* ws, size_t ws_bytes, void* stream) {
  ScanProblem p;
  int rc = scan_problem(desc, 0, &p);
  if (rc != SSM_OK) return rc;
  if (!x || !dt || !A || !B || !C || !y || !state_out) return SSM_ERR_INVALID_ARG;
  const int io = p.io;
  if (!check_act(x, io) || !check_act(dt, io) || !check_act(B, io) || !check_act(C, io) ||
      !check_act(y, io) || (z && !check_act(z, io)) || !aligned(A, 4) || !aligned(state_out, 4) ||
      (s0 && !aligned(s0, 4)) || (ids && !aligned(ids, 4)) || (D && !aligned(D, 4)) ||
      (dt_bias && !aligned(dt_bias, 4)) || (ckpt && !aligned(ckpt, 4)))
    return SSM_ERR_INVALID_ARG;
  if (!ids && s0 && p.state_rows < p.ns) return SSM_ERR_INVALID_ARG;
  const int sms = num_sms_current();
  if (sms <= 0) return SSM_ERR_CUDA;
  const size_t base = ssm::scan_fwd_ws_bytes(p, sms);
  const size_t need = a_log_of(desc) ? ssm::align_up(base, 256) + a_bytes(p) : base;
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return SSM_ERR_WORKSPACE;
  p.s0 = s0; p.ids = ids; p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.dt_bias = dt_bias;
  p.status = (int*)ws;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return SSM_ERR_CUDA;
  if ((rc = stage_a(desc, &p, ws, base, st)) != SSM_OK) return rc;
  cudaError_t e = ssm::launch_scan_fwd(p, y, state_out, ckpt, ws, sms, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_scan_bwd(const ssm_scan_desc* desc, const float* s0, const int32_t* ids, const void* x,
                 const void* dt, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, const float* ckpt, const void* dy,
                 const float* d_state_out, float* d_s0, void* d_x, void* d_dt, float* d_A,
                 void* d_B, void* d_C, float* d_D, void* d_z, float* d_dt_bias, void* ws,
                 size_t ws_bytes, void* stream) {
  ScanProblem p;
  int rc = scan_problem(desc, 1, &p);
  if (rc != SSM_OK) return rc;
  if (!x || !dt || !A || !B || !C || !dy || !d_x || !d_dt || !d_A || !d_B || !d_C)
    return SSM_ERR_INVALID_ARG;
  if ((d_D && !D) || (d_z && !z) || (d_dt_bias && !p.softplus)) return SSM_ERR_INVALID_ARG;
  const int io = p.io;
  if (!check_act(x, io) || !check_act(dt, io) || !check_act(B, io) || !check_act(C, io) ||
      !check_act(dy, io) || !check_act(d_x, io) || !check_act(d_dt, io) || !check_act(d_B, io) ||
      !check_act(d_C, io) || (z && !check_act(z, io)) || (d_z && !check_act(d_z, io)) ||
      !aligned(A, 4) || !aligned(d_A, 4) || (s0 && !aligned(s0, 4)) || (ids && !aligned(ids, 4)) ||
      (D && !aligned(D, 4)) || (d_D && !aligned(d_D, 4)) || (dt_bias && !aligned(dt_bias, 4)) ||
      (d_dt_bias && !aligned(d_dt_bias, 4)) || (ckpt && !aligned(ckpt, 4)) ||
      (d_state_out && !aligned(d_state_out, 4)) || (d_s0 && !aligned(d_s0, 4)))
    return SSM_ERR_INVALID_ARG;
  if (!ids && (s0 || d_s0) && p.state_rows < p.ns) return SSM_ERR_INVALID_ARG;
  const int sms = num_sms_current();
  if (sms <= 0) return SSM_ERR_CUDA;
  const size_t base = ssm::scan_bwd_ws_bytes(p, sms);
  const size_t need = a_log_of(desc) ? ssm::align_up(base, 256) + a_bytes(p) : base;
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return SSM_ERR_WORKSPACE;
  p.s0 = s0; p.ids = ids; p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.dt_bias = dt_bias;
  p.status = (int*)ws;
  ScanGrads g{dy, d_state_out, d_s0, d_x, d_dt, d_A, d_B, d_C, d_D, d_z, d_dt_bias};
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return SSM_ERR_CUDA;
  if ((rc = stage_a(desc, &p, ws, base, st)) != SSM_OK) return rc;
  cudaError_t e = ssm::launch_scan_bwd(p, ckpt, g, ws, sms, st);
  if (e == cudaSuccess && a_log_of(desc)) e = ssm::launch_scale_dA(d_A, p.A, a_count(p), st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// ---- fused conv1d + scan --------------------------------------------------------------------
}  // extern "C"

namespace {

// Workspace of the fused calls: the scan's own scratch (with the A_LOG buffer), then the conv
// output x (used only when the fused forward kernel does not apply, and by the backward), then
// (backward) dL/dx and the conv backward's partial sums.
struct ConvScanWs {
  size_t scan, x, dx, conv, bytes;
};

ConvScanWs conv_scan_ws(const ssm_scan_desc* d, const ScanProblem& p, int K, int backward,
                        int sms) {
  ConvScanWs w{};
  const size_t base = backward ? ssm::scan_bwd_ws_bytes(p, sms) : ssm::scan_fwd_ws_bytes(p, sms);
  w.scan = a_log_of(d) ? ssm::align_up(base, 256) + a_bytes(p) : base;
  const size_t xb = (size_t)p.ns * p.L * p.HP * io_size(p.io);
  w.x = ssm::align_up(w.scan, 256);
  size_t off = ssm::align_up(w.x + xb, 256);
  if (backward) {
    w.dx = off;
    off = ssm::align_up(w.dx + xb, 256);
    w.conv = off;
    off = ssm::align_up(w.conv + ssm::conv_bwd_ws_bytes(p.ns, p.HP, p.L, K), 256);
  }
  w.bytes = off;
  return w;
}

int conv_scan_check(const ssm_scan_desc* d, int K, unsigned conv_flags, const void* sx,
                    const float* c, const float* cb, int backward, ScanProblem* p) {
  int rc = scan_problem(d, backward, p);
  if (rc != SSM_OK) return rc;
  if (K <= 0 || conv_flags & ~(unsigned)SSM_CONV_SILU) return SSM_ERR_INVALID_ARG;
  if (K > SSM_MAX_D_CONV) return SSM_ERR_UNSUPPORTED;
  rc = conv_check(sx, c, sx, p->ns, p->HP, p->L, K, p->io);
  if (rc != SSM_OK) return rc;
  if (cb && !aligned(cb, 4)) return SSM_ERR_INVALID_ARG;
  return SSM_OK;
}

}  // namespace

extern "C" {

size_t ssm_conv_scan_workspace_size(const ssm_scan_desc* desc, int d_conv, int backward) {
  ScanProblem p;
  if (scan_problem(desc, backward, &p) != SSM_OK) return 0;
  if (d_conv <= 0 || d_conv > SSM_MAX_D_CONV) return 0;
  const int sms = num_sms_current();
  if (sms <= 0) return 0;
  return conv_scan_ws(desc, p, d_conv, backward, sms).bytes;
}

int ssm_conv_scan_fwd(const ssm_scan_desc* desc, int d_conv, unsigned conv_flags, const void* sx,
                      const float* conv_w, const float* conv_b, const float* s0,
                      const int32_t* ids, const void* dt, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* dt_bias,
                      void* y, float* state_out, float* ckpt, void* ws, size_t ws_bytes,
                      void* stream) {
  ScanProblem p;
  int rc = conv_scan_check(desc, d_conv, conv_flags, sx, conv_w, conv_b, 0, &p);
  if (rc != SSM_OK) return rc;
  if (!dt || !A || !B || !C || !y || !state_out) return SSM_ERR_INVALID_ARG;
  const int io = p.io;
  if (!check_act(dt, io) || !check_act(B, io) || !check_act(C, io) || !check_act(y, io) ||
      (z && !check_act(z, io)) || !aligned(A, 4) || !aligned(state_out, 4) ||
      (s0 && !aligned(s0, 4)) || (ids && !aligned(ids, 4)) || (D && !aligned(D, 4)) ||
      (dt_bias && !aligned(dt_bias, 4)) || (ckpt && !aligned(ckpt, 4)))
    return SSM_ERR_INVALID_ARG;
  if (!ids && s0 && p.state_rows < p.ns) return SSM_ERR_INVALID_ARG;
  const int sms = num_sms_current();
  if (sms <= 0) return SSM_ERR_CUDA;
  const ConvScanWs w = conv_scan_ws(desc, p, d_conv, 0, sms);
  if (!ws || ws_bytes < w.bytes || !aligned(ws, 256)) return SSM_ERR_WORKSPACE;
  p.s0 = s0; p.ids = ids; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.dt_bias = dt_bias;
  p.status = (int*)ws;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return SSM_ERR_CUDA;
  if ((rc = stage_a(desc, &p, ws, ssm::scan_fwd_ws_bytes(p, sms), st)) != SSM_OK) return rc;
  const int silu = (conv_flags & SSM_CONV_SILU) ? 1 : 0;
  // the fused kernel: x is computed from sx inside the scan and never stored
  ScanProblem pf = p;
  pf.sx = sx; pf.conv_w = conv_w; pf.conv_b = conv_b; pf.d_conv = d_conv; pf.conv_silu = silu;
  cudaError_t e = ssm::launch_scan_fwd_tma(pf, y, state_out, ckpt, ws, sms, st);
  if (e == cudaErrorNotSupported) {  // otherwise the conv into the workspace, then the scan
    void* x = (char*)ws + w.x;
    e = ssm::launch_conv_fwd(sx, conv_w, conv_b, x, nullptr, p.ns, p.HP, p.L, d_conv, io, silu, st);
    p.x = x;
    if (e == cudaSuccess) e = ssm::launch_scan_fwd(p, y, state_out, ckpt, ws, sms, st);
  }
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_conv_scan_bwd(const ssm_scan_desc* desc, int d_conv, unsigned conv_flags, const void* sx,
                      const float* conv_w, const float* conv_b, const float* s0,
                      const int32_t* ids, const void* dt, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* dt_bias,
                      const float* ckpt, const void* dy, const float* d_state_out, float* d_s0,
                      void* d_sx, float* d_conv_w, float* d_conv_b, void* d_dt, float* d_A,
                      void* d_B, void* d_C, float* d_D, void* d_z, float* d_dt_bias, void* ws,
                      size_t ws_bytes, void* stream) {
  ScanProblem p;
  int rc = conv_scan_check(desc, d_conv, conv_flags, sx, conv_w, conv_b, 1, &p);
  if (rc != SSM_OK) return rc;
  if (!dt || !A || !B || !C || !dy || !d_sx || !d_conv_w || !d_dt || !d_A || !d_B || !d_C)
    return SSM_ERR_INVALID_ARG;
  if ((d_D && !D) || (d_z && !z) || (d_dt_bias && !p.softplus)) return SSM_ERR_INVALID_ARG;
  const int io = p.io;
  if (!check_act(dt, io) || !check_act(B, io) || !check_act(C, io) || !check_act(dy, io) ||
      !check_act(d_sx, io) || !check_act(d_dt, io) || !check_act(d_B, io) ||
      !check_act(d_C, io) || (z && !check_act(z, io)) || (d_z && !check_act(d_z, io)) ||
      !aligned(A, 4) || !aligned(d_A, 4) || !aligned(d_conv_w, 4) ||
      (d_conv_b && !aligned(d_conv_b, 4)) || (s0 && !aligned(s0, 4)) ||
      (ids && !aligned(ids, 4)) || (D && !aligned(D, 4)) || (d_D && !aligned(d_D, 4)) ||
      (dt_bias && !aligned(dt_bias, 4)) || (d_dt_bias && !aligned(d_dt_bias, 4)) ||
      (ckpt && !aligned(ckpt, 4)) || (d_state_out && !aligned(d_state_out, 4)) ||
      (d_s0 && !aligned(d_s0, 4)))
    return SSM_ERR_INVALID_ARG;
  if (!ids && (s0 || d_s0) && p.state_rows < p.ns) return SSM_ERR_INVALID_ARG;
  const int sms = num_sms_current();
  if (sms <= 0) return SSM_ERR_CUDA;
  const ConvScanWs w = conv_scan_ws(desc, p, d_conv, 1, sms);
  if (!ws || ws_bytes < w.bytes || !aligned(ws, 256)) return SSM_ERR_WORKSPACE;
  p.s0 = s0; p.ids = ids; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.dt_bias = dt_bias;
  p.status = (int*)ws;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return SSM_ERR_CUDA;
  if ((rc = stage_a(desc, &p, ws, ssm::scan_bwd_ws_bytes(p, sms), st)) != SSM_OK) return rc;
  const int silu = (conv_flags & SSM_CONV_SILU) ? 1 : 0;
  // x recomputed from sx, the scan's backward into dL/dx, then the conv's backward
  void* x = (char*)ws + w.x;
  void* dx = (char*)ws + w.dx;
  cudaError_t e = ssm::launch_conv_fwd(sx, conv_w, conv_b, x, nullptr, p.ns, p.HP, p.L, d_conv,
                                       io, silu, st);
  p.x = x;
  ScanGrads g{dy, d_state_out, d_s0, dx, d_dt, d_A, d_B, d_C, d_D, d_z, d_dt_bias};
  if (e == cudaSuccess) e = ssm::launch_scan_bwd(p, ckpt, g, ws, sms, st);
  if (e == cudaSuccess && a_log_of(desc)) e = ssm::launch_scale_dA(d_A, p.A, a_count(p), st);
  if (e == cudaSuccess)
    e = ssm::launch_conv_bwd(sx, conv_w, conv_b, dx, d_sx, d_conv_w, d_conv_b, (char*)ws + w.conv,
                             p.ns, p.HP, p.L, d_conv, io, silu, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_decode_step(const ssm_scan_desc* desc, int d_conv, unsigned conv_flags,
                    const int32_t* ids, const void* x_new, void* conv_state, const float* c,
                    const float* bias, const void* dt, const float* A, const void* B,
                    const void* C, const float* D, const void* z, const float* dt_bias,
                    float* state, void* y, void* ws, size_t ws_bytes, void* stream) {
  ScanProblem p;
  int rc = scan_problem(desc, 0, &p);
  if (rc != SSM_OK) return rc;
  if (p.L != 1) return SSM_ERR_INVALID_ARG;
  if (d_conv <= 0) return SSM_ERR_INVALID_ARG;
  if (d_conv > SSM_MAX_D_CONV) return SSM_ERR_UNSUPPORTED;
  if (conv_flags & ~(unsigned)SSM_CONV_SILU) return SSM_ERR_INVALID_ARG;
  if (!x_new || !c || !dt || !A || !B || !C || !state || !y || (d_conv > 1 && !conv_state))
    return SSM_ERR_INVALID_ARG;
  const int io = p.io;
  if (!check_act(x_new, io) || !check_act(dt, io) || !check_act(B, io) || !check_act(C, io) ||
      !check_act(y, io) || (z && !check_act(z, io)) || (conv_state && !check_act(conv_state, io)) ||
      !aligned(c, 4) || (bias && !aligned(bias, 4)) || !aligned(A, 4) || !aligned(state, 4) ||
      (ids && !aligned(ids, 4)) || (D && !aligned(D, 4)) || (dt_bias && !aligned(dt_bias, 4)))
    return SSM_ERR_INVALID_ARG;
  if (!ids && p.state_rows < p.ns) return SSM_ERR_INVALID_ARG;
  if ((long long)p.state_rows * p.HP * p.N > kMaxTotal ||
      (long long)p.state_rows * p.HP * d_conv > kMaxTotal)
    return SSM_ERR_UNSUPPORTED;
  const size_t need = ssm::kStatusBytes + (a_log_of(desc) ? a_bytes(p) : 0);
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return SSM_ERR_WORKSPACE;
  p.ids = ids; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z; p.dt_bias = dt_bias;
  p.status = (int*)ws;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return SSM_ERR_CUDA;
  if ((rc = stage_a(desc, &p, ws, ssm::kStatusBytes, st)) != SSM_OK) return rc;
  cudaError_t e = ssm::launch_decode_step(p, d_conv, (conv_flags & SSM_CONV_SILU) ? 1 : 0, x_new,
                                          conv_state, c, bias, state, y, st);
  return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int ssm_scan_status(const void* ws, int* status, void* stream) {
  if (!ws || !status) return SSM_ERR_INVALID_ARG;
  int v = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSM_ERR_CUDA;
  *status = v;
  return SSM_OK;
}

}  // extern "C"

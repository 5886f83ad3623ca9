// kernels.cuh -- host-side launchers of the kernel files, called by the C ABI in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace ssm {

// ---- conv ---------------------------------------------------------------------------------
size_t conv_bwd_ws_bytes(int n_s, int D, int L, int K);
cudaError_t launch_conv_fwd(const void* sx, const float* c, const float* bias, void* out, void* cs,
                            int n_s, int D, int L, int K, int io, int silu, cudaStream_t st);
cudaError_t launch_conv_bwd(const void* sx, const float* c, const float* bias, const void* dout,
                            void* d_sx, float* d_c, float* d_bias, void* ws, int n_s, int D, int L,
                            int K, int io, int silu, cudaStream_t st);

// ---- scan ---------------------------------------------------------------------------------
// Everything a scan launch needs, validated by the caller.  Pointers are device pointers.
struct ScanProblem {
  int ns, L, H, P, N, G, HP;
  int a_per_state, softplus, check_finite;
  int state_rows, chunk, n_chunks;
  int io;
  int debug_flags;  // kDebugNoWait: cross-block waits give up at once (tests of the timeout path)
  int chunked;      // SSM_SCAN_CHUNKED: the Mamba-2 form's bf16 forward in chunked matrix form
  const float* s0;
  const int* ids;
  const void* x;
  const void* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* dt_bias;
  int* status;  // device status word
  // Fused conv1d prelude (ssm_conv_scan_fwd): when sx is set, x is not read from memory but
  // computed as act(sum_k sx[b][ch][t+k] conv_w[ch][k] + conv_b[ch]) (act = SiLU when conv_silu)
  // and rounded to the io type, as ssm_conv_fwd would store it.  sx is [ns][HP][L + d_conv - 1].
  const void* sx;
  const float* conv_w;
  const float* conv_b;
  int d_conv, conv_silu;
};

constexpr int kDebugNoWait = 1;

// Forward.  y may be NULL (states / checkpoints only), state_out may be NULL, ckpt may be NULL.
// launch_scan_fwd takes a fast path when one applies: scan_fwd_tma.cu (head_dim 1),
// scan_fwd_heads.cu (one A per head, head_dim a multiple of 64, d_state 128), or, asked for
// with SSM_SCAN_CHUNKED, scan_fwd_ssd.cu (the same shapes with bf16 I/O in chunked matrix form
// on the tensor cores).
size_t scan_fwd_ws_bytes(const ScanProblem& p, int num_sms);
size_t scan_fwd_tma_ws_bytes(const ScanProblem& p, int num_sms);  // 0: path does not apply
cudaError_t launch_scan_fwd_tma(const ScanProblem& p, void* y, float* state_out, float* ckpt,
                                void* ws, int num_sms, cudaStream_t st);
size_t scan_fwd_heads_ws_bytes(const ScanProblem& p, int num_sms);  // 0: path does not apply
cudaError_t launch_scan_fwd_heads(const ScanProblem& p, void* y, float* state_out, float* ckpt,
                                  void* ws, int num_sms, cudaStream_t st);
// scan_fwd_ssd.cu: the Mamba-2 form in chunked matrix form on the tensor cores (SSM_SCAN_CHUNKED;
// bf16 I/O, one A per head, head_dim a multiple of 64, d_state 128, checkpoint interval a
// multiple of 64).
size_t scan_fwd_ssd_ws_bytes(const ScanProblem& p);  // 0: path does not apply
cudaError_t launch_scan_fwd_ssd(const ScanProblem& p, void* y, float* state_out, float* ckpt,
                                void* ws, cudaStream_t st);
cudaError_t launch_scan_fwd(const ScanProblem& p, void* y, float* state_out, float* ckpt, void* ws,
                            int num_sms, cudaStream_t st);

struct ScanGrads {
  const void* dy;
  const float* d_state_out;
  float* d_s0;
  void* d_x;
  void* d_dt;
  float* d_A;
  void* d_B;
  void* d_C;
  float* d_D;
  void* d_z;
  float* d_dt_bias;
};

// Backward.  ckpt: checkpoints at interval p.chunk written by the forward, or NULL.
size_t scan_bwd_ws_bytes(const ScanProblem& p, int num_sms);
cudaError_t launch_scan_bwd(const ScanProblem& p, const float* ckpt, const ScanGrads& g, void* ws,
                            int num_sms, cudaStream_t st);

// A_log parameterisation (params.cu): a = -exp(a_log); d_a *= a.
cudaError_t launch_a_from_log(const float* a_log, float* a, int n, cudaStream_t st);
cudaError_t launch_scale_dA(float* d_a, const float* a, int n, cudaStream_t st);

// Single-token step (decode.cu): p describes one token per sequence (p.L == 1); conv_state
// [rows][HP][K-1] and state [rows][HP][N] are updated in place at row ids[b] (or b).
cudaError_t launch_decode_step(const ScanProblem& p, int K, int silu, const void* x_new,
                               void* conv_state, const float* c, const float* bias, float* state,
                               void* y, cudaStream_t st);

}  // namespace ssm

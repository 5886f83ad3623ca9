/*
 * ssm_oracle.h -- plain, sequential, double-precision CPU oracle for the
 * selective state-space scan and its causal depthwise conv1d prelude.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library under bwd_ssm_conv_gb300/.
 *
 * Every array is row-major, slowest index first, in double precision.
 *   conv:  sx[n_s][d_inner][n_t + d_conv - 1]   (time fastest: ggml's ssm_conv layout)
 *          c[d_inner][d_conv], bias[d_inner]     out[n_s][n_t][d_inner]
 *   scan:  x, z, y, dy  [n_s][L][H][P]           dt [n_s][L][H]
 *          A [H][N] (a_per_state = 1) or [H] (a_per_state = 0)
 *          B, C [n_s][L][G][N]                   D [H*P]   dt_bias [H]
 *          s0, d_s0 [state_rows][H][P][N]        state_out [n_s][H][P][N]
 *          ckpt [n_s][ceil(L/chunk)][H][P][N]    (state at the START of each chunk)
 * All functions return 0 on success, -1 on invalid sizes, -2 on allocation failure.
 */
#ifndef SSM_ORACLE_H
#define SSM_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int n_seqs, n_tok, n_head, head_dim, d_state, n_group;
  int a_per_state;   /* 1: A is [H][N] (Mamba-1 form); 0: A is [H] (one scalar per head) */
  int state_rows;    /* rows of s0 / d_s0 */
  int chunk;         /* checkpoint interval in tokens (>= 1) */
  int dt_softplus;   /* 1: delta = softplus(dt + dt_bias); 0: delta = dt */
} oracle_scan_dims;

int oracle_conv_fwd(const double* sx, const double* c, const double* bias, double* out,
                    double* conv_state_out, int n_s, int d_inner, int n_t, int d_conv, int silu);

int oracle_conv_bwd(const double* sx, const double* c, const double* bias, const double* dout,
                    double* d_sx, double* d_c, double* d_bias,
                    int n_s, int d_inner, int n_t, int d_conv, int silu);

int oracle_scan_fwd(const oracle_scan_dims* dm, const double* s0, const int* ids,
                    const double* x, const double* dt, const double* A, const double* B,
                    const double* C, const double* D, const double* z, const double* dt_bias,
                    double* y, double* state_out, double* ckpt);

/* Exact reverse-mode gradient; keeps the full state history of one channel. */
int oracle_scan_bwd(const oracle_scan_dims* dm, const double* s0, const int* ids,
                    const double* x, const double* dt, const double* A, const double* B,
                    const double* C, const double* D, const double* z, const double* dt_bias,
                    const double* dy, const double* d_state_out,
                    double* d_s0, double* d_x, double* d_dt, double* d_A, double* d_B,
                    double* d_C, double* d_D, double* d_z, double* d_dt_bias);

/* Same gradient by gradient checkpointing: each chunk is recomputed from its
 * checkpoint (as written by oracle_scan_fwd with the same chunk) and walked in
 * reverse, the adjoint carried from chunk to chunk. */
int oracle_scan_bwd_ckpt(const oracle_scan_dims* dm, const double* ckpt, const int* ids,
                         const double* x, const double* dt, const double* A, const double* B,
                         const double* C, const double* D, const double* z, const double* dt_bias,
                         const double* dy, const double* d_state_out,
                         double* d_s0, double* d_x, double* d_dt, double* d_A, double* d_B,
                         double* d_C, double* d_D, double* d_z, double* d_dt_bias);

/* States h_t for every token, [n_s][L][H][P][N], computed by composing the
 * per-step affine maps (a_t, u_t) in a balanced tree instead of left to right. */
int oracle_scan_states_assoc(const oracle_scan_dims* dm, const double* s0, const int* ids,
                             const double* x, const double* dt, const double* A,
                             const double* B, const double* dt_bias, double* states);

#ifdef __cplusplus
}
#endif
#endif

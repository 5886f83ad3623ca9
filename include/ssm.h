/*
 * ssm.h -- C ABI of the GB300 selective-scan library (libssm_gb300.so).
 *
 * What it computes (the diagonal selective state-space scan of Mamba-1, and its
 * scalar-A "Mamba-2 form"), with the causal depthwise conv1d that precedes it:
 *
 *   conv:  out[b][t][d] = act( sum_{k<K} sx[b][d][t+k] * c[d][k] + bias[d] ),  act = SiLU or identity
 *          -- ggmlR tests/testthat/test-ssm-rwkv.R, test "ggml_ssm_conv matches a depthwise
 *             convolution computed in R" (the last tap multiplies the newest input); bias and
 *             SiLU as in infotheory mamba1/model.rs (depthwise_conv_step, then silu).
 *   scan:  delta = dt                       (or softplus(dt + dt_bias), threshold 20, with SSM_DT_SOFTPLUS)
 *          a     = exp(delta * A[h][n])     (A[h] for every n in the scalar-A form)
 *          h_t   = a * h_{t-1} + (delta * x_t) * B_t[n]
 *          y_t   = ( sum_n C_t[n] * h_t[n] + D * x_t ) * silu(z_t)
 *          -- infotheory mamba1/model.rs, selective_scan_state16 and forward_impl; operand shapes
 *             and packing of ggml_ssm_scan in ggmlR test-ssm-rwkv.R (make_scan and the tests
 *             "ggml_ssm_scan packs outputs and states into one flat tensor" / "... views the
 *             trailing states").
 *   backward: the exact reverse-mode gradient (dx, ddt, dA, dB, dC, dD, dz, d dt_bias, dh0)
 *          -- infotheory mamba1/model.rs accumulate_token_step_gradients (per-token adjoint),
 *             kizzasi-model src/backprop_ssm.rs ssm_backward (reverse adjoint scan, initial-state
 *             gradient) and GradientCheckpointedSSM / online_train_segment_tbptt (recompute
 *             from per-chunk checkpoints).
 *
 * Layouts: row-major, slowest index first.  n_s = sequences, L = tokens per sequence,
 * H = heads (= d_inner in the Mamba-1 form), P = head_dim (1 in the Mamba-1 form),
 * N = d_state, G = groups (H % G == 0; head h uses group h / (H/G)), K = d_conv.
 *   sx, d_sx        [n_s][d_inner][K-1+L]   io dtype   (time fastest, ggml layout)
 *   out, dout       [n_s][L][d_inner]       io dtype   (channel fastest)
 *   c, d_c          [d_inner][K]            fp32       bias, d_bias [d_inner] fp32
 *   conv_state_out  [n_s][d_inner][K-1]     io dtype   (the K-1 newest columns of sx)
 *   x, z, y, dy, d_x, d_z  [n_s][L][H][P]   io dtype
 *   dt, d_dt        [n_s][L][H]             io dtype
 *   A, d_A          [H][N] (a_per_state=1) or [H] (a_per_state=0)   fp32
 *   B, C, d_B, d_C  [n_s][L][G][N]          io dtype
 *   D, d_D          [H*P]                   fp32       dt_bias, d_dt_bias [H] fp32
 *   s0, d_s0        [state_rows][H][P][N]   fp32       ids [n_s] int32 (row of s0 per sequence)
 *   state_out, d_state_out [n_s][H][P][N]   fp32
 *   ckpt            [n_s][ceil(L/chunk)][H][P][N] fp32: state at the START of each chunk
 *                   (ckpt[b][0] is the initial state).
 *
 * Ownership: every pointer is a caller-owned DEVICE pointer.  The library allocates,
 * frees and synchronises nothing; work is enqueued on `stream` (a cudaStream_t, passed as
 * void*; NULL = legacy default stream).  Scratch memory is the caller's `ws` buffer of at
 * least the size the *_workspace_size call returns; its contents need not be initialised.
 * Calls that share a workspace must not overlap on the GPU.
 *
 * Errors: argument errors are detected on the host before anything is enqueued and
 * returned synchronously (SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_WORKSPACE).
 * A failed launch returns SSM_ERR_CUDA.  Errors only the device can see (an `ids` entry
 * outside [0, state_rows), or a non-finite output when SSM_CHECK_FINITE is set) are
 * recorded in a status word inside the workspace; the offending element is skipped (an
 * out-of-range row reads as a zero state and receives no gradient), never read or written
 * out of bounds.  Read it with ssm_scan_status after the call.
 * Waits: a block waits only for its own tile copies and, in the persistent backward (see
 * ssm_scan_bwd), for the block that computes the adjoint at the end of its chunk.  Both waits
 * are bounded.  A wait that gives up records SSM_ERR_TIMEOUT; the block then waits (bounded)
 * for its own copies in flight and skips the rest of its work, and every other block gives up
 * at its next wait or unit once the status word is set.  No call can hang.
 */
#ifndef SSM_GB300_H
#define SSM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSM_ABI_VERSION 1

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

enum {
  SSM_OK = 0,
  SSM_ERR_INVALID_ARG = -1, /* null required pointer, size <= 0, H % G != 0, misalignment, bad id */
  SSM_ERR_UNSUPPORTED = -2, /* size beyond a documented limit (d_conv, d_state, element counts) */
  SSM_ERR_WORKSPACE = -3,   /* ws is NULL or smaller than the *_workspace_size result */
  SSM_ERR_CUDA = -4,        /* a kernel launch failed (cudaGetLastError after enqueue) */
  SSM_ERR_TIMEOUT = -5,     /* status word only: a bounded wait gave up (a staged tile that
                               never arrived, or the next chunk's adjoint in the persistent
                               backward); that block skipped the rest of its work, so the
                               call's outputs are incomplete */
  SSM_ERR_NONFINITE = -6    /* SSM_CHECK_FINITE: an output element was NaN or +-Inf */
};

enum {
  SSM_CONV_SILU = 1u,    /* conv: apply SiLU after the convolution (+bias) */
  SSM_DT_SOFTPLUS = 2u,  /* scan: delta = softplus(dt + dt_bias) instead of delta = dt */
  SSM_CHECK_FINITE = 4u, /* scan: record SSM_ERR_NONFINITE in the status word on a non-finite output */
  SSM_A_LOG = 8u,        /* scan: the A argument holds A_log and the scan uses A = -exp(A_log)
                            (infotheory's mamba1 parameterisation); d_A returns dL/dA_log =
                            dL/dA * A.  The workspace grows by a buffer for A: the
                            *_workspace_size results include it; ssm_decode_step then needs
                            ws_bytes >= 256 + 4 * (elements of A) rounded up to 256. */
  SSM_DEBUG_NO_WAIT = 16u, /* scan, for tests of the error path only: every wait of a block on
                             another block gives up at once, as if its bound had run out; the
                             call then records SSM_ERR_TIMEOUT and its outputs are incomplete.
                             Waits for this block's own copies keep their normal bound. */
  SSM_SCAN_CHUNKED = 32u   /* scan forward, Mamba-2 form with bf16 I/O (one A per head, head_dim
                              a multiple of 64, d_state 128, chunk a multiple of 64): compute it
                              in chunked matrix form on the tensor cores (64-token chunks, tf32
                              products with the computed operands split into two terms) instead
                              of as a recurrence.  Same results to bf16 rounding; the workspace
                              then holds every 64-token chunk's state in fp32.  Other shapes
                              ignore the flag.  (ggmlR ssm_scan with a [1, n_head] A; the chunk
                              composition is that of kizzasi's associative scan.) */
};

/* Limits (checked on the host; SSM_ERR_UNSUPPORTED beyond them).  Every tensor must also
 * hold fewer than 2^31 elements per sequence and 2^40 in total. */
#define SSM_MAX_D_CONV 64
#define SSM_MAX_D_STATE 512      /* forward */
#define SSM_MAX_D_STATE_BWD 128  /* backward */

typedef struct {
  int n_seqs;       /* n_s  >= 1 */
  int n_tok;        /* L    >= 1 */
  int n_head;       /* H    >= 1 */
  int head_dim;     /* P    >= 1 */
  int d_state;      /* N    >= 1 */
  int n_group;      /* G    >= 1, H % G == 0 */
  int a_per_state;  /* 1: A is [H][N];  0: A is [H] (one scalar per head, the Mamba-2 form) */
  int state_rows;   /* rows of s0 / d_s0; 0 means n_seqs.  Without ids, must be >= n_seqs */
  int chunk;        /* checkpoint interval in tokens; 0 means 256 */
  int io;           /* ssm_dtype of the activations */
  unsigned flags;   /* SSM_DT_SOFTPLUS | SSM_CHECK_FINITE | SSM_A_LOG | SSM_DEBUG_NO_WAIT |
                       SSM_SCAN_CHUNKED */
} ssm_scan_desc;

/* ---- causal depthwise conv1d (+bias, +SiLU) --------------------------------------------
 * Forward.  sx, out (and conv_state_out when non-NULL) in the io dtype; c, bias fp32.
 * bias may be NULL.  flags: SSM_CONV_SILU.  d_conv <= SSM_MAX_D_CONV. */
int ssm_conv_fwd(const void* sx, const float* c, const float* bias, void* out,
                 void* conv_state_out, int n_s, int d_inner, int n_t, int d_conv, int io,
                 unsigned flags, void* stream);

/* Bytes of scratch ssm_conv_bwd needs (per-tile partial sums of d_c and d_bias); 0 if the
 * sizes are invalid. */
size_t ssm_conv_workspace_size(int n_s, int d_inner, int n_t, int d_conv);

/* Backward (ggmlR's ssm_conv_back, test "ssm_conv gradients match a numeric gradient",
 * extended by the bias and SiLU).  Given dout = dL/dout, writes d_sx (every element,
 * including the K-1 leading state columns), d_c and (when non-NULL) d_bias.  The
 * pre-activation is recomputed from sx, c and bias.  Same flags as the forward.  d_c and
 * d_bias are reduced in a fixed order (bitwise reproducible). */
int ssm_conv_bwd(const void* sx, const float* c, const float* bias, const void* dout,
                 void* d_sx, float* d_c, float* d_bias, void* ws, size_t ws_bytes,
                 int n_s, int d_inner, int n_t, int d_conv, int io, unsigned flags,
                 void* stream);

/* Allocation-free variant of ssm_conv_bwd (no counterpart on the source pages).
 * For callers that cannot allocate device memory -- for example code running where a
 * cudaMalloc is not allowed because it can synchronise the device or block (a host callback,
 * a latency-bound serving loop, a plugin interface), or a process whose device memory is held
 * entirely by another framework's pool.  Same arguments as ssm_conv_bwd without the
 * workspace: the scratch is a fixed array of SSM_NOALLOC_SCRATCH_BYTES in the library's own
 * device memory, which every GPU that loads the library holds until the process exits.
 * Sizes whose scratch (ssm_conv_workspace_size) exceeds it return SSM_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  All calls on a
 * device share the array and it keeps the last call's contents (each call overwrites what it
 * reads), so calls that overlap on the GPU -- on different streams or threads -- race: keep
 * them ordered on one stream.  The looked-up address belongs to the device's current context:
 * calls after cudaDeviceReset (or anything else that replaces the primary context) are not
 * supported.  Allocates and frees nothing. */
#define SSM_NOALLOC_SCRATCH_BYTES (16u << 20)
int ssm_conv_bwd_noalloc(const void* sx, const float* c, const float* bias, const void* dout,
                         void* d_sx, float* d_c, float* d_bias, int n_s, int d_inner, int n_t,
                         int d_conv, int io, unsigned flags, void* stream);

/* ---- selective scan ---------------------------------------------------------------------
 * Which kernels run depends on the shape and the pointers; every combination gives the same
 * results up to summation order.
 *   - Mamba-1 form (head_dim 1, one A per state): TMA-staged kernels when all of these hold:
 *     - the activation pointers (x, dt, B, C, z, y, dy, d_x, d_dt, d_z) are 16-byte aligned;
 *     - a token's row of each (H*P or G*N elements) is a multiple of 16 bytes;
 *     - chunk is a multiple of 16;
 *     - a group's channels fill whole blocks (32 channels for d_state 16).
 *     The forward takes d_state a multiple of 4 up to 256; the backward takes d_state 16.
 *   - Mamba-2 form (one A per head): head-tiled kernels for head_dim a multiple of 64 (forward)
 *     or 32 (backward) with d_state 128.
 *   - Anything else runs the general kernels, which are slower but take any alignment
 *     of the element type and any size within the limits above.
 * Bytes of scratch ssm_scan_fwd (backward = 0) or ssm_scan_bwd (backward = 1) needs for this
 * descriptor on the current device; 0 if the descriptor is invalid.  Always >= 256 (the
 * status word lives there).  The backward size assumes ckpt may be NULL. */
size_t ssm_scan_workspace_size(const ssm_scan_desc* desc, int backward);

/* Forward.  Required: desc, x, dt, A, B, C, y, state_out, ws.  Optional (NULL): s0 (zero
 * initial state), ids (sequence b starts from row b), D, z (no gate), dt_bias (used only with
 * SSM_DT_SOFTPLUS), ckpt (no checkpoints written).  y and state_out are what ggml packs into
 * one tensor [y | final states]; for fp32 io pass y = packed and state_out = packed +
 * n_s*L*H*P to get that packing. */
int ssm_scan_fwd(const ssm_scan_desc* desc, const float* s0, const int32_t* ids, const void* x,
                 const void* dt, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, void* y, float* state_out, float* ckpt,
                 void* ws, size_t ws_bytes, void* stream);

/* Backward.  Inputs as in the forward, plus dy (dL/dy), d_state_out (dL/dstate_out, NULL =
 * zero) and ckpt (the forward's checkpoints for the same desc; NULL = recomputed here from
 * s0, which costs one more forward pass).  Outputs d_x, d_dt, d_A, d_B, d_C are required;
 * d_s0 (rows that no sequence starts from are zeroed; duplicate ids accumulate), d_D
 * (requires D), d_z (requires z) and d_dt_bias (requires SSM_DT_SOFTPLUS) may be NULL.  All
 * outputs are overwritten, none accumulated into.  Reductions run in a fixed order: results
 * are bitwise reproducible from run to run on the same GPU and launch configuration. */
int ssm_scan_bwd(const ssm_scan_desc* desc, const float* s0, const int32_t* ids, const void* x,
                 const void* dt, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, const float* ckpt, const void* dy,
                 const float* d_state_out, float* d_s0, void* d_x, void* d_dt, float* d_A,
                 void* d_B, void* d_C, float* d_D, void* d_z, float* d_dt_bias, void* ws,
                 size_t ws_bytes, void* stream);

/* ---- conv1d + scan in one call ----------------------------------------------------------
 * The Mamba layer's prelude and scan without the conv output x ever reaching memory in the
 * forward: x = act(conv1d(sx) + bias) (act = SiLU with SSM_CONV_SILU) is computed inside the
 * scan kernel from the staged sx columns, as a conv -> silu -> scan per token does in
 * infotheory mamba1/model.rs forward_impl, and as lattice gdn_backward.rs conv1d_silu_fwd feeds
 * its recurrence.  x is rounded to the io type, exactly as ssm_conv_fwd would store it, so the
 * results equal ssm_conv_fwd followed by ssm_scan_fwd (up to summation order).
 *   sx, c, bias, d_conv, conv_flags   as in ssm_conv_fwd, with d_inner = H * P
 *   the scan arguments                as in ssm_scan_fwd, without x
 * When the fused kernel does not apply (it takes the shapes and pointers of the TMA-staged
 * Mamba-1 forward with d_state 16 and d_conv <= 4), x is computed by the conv kernel into the
 * workspace and scanned from there.
 * Workspace: ssm_conv_scan_workspace_size(desc, d_conv, 0) bytes (it includes room for x). */
size_t ssm_conv_scan_workspace_size(const ssm_scan_desc* desc, int d_conv, int backward);
int ssm_conv_scan_fwd(const ssm_scan_desc* desc, int d_conv, unsigned conv_flags, const void* sx,
                      const float* c, const float* bias, const float* s0, const int32_t* ids,
                      const void* dt, const float* A, const void* B, const void* C,
                      const float* D, const void* z, const float* dt_bias, void* y,
                      float* state_out, float* ckpt, void* ws, size_t ws_bytes, void* stream);

/* Backward of ssm_conv_scan_fwd: recomputes x from sx (the conv is not stored by the forward),
 * runs the scan's backward into dL/dx and the conv's backward into d_sx, d_c and (when non-NULL)
 * d_bias.  Scan arguments and outputs as in ssm_scan_bwd (ckpt: the forward's checkpoints, or
 * NULL); d_x is replaced by d_sx [n_s][d_inner][K-1+L].  Workspace:
 * ssm_conv_scan_workspace_size(desc, d_conv, 1) bytes (x, dL/dx and the conv's partial sums
 * live there).  Every output is overwritten; reductions run in a fixed order. */
int ssm_conv_scan_bwd(const ssm_scan_desc* desc, int d_conv, unsigned conv_flags, const void* sx,
                      const float* c, const float* bias, const float* s0, const int32_t* ids,
                      const void* dt, const float* A, const void* B, const void* C,
                      const float* D, const void* z, const float* dt_bias, const float* ckpt,
                      const void* dy, const float* d_state_out, float* d_s0, void* d_sx,
                      float* d_c, float* d_bias, void* d_dt, float* d_A, void* d_B, void* d_C,
                      float* d_D, void* d_z, float* d_dt_bias, void* ws, size_t ws_bytes,
                      void* stream);

/* ---- single-token decode step -----------------------------------------------------------
 * One token per sequence in one launch: the conv ring-state roll, conv1d(+bias, SiLU) of the
 * new input column, and one step of the scan.  This is the per-token loop of infotheory's
 * mamba1 runtime (forward_impl on one token: depthwise_conv_step on its conv ring buffer,
 * then selective_scan_state16 on its recurrent state) and ggml's ssm_conv + ssm_scan with
 * n_seq_tokens = 1 (ggmlR tests).  The results equal ssm_conv_fwd on
 * [conv_state | x_new] (x rounded to the io type as that call stores it) followed by
 * ssm_scan_fwd on one token from `state`.
 *   desc        the scan descriptor with n_tok == 1 (chunk is ignored); d_inner = H*P
 *   d_conv      K (1 .. SSM_MAX_D_CONV); conv_flags: SSM_CONV_SILU
 *   ids         [n_s] int32 or NULL: sequence b uses row ids[b] of conv_state and state (rows
 *               = state_rows, or n_s when 0); the rows of one call must be distinct.  An id
 *               outside [0, rows) is recorded in the status word and that sequence is skipped.
 *   x_new       [n_s][H*P] io: the new pre-conv input column
 *   conv_state  [rows][H*P][K-1] io, in/out (oldest first); may be NULL when K == 1
 *   c, bias     [H*P][K], [H*P] fp32; bias may be NULL
 *   dt [n_s][H], A, B / C [n_s][G][N], D, z [n_s][H*P], dt_bias: as in ssm_scan_fwd
 *   state       [rows][H][P][N] fp32, in/out
 *   y           [n_s][H*P] io, out
 *   ws          >= 256 bytes, 256-byte aligned: the status word (read with ssm_scan_status)
 * Allocates, frees and synchronises nothing. */
int ssm_decode_step(const ssm_scan_desc* desc, int d_conv, unsigned conv_flags,
                    const int32_t* ids, const void* x_new, void* conv_state, const float* c,
                    const float* bias, const void* dt, const float* A, const void* B,
                    const void* C, const float* D, const void* z, const float* dt_bias,
                    float* state, void* y, void* ws, size_t ws_bytes, void* stream);

/* Reads the device status word of the last scan call that used `ws` (waits for `stream`).
 * Writes SSM_OK, SSM_ERR_INVALID_ARG (bad id), SSM_ERR_NONFINITE or SSM_ERR_TIMEOUT to
 * *status and returns SSM_OK; returns SSM_ERR_INVALID_ARG for NULL pointers or SSM_ERR_CUDA.
 * The first error recorded stays until the next call that uses `ws` clears it. */
int ssm_scan_status(const void* ws, int* status, void* stream);

/* Static description of a status code. */
const char* ssm_status_string(int status);

/* SSM_ABI_VERSION of the loaded library. */
int ssm_abi_version(void);

/* Diagnostic: number of kernels this library has enqueued in this process so far (all
 * devices, all streams).  Lets a caller count the launches of a region of its program. */
unsigned long long ssm_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif

"""ctypes binding of libssm_gb300.so (the C ABI of include/ssm.h).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  Tensors must be CUDA tensors, contiguous, of the dtypes the header states
(activations in the I/O dtype, parameters and states fp32).  Work is enqueued on PyTorch's
current stream.  If the library is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssm_gb300.so")

SSM_F32, SSM_BF16 = 0, 1
SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_WORKSPACE = 0, -1, -2, -3
SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_NONFINITE = -4, -5, -6
SSM_CONV_SILU, SSM_DT_SOFTPLUS, SSM_CHECK_FINITE, SSM_A_LOG = 1, 2, 4, 8
SSM_DEBUG_NO_WAIT = 16  # tests of the timeout path only (include/ssm.h)
SSM_SCAN_CHUNKED = 32   # the Mamba-2 form's bf16 forward in chunked matrix form (tensor cores)

EXPORTED = ("ssm_conv_fwd", "ssm_conv_workspace_size", "ssm_conv_bwd", "ssm_scan_workspace_size",
            "ssm_scan_fwd", "ssm_scan_bwd", "ssm_conv_scan_workspace_size", "ssm_conv_scan_fwd",
            "ssm_conv_scan_bwd", "ssm_decode_step", "ssm_scan_status", "ssm_status_string",
            "ssm_abi_version", "ssm_kernel_launches")


class SsmError(RuntimeError):
    def __init__(self, name, code, msg):
        super().__init__(f"{name} failed: {code} ({msg})")
        self.code = code


class ScanDesc(ctypes.Structure):
    _fields_ = [("n_seqs", ctypes.c_int), ("n_tok", ctypes.c_int), ("n_head", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("d_state", ctypes.c_int), ("n_group", ctypes.c_int),
                ("a_per_state", ctypes.c_int), ("state_rows", ctypes.c_int),
                ("chunk", ctypes.c_int), ("io", ctypes.c_int), ("flags", ctypes.c_uint)]


_lib = None
_vp, _sz, _i, _u = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint


def lib():
    """The loaded library (loads on first use; raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m bwd_ssm_conv_gb300.build` "
                "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        L.ssm_conv_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _u, _vp]
        L.ssm_conv_workspace_size.argtypes = [_i, _i, _i, _i]
        L.ssm_conv_workspace_size.restype = _sz
        L.ssm_conv_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i,
                                   _u, _vp]
        L.ssm_scan_workspace_size.argtypes = [ctypes.POINTER(ScanDesc), _i]
        L.ssm_scan_workspace_size.restype = _sz
        L.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanDesc)] + [_vp] * 13 + [_sz, _vp]
        L.ssm_scan_bwd.argtypes = [ctypes.POINTER(ScanDesc)] + [_vp] * 23 + [_sz, _vp]
        L.ssm_decode_step.argtypes = ([ctypes.POINTER(ScanDesc), _i, _u] + [_vp] * 15 +
                                      [_sz, _vp])
        L.ssm_conv_scan_workspace_size.argtypes = [ctypes.POINTER(ScanDesc), _i, _i]
        L.ssm_conv_scan_workspace_size.restype = _sz
        L.ssm_conv_scan_fwd.argtypes = ([ctypes.POINTER(ScanDesc), _i, _u] + [_vp] * 16 +
                                        [_sz, _vp])
        L.ssm_conv_scan_bwd.argtypes = ([ctypes.POINTER(ScanDesc), _i, _u] + [_vp] * 27 +
                                        [_sz, _vp])
        L.ssm_scan_status.argtypes = [_vp, ctypes.POINTER(_i), _vp]
        L.ssm_status_string.argtypes = [_i]
        L.ssm_status_string.restype = ctypes.c_char_p
        L.ssm_abi_version.restype = _i
        L.ssm_kernel_launches.restype = ctypes.c_ulonglong
        _lib = L
    return _lib


def _check(name, rc):
    if rc != SSM_OK:
        raise SsmError(name, rc, lib().ssm_status_string(rc).decode())


def _io_of(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"activations must be float32 or bfloat16, got {t.dtype}")


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _workspace(nbytes, device, ws=None):
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


# ---- conv ---------------------------------------------------------------------------------

def ssm_conv_fwd(sx, c, bias=None, silu=True, want_state=False, out=None, stream=None):
    """out[n_s][n_t][d] = act(sum_k sx[b][d][t+k] c[d][k] + bias[d]); sx is [n_s][d][K-1+n_t]."""
    n_s, d, w = sx.shape
    k = c.shape[1]
    n_t = w - k + 1
    io = _io_of(sx)
    if out is None:
        out = torch.empty(n_s, n_t, d, dtype=sx.dtype, device=sx.device)
    cs = torch.empty(n_s, d, k - 1, dtype=sx.dtype, device=sx.device) if want_state and k > 1 else None
    rc = lib().ssm_conv_fwd(_ptr(sx, name="sx"), _ptr(c, torch.float32, "c"),
                            _ptr(bias, torch.float32, "bias"), _ptr(out, sx.dtype, "out"),
                            _ptr(cs, sx.dtype, "conv_state_out"), n_s, d, n_t, k, io,
                            SSM_CONV_SILU if silu else 0, _stream(stream))
    _check("ssm_conv_fwd", rc)
    return (out, cs) if want_state else out


def ssm_conv_workspace_size(n_s, d_inner, n_t, d_conv) -> int:
    return int(lib().ssm_conv_workspace_size(n_s, d_inner, n_t, d_conv))


def ssm_conv_bwd(sx, c, dout, bias=None, silu=True, want_bias_grad=None, ws=None, out=None,
                 stream=None):
    """Returns (d_sx, d_c, d_bias); d_bias is None unless bias is given or want_bias_grad."""
    n_s, d, w = sx.shape
    k = c.shape[1]
    n_t = w - k + 1
    io = _io_of(sx)
    need = ssm_conv_workspace_size(n_s, d, n_t, k)
    ws = _workspace(need, sx.device, ws)
    if out is None:
        d_sx = torch.empty_like(sx)
        d_c = torch.empty_like(c)
        want_b = want_bias_grad if want_bias_grad is not None else bias is not None
        d_b = torch.empty(d, dtype=torch.float32, device=sx.device) if want_b else None
    else:
        d_sx, d_c, d_b = out
    rc = lib().ssm_conv_bwd(_ptr(sx, name="sx"), _ptr(c, torch.float32, "c"),
                            _ptr(bias, torch.float32, "bias"), _ptr(dout, sx.dtype, "dout"),
                            _ptr(d_sx, sx.dtype, "d_sx"), _ptr(d_c, torch.float32, "d_c"),
                            _ptr(d_b, torch.float32, "d_bias"), _ptr(ws), ws.numel(),
                            n_s, d, n_t, k, io, SSM_CONV_SILU if silu else 0, _stream(stream))
    _check("ssm_conv_bwd", rc)
    return d_sx, d_c, d_b


# ---- scan ---------------------------------------------------------------------------------

@dataclass
class ScanShape:
    n_seqs: int
    n_tok: int
    n_head: int
    head_dim: int
    d_state: int
    n_group: int
    a_per_state: int
    state_rows: int = 0
    chunk: int = 256
    io: int = SSM_F32
    flags: int = 0

    def desc(self) -> ScanDesc:
        return ScanDesc(self.n_seqs, self.n_tok, self.n_head, self.head_dim, self.d_state,
                        self.n_group, self.a_per_state, self.state_rows, self.chunk, self.io,
                        self.flags)

    @property
    def n_chunks(self) -> int:
        return (self.n_tok + self.chunk - 1) // self.chunk


def scan_shape(x, dt, A, B, s0=None, chunk=256, softplus=False, check_finite=False,
               state_rows=0, a_log=False, debug_flags=0, chunked=False) -> ScanShape:
    n_s, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    a_per_state = 1 if A.dim() == 2 else 0
    rows = state_rows if state_rows else (s0.shape[0] if s0 is not None else 0)
    flags = ((SSM_DT_SOFTPLUS if softplus else 0) | (SSM_CHECK_FINITE if check_finite else 0) |
             (SSM_A_LOG if a_log else 0) | (SSM_SCAN_CHUNKED if chunked else 0) | debug_flags)
    return ScanShape(n_s, L, H, P, N, G, a_per_state, rows, chunk, _io_of(x), flags)


def ssm_scan_workspace_size(shape: ScanShape, backward: bool) -> int:
    d = shape.desc()
    return int(lib().ssm_scan_workspace_size(ctypes.byref(d), 1 if backward else 0))


def ssm_scan_fwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, s0=None, ids=None, chunk=256,
                 softplus=False, check_finite=False, want_ckpt=True, state_rows=0, ws=None,
                 out=None, stream=None, a_log=False, chunked=False):
    """Returns (y, state_out, ckpt).  ``out`` = (y, state_out, ckpt) preallocated, optional.
    ``a_log``: A holds A_log (the scan uses -exp(A_log)).  ``chunked``: SSM_SCAN_CHUNKED."""
    sh = scan_shape(x, dt, A, B, s0, chunk, softplus, check_finite, state_rows, a_log,
                    chunked=chunked)
    io = x.dtype
    dev = x.device
    if out is None:
        y = torch.empty_like(x)
        st = torch.empty(sh.n_seqs, sh.n_head, sh.head_dim, sh.d_state, dtype=torch.float32,
                         device=dev)
        ck = (torch.empty(sh.n_seqs, sh.n_chunks, sh.n_head, sh.head_dim, sh.d_state,
                          dtype=torch.float32, device=dev) if want_ckpt else None)
    else:
        y, st, ck = out
    ws = _workspace(ssm_scan_workspace_size(sh, False), dev, ws)
    d = sh.desc()
    rc = lib().ssm_scan_fwd(ctypes.byref(d), _ptr(s0, torch.float32, "s0"),
                            _ptr(ids, torch.int32, "ids"), _ptr(x, io, "x"), _ptr(dt, io, "dt"),
                            _ptr(A, torch.float32, "A"), _ptr(B, io, "B"), _ptr(C, io, "C"),
                            _ptr(D, torch.float32, "D"), _ptr(z, io, "z"),
                            _ptr(dt_bias, torch.float32, "dt_bias"), _ptr(y, io, "y"),
                            _ptr(st, torch.float32, "state_out"), _ptr(ck, torch.float32, "ckpt"),
                            _ptr(ws), ws.numel(), _stream(stream))
    _check("ssm_scan_fwd", rc)
    return y, st, ck


def ssm_decode_step(x_new, conv_state, c, dt, A, B, C, state, bias=None, D=None, z=None,
                    dt_bias=None, ids=None, silu=True, softplus=False, check_finite=False,
                    ws=None, out=None, stream=None, a_log=False):
    """One token per sequence: rolls ``conv_state`` [rows][H*P][K-1] and updates ``state``
    [rows][H][P][N] in place, returns y [n_s][H][P].  x_new [n_s][H][P] (the pre-conv input),
    dt [n_s][H], B / C [n_s][G][N], z [n_s][H][P]; the rest as in ssm_scan_fwd."""
    n_s, H, P = x_new.shape
    rows, _, _, N = state.shape
    G = B.shape[1]
    K = c.shape[1]
    io = x_new.dtype
    dev = x_new.device
    flags = ((SSM_DT_SOFTPLUS if softplus else 0) | (SSM_CHECK_FINITE if check_finite else 0) |
             (SSM_A_LOG if a_log else 0))
    sh = ScanShape(n_s, 1, H, P, N, G, 1 if A.dim() == 2 else 0, rows, 1, _io_of(x_new), flags)
    y = torch.empty_like(x_new) if out is None else out
    ws = _workspace(256 + (-(-4 * A.numel() // 256) * 256 if a_log else 0), dev, ws)
    d = sh.desc()
    rc = lib().ssm_decode_step(ctypes.byref(d), K, SSM_CONV_SILU if silu else 0,
                               _ptr(ids, torch.int32, "ids"), _ptr(x_new, io, "x_new"),
                               _ptr(conv_state, io, "conv_state"), _ptr(c, torch.float32, "c"),
                               _ptr(bias, torch.float32, "bias"), _ptr(dt, io, "dt"),
                               _ptr(A, torch.float32, "A"), _ptr(B, io, "B"), _ptr(C, io, "C"),
                               _ptr(D, torch.float32, "D"), _ptr(z, io, "z"),
                               _ptr(dt_bias, torch.float32, "dt_bias"),
                               _ptr(state, torch.float32, "state"), _ptr(y, io, "y"), _ptr(ws),
                               ws.numel(), _stream(stream))
    _check("ssm_decode_step", rc)
    return y


GRAD_NAMES = ("d_s0", "d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_dt_bias")


def ssm_scan_bwd(x, dt, A, B, C, dy, D=None, z=None, dt_bias=None, s0=None, ids=None, ckpt=None,
                 d_state_out=None, chunk=256, softplus=False, check_finite=False, state_rows=0,
                 want_ds0=True, ws=None, out=None, stream=None, a_log=False, debug_flags=0):
    """Returns a dict keyed by GRAD_NAMES (None where not requested / not applicable).
    ``a_log``: A holds A_log and d_A is dL/dA_log.  ``debug_flags``: SSM_DEBUG_NO_WAIT (tests
    of the timeout path only)."""
    sh = scan_shape(x, dt, A, B, s0, chunk, softplus, check_finite, state_rows, a_log,
                    debug_flags)
    io = x.dtype
    dev = x.device
    if out is None:
        rows = sh.state_rows if sh.state_rows else sh.n_seqs
        g = dict(
            d_s0=(torch.empty(rows, sh.n_head, sh.head_dim, sh.d_state, dtype=torch.float32,
                              device=dev) if want_ds0 else None),
            d_x=torch.empty_like(x), d_dt=torch.empty_like(dt), d_A=torch.empty_like(A),
            d_B=torch.empty_like(B), d_C=torch.empty_like(C),
            d_D=torch.empty_like(D) if D is not None else None,
            d_z=torch.empty_like(z) if z is not None else None,
            d_dt_bias=torch.empty_like(dt_bias) if (dt_bias is not None and softplus) else None)
    else:
        g = out
    ws = _workspace(ssm_scan_workspace_size(sh, True), dev, ws)
    d = sh.desc()
    f32 = torch.float32
    rc = lib().ssm_scan_bwd(
        ctypes.byref(d), _ptr(s0, f32, "s0"), _ptr(ids, torch.int32, "ids"), _ptr(x, io, "x"),
        _ptr(dt, io, "dt"), _ptr(A, f32, "A"), _ptr(B, io, "B"), _ptr(C, io, "C"),
        _ptr(D, f32, "D"), _ptr(z, io, "z"), _ptr(dt_bias, f32, "dt_bias"),
        _ptr(ckpt, f32, "ckpt"), _ptr(dy, io, "dy"), _ptr(d_state_out, f32, "d_state_out"),
        _ptr(g["d_s0"], f32, "d_s0"), _ptr(g["d_x"], io, "d_x"), _ptr(g["d_dt"], io, "d_dt"),
        _ptr(g["d_A"], f32, "d_A"), _ptr(g["d_B"], io, "d_B"), _ptr(g["d_C"], io, "d_C"),
        _ptr(g["d_D"], f32, "d_D"), _ptr(g["d_z"], io, "d_z"), _ptr(g["d_dt_bias"], f32, "d_dt_bias"),
        _ptr(ws), ws.numel(), _stream(stream))
    _check("ssm_scan_bwd", rc)
    g["_ws"] = ws
    return g


# ---- conv1d + scan in one call ------------------------------------------------------------

def conv_scan_shape(sx, c, dt, A, B, s0=None, chunk=256, softplus=False, check_finite=False,
                    state_rows=0, a_log=False) -> ScanShape:
    """The scan descriptor of a fused call: d_inner = sx.shape[1] channels, head_dim 1."""
    n_s, d, w = sx.shape
    L = w - c.shape[1] + 1
    G, N = B.shape[2], B.shape[3]
    rows = state_rows if state_rows else (s0.shape[0] if s0 is not None else 0)
    flags = ((SSM_DT_SOFTPLUS if softplus else 0) | (SSM_CHECK_FINITE if check_finite else 0) |
             (SSM_A_LOG if a_log else 0))
    return ScanShape(n_s, L, d, 1, N, G, 1 if A.dim() == 2 else 0, rows, chunk, _io_of(sx), flags)


def ssm_conv_scan_workspace_size(shape: ScanShape, d_conv: int, backward: bool) -> int:
    d = shape.desc()
    return int(lib().ssm_conv_scan_workspace_size(ctypes.byref(d), d_conv, 1 if backward else 0))


def ssm_conv_scan_fwd(sx, c, dt, A, B, C, bias=None, silu=True, D=None, z=None, dt_bias=None,
                      s0=None, ids=None, chunk=256, softplus=False, check_finite=False,
                      want_ckpt=True, state_rows=0, ws=None, out=None, stream=None, a_log=False):
    """conv1d(+bias, SiLU) of sx fused into the scan forward; returns (y, state_out, ckpt) with
    y [n_s][L][d_inner][1].  sx [n_s][d_inner][K-1+L], c [d_inner][K]; the rest as in
    ssm_scan_fwd with head_dim 1."""
    sh = conv_scan_shape(sx, c, dt, A, B, s0, chunk, softplus, check_finite, state_rows, a_log)
    io, dev, K = sx.dtype, sx.device, c.shape[1]
    if out is None:
        y = torch.empty(sh.n_seqs, sh.n_tok, sh.n_head, 1, dtype=io, device=dev)
        st = torch.empty(sh.n_seqs, sh.n_head, 1, sh.d_state, dtype=torch.float32, device=dev)
        ck = (torch.empty(sh.n_seqs, sh.n_chunks, sh.n_head, 1, sh.d_state, dtype=torch.float32,
                          device=dev) if want_ckpt else None)
    else:
        y, st, ck = out
    ws = _workspace(ssm_conv_scan_workspace_size(sh, K, False), dev, ws)
    d = sh.desc()
    f32 = torch.float32
    rc = lib().ssm_conv_scan_fwd(
        ctypes.byref(d), K, SSM_CONV_SILU if silu else 0, _ptr(sx, io, "sx"), _ptr(c, f32, "c"),
        _ptr(bias, f32, "bias"), _ptr(s0, f32, "s0"), _ptr(ids, torch.int32, "ids"),
        _ptr(dt, io, "dt"), _ptr(A, f32, "A"), _ptr(B, io, "B"), _ptr(C, io, "C"),
        _ptr(D, f32, "D"), _ptr(z, io, "z"), _ptr(dt_bias, f32, "dt_bias"), _ptr(y, io, "y"),
        _ptr(st, f32, "state_out"), _ptr(ck, f32, "ckpt"), _ptr(ws), ws.numel(),
        _stream(stream))
    _check("ssm_conv_scan_fwd", rc)
    return y, st, ck


CONV_SCAN_GRAD_NAMES = ("d_s0", "d_sx", "d_c", "d_bias", "d_dt", "d_A", "d_B", "d_C", "d_D",
                        "d_z", "d_dt_bias")


def ssm_conv_scan_bwd(sx, c, dt, A, B, C, dy, bias=None, silu=True, D=None, z=None,
                      dt_bias=None, s0=None, ids=None, ckpt=None, d_state_out=None, chunk=256,
                      softplus=False, check_finite=False, state_rows=0, want_ds0=True,
                      want_bias_grad=None, ws=None, out=None, stream=None, a_log=False):
    """Backward of ssm_conv_scan_fwd; returns a dict keyed by CONV_SCAN_GRAD_NAMES."""
    sh = conv_scan_shape(sx, c, dt, A, B, s0, chunk, softplus, check_finite, state_rows, a_log)
    io, dev, K = sx.dtype, sx.device, c.shape[1]
    f32 = torch.float32
    if out is None:
        rows = sh.state_rows if sh.state_rows else sh.n_seqs
        want_b = want_bias_grad if want_bias_grad is not None else bias is not None
        g = dict(
            d_s0=(torch.empty(rows, sh.n_head, 1, sh.d_state, dtype=f32, device=dev)
                  if want_ds0 else None),
            d_sx=torch.empty_like(sx), d_c=torch.empty_like(c),
            d_bias=torch.empty(sh.n_head, dtype=f32, device=dev) if want_b else None,
            d_dt=torch.empty_like(dt), d_A=torch.empty_like(A), d_B=torch.empty_like(B),
            d_C=torch.empty_like(C), d_D=torch.empty_like(D) if D is not None else None,
            d_z=torch.empty_like(z) if z is not None else None,
            d_dt_bias=torch.empty_like(dt_bias) if (dt_bias is not None and softplus) else None)
    else:
        g = out
    ws = _workspace(ssm_conv_scan_workspace_size(sh, K, True), dev, ws)
    d = sh.desc()
    rc = lib().ssm_conv_scan_bwd(
        ctypes.byref(d), K, SSM_CONV_SILU if silu else 0, _ptr(sx, io, "sx"), _ptr(c, f32, "c"),
        _ptr(bias, f32, "bias"), _ptr(s0, f32, "s0"), _ptr(ids, torch.int32, "ids"),
        _ptr(dt, io, "dt"), _ptr(A, f32, "A"), _ptr(B, io, "B"), _ptr(C, io, "C"),
        _ptr(D, f32, "D"), _ptr(z, io, "z"), _ptr(dt_bias, f32, "dt_bias"),
        _ptr(ckpt, f32, "ckpt"), _ptr(dy, io, "dy"), _ptr(d_state_out, f32, "d_state_out"),
        _ptr(g["d_s0"], f32, "d_s0"), _ptr(g["d_sx"], io, "d_sx"), _ptr(g["d_c"], f32, "d_c"),
        _ptr(g["d_bias"], f32, "d_bias"), _ptr(g["d_dt"], io, "d_dt"), _ptr(g["d_A"], f32, "d_A"),
        _ptr(g["d_B"], io, "d_B"), _ptr(g["d_C"], io, "d_C"), _ptr(g["d_D"], f32, "d_D"),
        _ptr(g["d_z"], io, "d_z"), _ptr(g["d_dt_bias"], f32, "d_dt_bias"), _ptr(ws), ws.numel(),
        _stream(stream))
    _check("ssm_conv_scan_bwd", rc)
    g["_ws"] = ws
    return g


def ssm_scan_status(ws, stream=None) -> int:
    v = ctypes.c_int(0)
    _check("ssm_scan_status", lib().ssm_scan_status(_ptr(ws), ctypes.byref(v), _stream(stream)))
    return v.value


def ssm_status_string(code: int) -> str:
    return lib().ssm_status_string(code).decode()


def ssm_abi_version() -> int:
    return int(lib().ssm_abi_version())


def ssm_kernel_launches() -> int:
    return int(lib().ssm_kernel_launches())


# ---- ggml packing (ggmlR test-ssm-rwkv.R) --------------------------------------------------

def pack_scan_result(y, state_out):
    """ggml_ssm_scan's single result: [y (nelements(x)) | final states]."""
    return torch.cat([y.reshape(-1).float(), state_out.reshape(-1)])


def pack_scan_grads(g):
    """ggml_ssm_scan_back's result order [d_s | d_x | d_dt | d_A | d_B | d_C]."""
    return torch.cat([g[k].reshape(-1).float() for k in ("d_s0", "d_x", "d_dt", "d_A", "d_B", "d_C")])


def pack_conv_grads(d_sx, d_c):
    """ggml_ssm_conv_back's result order [d_sx | d_c]."""
    return torch.cat([d_sx.reshape(-1).float(), d_c.reshape(-1)])

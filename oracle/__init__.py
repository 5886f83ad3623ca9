"""CPU oracle for the selective scan and the causal depthwise conv1d prelude.

TEST INFRASTRUCTURE ONLY.  The test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package; the product package never does.  The
arithmetic lives in ``ssm_oracle.c`` (plain sequential double-precision loops); this module
only compiles it, converts arrays to float64 and passes pointers.

Every function takes numpy arrays or CPU tensors (any float dtype; converted to float64
exactly) and returns float64 arrays with the layouts documented in ``ssm_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_HDR = os.path.join(_HERE, "ssm_oracle.h")
_LIB_PATH = os.path.join(_HERE, "libssm_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into libssm_oracle.so (no fast-math: IEEE double order kept)."""
    stale = (not os.path.exists(_LIB_PATH) or
             os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [
        ("n_seqs", ctypes.c_int), ("n_tok", ctypes.c_int), ("n_head", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("d_state", ctypes.c_int), ("n_group", ctypes.c_int),
        ("a_per_state", ctypes.c_int), ("state_rows", ctypes.c_int), ("chunk", ctypes.c_int),
        ("dt_softplus", ctypes.c_int),
    ]


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB_PATH)
    return _lib


@dataclass
class ScanDims:
    n_seqs: int
    n_tok: int
    n_head: int
    head_dim: int
    d_state: int
    n_group: int = 1
    a_per_state: int = 1
    state_rows: int = 0
    chunk: int = 256
    dt_softplus: int = 0

    @property
    def rows(self) -> int:
        return self.state_rows if self.state_rows > 0 else self.n_seqs

    @property
    def n_chunks(self) -> int:
        return (self.n_tok + self.chunk - 1) // self.chunk

    def c(self) -> _Dims:
        return _Dims(self.n_seqs, self.n_tok, self.n_head, self.head_dim, self.d_state,
                     self.n_group, self.a_per_state, self.rows, self.chunk, self.dt_softplus)


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _ids(ids):
    if ids is None:
        return None, None
    if hasattr(ids, "detach"):
        ids = ids.detach().cpu().numpy()
    arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    return arr, arr.ctypes.data_as(ctypes.c_void_p)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle {name} failed with status {rc}")


def conv_fwd(sx, c, bias=None, silu=True, want_state=False):
    """out[n_s][n_t][d] = act(sum_k sx[b][d][t+k] * c[d][k] + bias[d]); sx is [n_s][d][n_t+K-1]."""
    lib = _load()
    sx, c, bias = _f64(sx), _f64(c), _f64(bias)
    n_s, d, w = sx.shape
    k = c.shape[1]
    n_t = w - k + 1
    out = np.empty((n_s, n_t, d))
    st = np.empty((n_s, d, k - 1)) if want_state else None
    _check(lib.oracle_conv_fwd(_p(sx), _p(c), _p(bias), _p(out), _p(st), n_s, d, n_t, k,
                               int(silu)), "conv_fwd")
    return (out, st) if want_state else out


def conv_bwd(sx, c, dout, bias=None, silu=True):
    """Returns (d_sx, d_c, d_bias)."""
    lib = _load()
    sx, c, bias, dout = _f64(sx), _f64(c), _f64(bias), _f64(dout)
    n_s, d, w = sx.shape
    k = c.shape[1]
    n_t = w - k + 1
    d_sx = np.empty_like(sx)
    d_c = np.empty_like(c)
    d_b = np.empty(d)
    _check(lib.oracle_conv_bwd(_p(sx), _p(c), _p(bias), _p(dout), _p(d_sx), _p(d_c), _p(d_b),
                               n_s, d, n_t, k, int(silu)), "conv_bwd")
    return d_sx, d_c, d_b


def scan_fwd(dims: ScanDims, x, dt, A, B, C, D=None, z=None, dt_bias=None, s0=None, ids=None,
             want_ckpt=True):
    """Returns (y, state_out, ckpt) with the layouts of ssm_oracle.h."""
    lib = _load()
    x, dt, A, B, C, D, z, dt_bias, s0 = map(_f64, (x, dt, A, B, C, D, z, dt_bias, s0))
    _ids_arr, ids_p = _ids(ids)
    m = dims
    y = np.empty((m.n_seqs, m.n_tok, m.n_head, m.head_dim))
    st = np.empty((m.n_seqs, m.n_head, m.head_dim, m.d_state))
    ck = (np.empty((m.n_seqs, m.n_chunks, m.n_head, m.head_dim, m.d_state))
          if want_ckpt else None)
    cd = m.c()
    _check(lib.oracle_scan_fwd(ctypes.byref(cd), _p(s0), ids_p, _p(x), _p(dt), _p(A), _p(B),
                               _p(C), _p(D), _p(z), _p(dt_bias), _p(y), _p(st), _p(ck)),
           "scan_fwd")
    return y, st, ck


GRAD_ORDER = ("d_s0", "d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_dt_bias")


def _bwd_outputs(m: ScanDims, has_D, has_z, has_bias):
    return dict(
        d_s0=np.empty((m.rows, m.n_head, m.head_dim, m.d_state)),
        d_x=np.empty((m.n_seqs, m.n_tok, m.n_head, m.head_dim)),
        d_dt=np.empty((m.n_seqs, m.n_tok, m.n_head)),
        d_A=np.empty((m.n_head, m.d_state) if m.a_per_state else (m.n_head,)),
        d_B=np.empty((m.n_seqs, m.n_tok, m.n_group, m.d_state)),
        d_C=np.empty((m.n_seqs, m.n_tok, m.n_group, m.d_state)),
        d_D=np.empty((m.n_head * m.head_dim,)) if has_D else None,
        d_z=np.empty((m.n_seqs, m.n_tok, m.n_head, m.head_dim)) if has_z else None,
        d_dt_bias=np.empty((m.n_head,)) if has_bias else None,
    )


def scan_bwd(dims: ScanDims, x, dt, A, B, C, dy, D=None, z=None, dt_bias=None, s0=None, ids=None,
             d_state_out=None, ckpt=None):
    """Exact gradient.  With ``ckpt`` given, uses the chunked recompute (TBPTT) form.

    Returns a dict keyed by GRAD_ORDER (None where the corresponding input is absent)."""
    lib = _load()
    x, dt, A, B, C, D, z, dt_bias, s0, dy, d_state_out, ckpt = map(
        _f64, (x, dt, A, B, C, D, z, dt_bias, s0, dy, d_state_out, ckpt))
    _ids_arr, ids_p = _ids(ids)
    m = dims
    out = _bwd_outputs(m, D is not None, z is not None, dt_bias is not None and m.dt_softplus)
    cd = m.c()
    ptrs = [_p(out[k]) for k in GRAD_ORDER]
    if ckpt is None:
        rc = lib.oracle_scan_bwd(ctypes.byref(cd), _p(s0), ids_p, _p(x), _p(dt), _p(A), _p(B),
                                 _p(C), _p(D), _p(z), _p(dt_bias), _p(dy), _p(d_state_out), *ptrs)
    else:
        rc = lib.oracle_scan_bwd_ckpt(ctypes.byref(cd), _p(ckpt), ids_p, _p(x), _p(dt), _p(A),
                                      _p(B), _p(C), _p(D), _p(z), _p(dt_bias), _p(dy),
                                      _p(d_state_out), *ptrs)
    _check(rc, "scan_bwd")
    return out


def scan_states_assoc(dims: ScanDims, x, dt, A, B, dt_bias=None, s0=None, ids=None):
    """All states h_t, [n_s][L][H][P][N], by balanced-tree composition of the affine steps."""
    lib = _load()
    x, dt, A, B, dt_bias, s0 = map(_f64, (x, dt, A, B, dt_bias, s0))
    _ids_arr, ids_p = _ids(ids)
    m = dims
    st = np.empty((m.n_seqs, m.n_tok, m.n_head, m.head_dim, m.d_state))
    cd = m.c()
    _check(lib.oracle_scan_states_assoc(ctypes.byref(cd), _p(s0), ids_p, _p(x), _p(dt), _p(A),
                                        _p(B), _p(dt_bias), _p(st)), "scan_states_assoc")
    return st

"""The C ABI without a GPU: the library builds and loads, exports exactly the functions
include/ssm.h declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 20  # a non-null, 256-byte-aligned pointer value: never dereferenced by these tests


def _declared():
    names = set()
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ssm_\w+)\s*\(", text,
                                    re.M))
    return names


@pytest.fixture(scope="module")
def L():
    build()
    return binding.lib()


def test_library_exports_every_declared_symbol(L):
    declared = _declared()
    assert declared >= set(binding.EXPORTED)
    for name in declared:
        assert hasattr(L, name), name


def test_abi_version_and_status_strings(L):
    assert binding.ssm_abi_version() == 1
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert binding.ssm_status_string(code)
    assert binding.ssm_status_string(-99) == "unknown status"


def _desc(**kw):
    base = dict(n_seqs=2, n_tok=8, n_head=4, head_dim=1, d_state=16, n_group=1, a_per_state=1,
                state_rows=0, chunk=0, io=0, flags=0)
    base.update(kw)
    return binding.ScanDesc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(n_seqs=0), binding.SSM_ERR_INVALID_ARG),
    (dict(n_tok=-1), binding.SSM_ERR_INVALID_ARG),
    (dict(n_group=3), binding.SSM_ERR_INVALID_ARG),          # H % G != 0
    (dict(io=7), binding.SSM_ERR_INVALID_ARG),
    (dict(flags=64), binding.SSM_ERR_INVALID_ARG),
    (dict(a_per_state=2), binding.SSM_ERR_INVALID_ARG),
    (dict(d_state=513), binding.SSM_ERR_UNSUPPORTED),
    (dict(n_tok=1 << 20, n_head=1 << 12), binding.SSM_ERR_UNSUPPORTED),
])
def test_scan_fwd_rejects_bad_descriptors(L, kw, code):
    d = _desc(**kw)
    args = [ctypes.byref(d), None, None] + [FAKE] * 5 + [None] * 3 + [FAKE, FAKE, None, FAKE,
                                                                       1 << 30, None]
    assert L.ssm_scan_fwd(*args) == code
    assert L.ssm_scan_workspace_size(ctypes.byref(d), 0) == 0


def test_scan_fwd_rejects_null_and_misaligned(L):
    d = _desc()
    good = [ctypes.byref(d), None, None] + [FAKE] * 5 + [None] * 3 + [FAKE, FAKE, None, FAKE,
                                                                       1 << 30, None]
    for i in (3, 4, 5, 6, 7, 11, 12):  # x, dt, A, B, C, y, state_out
        args = list(good)
        args[i] = None
        assert L.ssm_scan_fwd(*args) == binding.SSM_ERR_INVALID_ARG, i
    args = list(good)
    args[3] = FAKE + 2  # x misaligned for fp32
    assert L.ssm_scan_fwd(*args) == binding.SSM_ERR_INVALID_ARG
    # s0 without ids needs state_rows >= n_seqs
    d2 = _desc(state_rows=1)
    args = list(good)
    args[0] = ctypes.byref(d2)
    args[1] = FAKE
    assert L.ssm_scan_fwd(*args) == binding.SSM_ERR_INVALID_ARG


def test_scan_bwd_rejects_bad_arguments(L):
    d = _desc()
    base = ([ctypes.byref(d), None, None] + [FAKE] * 5 + [None, None, None, None, FAKE, None,
                                                          None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                                          None, None, None, FAKE, 1 << 30, None])
    assert len(base) == 26
    # d_state beyond the backward limit
    d_big = _desc(d_state=256)
    args = list(base)
    args[0] = ctypes.byref(d_big)
    assert L.ssm_scan_bwd(*args) == binding.SSM_ERR_UNSUPPORTED
    # d_D without D, d_z without z, d_dt_bias without softplus
    for i in (20, 21, 22):
        args = list(base)
        args[i] = FAKE
        assert L.ssm_scan_bwd(*args) == binding.SSM_ERR_INVALID_ARG, i
    # required outputs
    for i in (12, 15, 16, 17, 18, 19):
        args = list(base)
        args[i] = None
        assert L.ssm_scan_bwd(*args) == binding.SSM_ERR_INVALID_ARG, i


def test_conv_rejects_bad_arguments(L):
    S = binding.SSM_CONV_SILU
    assert L.ssm_conv_fwd(None, FAKE, None, FAKE, None, 1, 4, 8, 4, 0, S, None) == -1
    assert L.ssm_conv_fwd(FAKE, FAKE, None, FAKE, None, 1, 0, 8, 4, 0, S, None) == -1
    assert L.ssm_conv_fwd(FAKE, FAKE, None, FAKE, None, 1, 4, 8, 65, 0, S, None) == -2
    assert L.ssm_conv_fwd(FAKE, FAKE, None, FAKE, None, 1, 4, 8, 4, 0, 8, None) == -1
    assert L.ssm_conv_fwd(FAKE + 2, FAKE, None, FAKE, None, 1, 4, 8, 4, 0, S, None) == -1
    assert L.ssm_conv_workspace_size(1, 4, 8, 4) > 0
    assert L.ssm_conv_workspace_size(1, 4, 8, 0) == 0
    # workspace missing / too small
    assert L.ssm_conv_bwd(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, 0, 1, 4, 8, 4, 0, S,
                          None) == -3
    assert L.ssm_conv_bwd(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, 16, 1, 4, 8, 4, 0, S,
                          None) == -3


def test_status_rejects_null(L):
    v = ctypes.c_int(0)
    assert L.ssm_scan_status(None, ctypes.byref(v), None) == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


def _decode_args(d, K=4, flags=1, **over):
    # desc, d_conv, conv_flags, ids, x_new, conv_state, c, bias, dt, A, B, C, D, z, dt_bias,
    # state, y, ws, ws_bytes, stream
    a = dict(ids=None, x_new=FAKE, conv_state=FAKE, c=FAKE, bias=None, dt=FAKE, A=FAKE, B=FAKE,
             C=FAKE, D=None, z=None, dt_bias=None, state=FAKE, y=FAKE, ws=None, ws_bytes=0)
    a.update(over)
    return [ctypes.byref(d), K, flags, a["ids"], a["x_new"], a["conv_state"], a["c"], a["bias"],
            a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"], a["dt_bias"], a["state"], a["y"],
            a["ws"], a["ws_bytes"], None]


def test_decode_step_rejects_bad_arguments(L):
    one = _desc(n_tok=1)
    INV, UNS, WS = binding.SSM_ERR_INVALID_ARG, binding.SSM_ERR_UNSUPPORTED, binding.SSM_ERR_WORKSPACE
    assert L.ssm_decode_step(*_decode_args(_desc(n_tok=2))) == INV      # one token only
    assert L.ssm_decode_step(*_decode_args(one, K=0)) == INV
    assert L.ssm_decode_step(*_decode_args(one, K=65)) == UNS
    assert L.ssm_decode_step(*_decode_args(one, flags=2)) == INV       # conv flags: SiLU only
    for name in ("x_new", "c", "dt", "A", "B", "C", "state", "y", "conv_state"):
        assert L.ssm_decode_step(*_decode_args(one, **{name: None})) == INV, name
    assert L.ssm_decode_step(*_decode_args(one, x_new=FAKE + 2)) == INV  # misaligned fp32
    assert L.ssm_decode_step(*_decode_args(_desc(n_tok=1, state_rows=1))) == INV  # rows < n_s
    # valid arguments reach the workspace check: K = 1 needs no conv state
    assert L.ssm_decode_step(*_decode_args(one, K=1, conv_state=None)) == WS
    assert L.ssm_decode_step(*_decode_args(one, ws=FAKE, ws_bytes=128)) == WS


def test_conv_workspace_is_one_partial_per_launched_tile(L):
    """d_conv <= 4 runs 256-token tiles, larger d_conv 64-token tiles: one fp32 partial of d_c
    (K values) and d_bias per (sequence, tile, channel), rounded up to 256 bytes."""
    def expect(n_s, d, L_, K, tile):
        n = n_s * (-(-(L_ + K - 1) // tile)) * d * (K + 1) * 4
        return -(-n // 256) * 256
    assert binding.ssm_conv_workspace_size(16, 1024, 4096, 4) == expect(16, 1024, 4096, 4, 256)
    assert binding.ssm_conv_workspace_size(2, 37, 130, 3) == expect(2, 37, 130, 3, 256)
    assert binding.ssm_conv_workspace_size(2, 37, 130, 9) == expect(2, 37, 130, 9, 64)
    assert binding.ssm_conv_workspace_size(0, 37, 130, 4) == 0


def test_conv_scan_rejects_bad_arguments(L):
    """The fused conv + scan calls check their conv arguments on the host, like ssm_conv_fwd."""
    d = _desc()
    p = ctypes.c_void_p(FAKE)
    assert binding.lib().ssm_conv_scan_workspace_size(ctypes.byref(d), 0, 0) == 0
    assert binding.lib().ssm_conv_scan_workspace_size(ctypes.byref(d), 65, 1) == 0

    def fwd(K=4, flags=1, sx=p, c=p, dt=p, y=p):
        return binding.lib().ssm_conv_scan_fwd(ctypes.byref(d), K, flags, sx, c, None, None, None,
                                               dt, p, p, p, None, None, None, y, p, None, p,
                                               1 << 30, None)
    assert fwd(K=0) == binding.SSM_ERR_INVALID_ARG
    assert fwd(K=65) == binding.SSM_ERR_UNSUPPORTED
    assert fwd(flags=2) == binding.SSM_ERR_INVALID_ARG
    assert fwd(sx=None) == binding.SSM_ERR_INVALID_ARG
    assert fwd(c=None) == binding.SSM_ERR_INVALID_ARG
    assert fwd(dt=None) == binding.SSM_ERR_INVALID_ARG
    assert fwd(y=None) == binding.SSM_ERR_INVALID_ARG
    assert fwd(sx=ctypes.c_void_p(FAKE + 1)) == binding.SSM_ERR_INVALID_ARG  # misaligned fp32

    names = ("sx c bias s0 ids dt A B C D z dt_bias ckpt dy d_state_out d_s0 d_sx d_c d_bias "
             "d_dt d_A d_B d_C d_D d_z d_dt_bias").split()
    required = set("sx c dt A B C dy d_sx d_c d_dt d_A d_B d_C".split())

    def bwd(ws_bytes=1 << 30, **override):
        args = [override.get(n, p if n in required else None) for n in names]
        return binding.lib().ssm_conv_scan_bwd(ctypes.byref(d), 4, 1, *args, p, ws_bytes, None)
    assert bwd(d_sx=None) == binding.SSM_ERR_INVALID_ARG
    assert bwd(d_c=None) == binding.SSM_ERR_INVALID_ARG

"""ssm_conv_bwd_noalloc: the conv backward for callers that cannot allocate device memory.

Such callers (code where a cudaMalloc may not run because it can synchronise the device or
block, or whose device memory is all held by another framework's pool) get the same result
as ssm_conv_bwd without passing a workspace.  This test calls the new entry point through
the C ABI twice in a row, on different inputs, and compares each result with the regular
entry point's.  It lives in a file of its own that runs last, and passes both alone in a
fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import random_conv_inputs

pytestmark = pytest.mark.gpu


def _noalloc(lib, sx, c, bias, dout, silu, out):
    fn = lib.ssm_conv_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [ctypes.c_uint, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    n_s, d, w = sx.shape
    k = c.shape[1]
    d_sx, d_c, d_b = out
    return fn(sx.data_ptr(), c.data_ptr(), bias.data_ptr() if bias is not None else None,
              dout.data_ptr(), d_sx.data_ptr(), d_c.data_ptr(),
              d_b.data_ptr() if d_b is not None else None, n_s, d, w - k + 1, k,
              binding.SSM_BF16 if sx.dtype == torch.bfloat16 else binding.SSM_F32,
              binding.SSM_CONV_SILU if silu else 0, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_noalloc_matches_regular_entry_point_twice(io):
    lib = binding.lib()
    for seed, (n_s, d, L, K, bias) in enumerate([(2, 37, 130, 4, True), (3, 64, 300, 3, False)]):
        inp = random_conv_inputs(n_s, d, L, K, io=io, bias=bias, seed=100 + seed)
        sx, c, dout = inp["sx"].cuda(), inp["c"].cuda(), inp["dout"].cuda()
        bv = inp["bias"].cuda() if bias else None
        ref = binding.ssm_conv_bwd(sx, c, dout, bv, silu=True, want_bias_grad=True)
        out = (torch.full_like(sx, float("nan")), torch.full_like(c, float("nan")),
               torch.full((d,), float("nan"), device="cuda"))
        rc = _noalloc(lib, sx, c, bv, dout, True, out)
        assert rc == binding.SSM_OK, binding.ssm_status_string(rc)
        torch.cuda.synchronize()
        # the same kernels with the same fixed-order reduction: bitwise equal
        for name, got, want in zip(("d_sx", "d_c", "d_bias"), out, ref):
            assert torch.equal(got.cpu(), want.cpu()), name


def test_noalloc_takes_a_shape_whose_scratch_fits():
    """16 sequences x 1024 channels x 4096 tokens with d_conv 4 needs about 5.6 MB of partial
    sums (one per 256-token tile), within the 16 MiB array."""
    lib = binding.lib()
    n_s, d, L, K = 16, 1024, 4096, 4
    need = binding.ssm_conv_workspace_size(n_s, d, L, K)
    assert need <= 16 << 20
    inp = random_conv_inputs(n_s, d, L, K, io="bf16", bias=True, seed=7)
    sx, c, dout = inp["sx"].cuda(), inp["c"].cuda(), inp["dout"].cuda()
    bv = inp["bias"].cuda()
    ref = binding.ssm_conv_bwd(sx, c, dout, bv, silu=True, want_bias_grad=True)
    out = (torch.empty_like(sx), torch.empty_like(c), torch.empty(d, device="cuda"))
    rc = _noalloc(lib, sx, c, bv, dout, True, out)
    assert rc == binding.SSM_OK, binding.ssm_status_string(rc)
    torch.cuda.synchronize()
    for name, got, want in zip(("d_sx", "d_c", "d_bias"), out, ref):
        assert torch.equal(got.cpu(), want.cpu()), name


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = binding.lib()
    x = torch.zeros(1, device="cuda")
    # 64 sequences x 4096 channels x 4096 tokens needs far more than the 16 MiB scratch
    need = binding.ssm_conv_workspace_size(64, 4096, 4096, 4)
    assert need > 16 << 20
    fn = lib.ssm_conv_bwd_noalloc
    fn.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [ctypes.c_uint, ctypes.c_void_p]
    p = x.data_ptr()
    assert fn(p, p, None, p, p, p, None, 64, 4096, 4096, 4, 0, 1, None) == \
        binding.SSM_ERR_UNSUPPORTED

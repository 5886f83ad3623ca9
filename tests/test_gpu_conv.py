"""GPU parity of the causal depthwise conv1d (+bias, +SiLU) forward and backward."""
import pytest
import torch

import oracle
from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import make_inputs, random_conv_inputs, workload
from gpu_util import assert_close, nan_like, tol

pytestmark = pytest.mark.gpu

# n_s, d_inner, n_t, d_conv, io, bias, silu
CASES = [
    (1, 16, 64, 4, "f32", False, True),     # the tiny workload's shape
    (2, 37, 130, 3, "f32", True, True),     # ragged channels and time
    (3, 33, 65, 1, "f32", False, False),    # K = 1
    (2, 64, 200, 7, "bf16", True, True),
    (1, 5, 2, 4, "f32", True, True),        # L < K
    (2, 40, 300, 64, "f32", True, True),    # the largest supported K
    (3, 45, 513, 4, "bf16", True, True),    # 256-token tiles: 3 tiles, ragged channels
    (2, 32, 512, 4, "bf16", False, True),   # L a multiple of the tile: a tail tile of K-1 columns
    (2, 19, 300, 2, "bf16", True, False),   # K = 2 without SiLU
    (1, 64, 256, 4, "f32", True, True),     # one full tile, fp32
    (4, 7, 777, 3, "f32", False, True),     # rows of every alignment, several tiles
]


def _run(n_s, d, L, K, io, bias, silu, seed):
    inp = random_conv_inputs(n_s, d, L, K, io=io, bias=bias, seed=seed)
    sx, c = inp["sx"].cuda(), inp["c"].cuda()
    bv = inp["bias"].cuda() if bias else None
    # NaN-filled outputs: an element the kernels never write fails the check
    out, cs = binding.ssm_conv_fwd(sx, c, bv, silu=silu, want_state=True,
                                   out=nan_like(sx, (n_s, L, d)))
    ref, cs_ref = oracle.conv_fwd(inp["sx"], inp["c"], inp["bias"], silu=silu, want_state=True)
    assert_close("out", out, ref, tol(io, False))
    if K > 1:
        assert torch.equal(cs.cpu(), inp["sx"][:, :, -(K - 1):])
    d_sx, d_c, d_b = binding.ssm_conv_bwd(sx, c, inp["dout"].cuda(), bv, silu=silu,
                                          out=(nan_like(sx), nan_like(c),
                                               nan_like(None, (d,), torch.float32)))
    r_sx, r_c, r_b = oracle.conv_bwd(inp["sx"], inp["c"], inp["dout"], bias=inp["bias"], silu=silu)
    assert_close("d_sx", d_sx, r_sx, tol(io, True))
    assert_close("d_c", d_c, r_c, tol(io, True))
    assert_close("d_bias", d_b, r_b, tol(io, True))
    return d_sx, d_c, d_b


@pytest.mark.parametrize("case", CASES)
def test_conv_parity(case):
    _run(*case, seed=sum(case[:4]))


def test_conv_bwd_deterministic():
    a = _run(2, 37, 130, 3, "f32", True, True, seed=3)
    b = _run(2, 37, 130, 3, "f32", True, True, seed=3)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("name", ["mamba1_tiny_f32_b1_l64_d16_n4",
                                  "mamba1_layer_f32_b8_l1024_d512_n16",
                                  "mamba1_long_bf16_b1_l16384_d2048_n16",
                                  "mamba1_train_bf16_b16_l2048_d1536_n16"])
def test_conv_full_workload(name):
    w = workload(name)
    inp = make_inputs(w)
    sx, c = inp["sx"].cuda(), inp["c"].cuda()
    out = binding.ssm_conv_fwd(sx, c, None, silu=True,
                               out=nan_like(sx, (w.n_seqs, w.n_tok, w.channels)))
    ref = oracle.conv_fwd(inp["sx"], inp["c"], None, silu=True)
    assert_close("out", out, ref, tol(w.io, False))
    dout = inp["dy"].view(w.n_seqs, w.n_tok, w.channels)
    d_sx, d_c, _ = binding.ssm_conv_bwd(sx, c, dout.cuda(), None, silu=True,
                                        out=(nan_like(sx), nan_like(c), None))
    r_sx, r_c, _ = oracle.conv_bwd(inp["sx"], inp["c"], dout, silu=True)
    assert_close("d_sx", d_sx, r_sx, tol(w.io, True))
    assert_close("d_c", d_c, r_c, tol(w.io, True))


def _at(t, off):
    """A CUDA copy of t that starts `off` elements into its buffer."""
    flat = torch.empty(t.numel() + off, dtype=t.dtype, device="cuda")
    v = flat[off:].view(t.shape)
    v.copy_(t.cuda())
    return v


# (io, sx offset, d_sx offset, dout offset) in elements.  sx and d_sx rows in different 16-byte
# phases take the general kernel; the same non-zero phase takes the row kernel with shifted
# row starts; an unaligned dout is staged element by element.
OFFSET_CASES = [
    ("bf16", 1, 0, 0),
    ("bf16", 3, 3, 1),
    ("f32", 2, 2, 0),
    ("f32", 0, 1, 3),
]


@pytest.mark.parametrize("case", OFFSET_CASES)
def test_conv_bwd_offset_views(case):
    io, o_sx, o_dsx, o_dout = case
    n_s, d, L, K = 2, 40, 300, 4
    inp = random_conv_inputs(n_s, d, L, K, io=io, bias=True, seed=17 + o_sx + o_dsx)
    sx, dout = _at(inp["sx"], o_sx), _at(inp["dout"], o_dout)
    d_sx = _at(torch.full_like(inp["sx"], float("nan")), o_dsx)
    d_c = nan_like(inp["c"])
    d_b = nan_like(None, (d,), torch.float32)
    binding.ssm_conv_bwd(sx, inp["c"].cuda(), dout, inp["bias"].cuda(), silu=True,
                         out=(d_sx, d_c, d_b))
    r_sx, r_c, r_b = oracle.conv_bwd(inp["sx"], inp["c"], inp["dout"], bias=inp["bias"], silu=True)
    assert_close("d_sx", d_sx, r_sx, tol(io, True))
    assert_close("d_c", d_c, r_c, tol(io, True))
    assert_close("d_bias", d_b, r_b, tol(io, True))

"""The Mamba-2 form's forward on the tensor cores (SSM_SCAN_CHUNKED; bf16 I/O, one A per head,
head_dim a multiple of 64, d_state 128, checkpoint interval a multiple of 64): y, the final state
and the checkpoints against the oracle's sequential recurrence, at the bf16 gate.

The chunked form composes the recurrence over 64-token chunks exactly (products of the affine
steps); its computed operands enter the tf32 products as two tf32 terms each, so it matches the
oracle to bf16 rounding, not bitwise.
Cases cover one chunk and many, a ragged last chunk, checkpoints every 64 / 128 / 256 tokens,
the gate z and skip D, softplus with dt_bias (large decays), groups, start states selected by ids,
and two 64-channel blocks per head."""
import numpy as np
import pytest
import torch

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import random_scan_inputs
from gpu_util import assert_close, gpu_bwd, gpu_fwd, oracle_bwd, oracle_fwd, tol

pytestmark = pytest.mark.gpu

# name, (ns, L, H, P, N, G), chunk, softplus, has_z, has_D, ids
CASES = [
    ("one_chunk", (3, 64, 2, 64, 128, 1), 64, False, True, True, False),
    ("ragged_gate_skip", (2, 200, 3, 64, 128, 1), 64, False, True, True, False),
    ("softplus_groups", (1, 130, 4, 128, 128, 2), 128, True, False, True, False),
    ("ids_chunk256", (3, 300, 2, 64, 128, 1), 256, False, False, False, True),
    ("long", (1, 1000, 2, 64, 128, 1), 128, False, True, False, False),
]


def _inputs(case, seed):
    name, shape, chunk, softplus, has_z, has_D, ids = case
    ns, L, H, P, N, G = shape
    inp = random_scan_inputs(ns, L, H, P, N, n_group=G, io="bf16", scalar_a=True, has_z=has_z,
                             has_D=has_D, seed=seed, dt_raw=softplus)
    if softplus:
        inp["dt_bias"] = torch.linspace(-0.5, 0.5, H).float()
    return inp


def test_tensor_core_path_applies_to_these_shapes():
    """With SSM_SCAN_CHUNKED each case's workspace holds the chunk states [ns][H][L/64][P][128]
    in fp32, which only the tensor-core path keeps."""
    for case in CASES:
        name, shape, chunk = case[0], case[1], case[2]
        ns, L, H, P, N, G = shape
        x = torch.empty(ns, L, H, P, dtype=torch.bfloat16)
        dt = torch.empty(ns, L, H, dtype=torch.bfloat16)
        A = torch.empty(H)
        B = torch.empty(ns, L, G, N, dtype=torch.bfloat16)
        need = ns * H * ((L + 63) // 64) * P * N * 4
        sh = binding.scan_shape(x, dt, A, B, None, chunk, chunked=True)
        assert binding.ssm_scan_workspace_size(sh, False) >= need, name


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tensor_core_forward_matches_the_recurrence_oracle(case):
    name, shape, chunk, softplus, has_z, has_D, use_ids = case
    inp = _inputs(case, 70 + len(name))
    ids = None
    if use_ids:
        ids = torch.tensor(list(reversed(range(shape[0]))), dtype=torch.int32)
    y, st, ck = gpu_fwd(inp, chunk, softplus, ids=ids, chunked=True)
    yo, so, co = oracle_fwd(inp, chunk, softplus, ids=ids)
    t = tol("bf16", grad=False)
    assert_close("y", y, yo, t)
    assert_close("state_out", st, so, t)
    assert_close("ckpt", ck, co, t)


def test_backward_from_tensor_core_checkpoints():
    """The backward recomputes from the checkpoints the tensor-core forward wrote."""
    case = CASES[1]
    inp = _inputs(case, 91)
    _, _, ck = gpu_fwd(inp, case[2], case[3], chunked=True)
    g = gpu_bwd(inp, case[2], ckpt=ck, softplus=case[3])
    o = oracle_bwd(inp, case[2], case[3])
    t = tol("bf16", grad=True)
    for k in ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0"):
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], t)


def test_tensor_core_forward_is_deterministic():
    case = CASES[2]
    inp = _inputs(case, 5)
    a = gpu_fwd(inp, case[2], case[3], chunked=True)
    b = gpu_fwd(inp, case[2], case[3], chunked=True)
    for name, u, v in zip(("y", "state_out", "ckpt"), a, b):
        assert torch.equal(u.cpu(), v.cpu()), name

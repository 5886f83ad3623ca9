"""SSM_A_LOG: A passed as A_log with A = -exp(A_log) (infotheory's mamba1 parameterisation).
Forward outputs equal the oracle's with that A; the backward's d_A is dL/dA_log = dL/dA * A; the
decode step agrees with the plain-A call."""
import numpy as np
import pytest
import torch

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import random_scan_inputs
from gpu_util import assert_close, cuda, oracle_bwd, oracle_fwd, tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,io,scalar_a,chunk", [
    ((2, 100, 64, 1, 16, 1), "bf16", False, 16),   # Mamba-1 layout (TMA paths)
    ((2, 80, 4, 8, 32, 2), "f32", True, 16),       # Mamba-2 form, two groups
])
def test_a_log_forward_and_gradient(shape, io, scalar_a, chunk):
    ns, L, H, P, N, G = shape
    inp = random_scan_inputs(ns, L, H, P, N, n_group=G, io=io, scalar_a=scalar_a, seed=41,
                             has_z=not scalar_a, has_D=not scalar_a)
    a_log = torch.log(-inp["A"].double()).float()          # the parameter the caller holds
    ref = dict(inp)
    ref["A"] = -torch.exp(a_log.double())                   # the A the scan must use
    d = cuda(inp)
    y, st, ck = binding.ssm_scan_fwd(d["x"], d["dt"], a_log.cuda(), d["B"], d["C"], D=d.get("D"),
                                     z=d.get("z"), s0=d.get("s0"), chunk=chunk, a_log=True)
    yo, so, _ = oracle_fwd(ref, chunk)
    t = tol(io, grad=False)
    assert_close("y", y, yo, t)
    assert_close("state_out", st, so, t)
    g = binding.ssm_scan_bwd(d["x"], d["dt"], a_log.cuda(), d["B"], d["C"], d["dy"],
                             D=d.get("D"), z=d.get("z"), s0=d.get("s0"), ckpt=ck,
                             d_state_out=d["d_state_out"], chunk=chunk, a_log=True)
    o = oracle_bwd(ref, chunk)
    tg = tol(io, grad=True)
    assert_close("d_A_log", g["d_A"], np.asarray(o["d_A"]) * ref["A"].numpy(), tg)
    assert_close("d_x", g["d_x"], o["d_x"], tg)
    assert binding.ssm_scan_status(g["_ws"]) == 0


def test_a_log_decode_step_matches_plain_a():
    ns, H, N, K = 3, 32, 16, 4
    sc = random_scan_inputs(ns, 1, H, 1, N, io="f32", seed=42)
    a_log = torch.log(-sc["A"]).float().cuda()
    a = (-torch.exp(a_log.double())).float()
    g = torch.Generator().manual_seed(43)
    cs0 = torch.randn(ns, H, K - 1, generator=g).cuda()
    x_new = torch.randn(ns, H, 1, generator=g).cuda()
    c = (torch.rand(H, K, generator=g) - 0.5).cuda()
    args = dict(dt=sc["dt"][:, 0].contiguous().cuda(), B=sc["B"][:, 0].contiguous().cuda(),
                C=sc["C"][:, 0].contiguous().cuda())
    outs = []
    for A, flag in ((a, False), (a_log, True)):
        cs, st = cs0.clone(), sc["s0"].clone().cuda()
        y = binding.ssm_decode_step(x_new, cs, c, args["dt"], A, args["B"], args["C"], st,
                                    a_log=flag)
        outs.append((y, st))
    torch.cuda.synchronize()
    assert_close("y", outs[1][0], outs[0][0].cpu().numpy(), 1e-5)
    assert_close("state", outs[1][1], outs[0][1].cpu().numpy(), 1e-5)

"""GPU parity of the selective scan (forward and backward) against the f64 oracle.

Small cases span several blocks, several time segments and ragged tails (tokens not a
multiple of the chunk or of the 8-token sub-chunk, channels not a multiple of the block,
padded state counts); the benchmark configurations run at full size with the oracle on
sampled channels; dB / dC at full size use an upstream gradient that is non-zero on the
sampled channels only, so that the oracle's subset sums are exact.
"""
import zlib

import numpy as np
import pytest
import torch

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import make_inputs, random_scan_inputs, workload
from gpu_util import (assert_close, channel_subset, gpu_bwd, gpu_fwd, oracle_bwd, oracle_fwd, tol)

pytestmark = pytest.mark.gpu

GRADS = ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0", "d_dt_bias")

# name, shape (ns, L, H, P, N, G), io, scalar_a, chunk, softplus, with ids
CASES = [
    ("cfg0_shape", (1, 64, 16, 1, 4, 1), "f32", False, 16, False, False),
    ("multiseg_ragged", (2, 1000, 24, 1, 16, 1), "f32", False, 100, False, False),
    ("padded_groups_ids_softplus", (3, 77, 6, 2, 3, 3), "f32", False, 16, True, True),
    ("mamba2_form", (2, 300, 4, 8, 32, 2), "f32", True, 64, False, False),
    ("bf16", (2, 333, 48, 1, 16, 1), "bf16", False, 128, False, False),
    ("n24_padded", (1, 50, 8, 1, 24, 1), "f32", False, 7, False, False),
    ("big_chunk_rechunked", (1, 1300, 5, 1, 16, 1), "f32", False, 600, False, False),
    ("single_token", (2, 1, 3, 1, 16, 1), "f32", False, 256, False, False),
    ("n128_mamba2", (1, 40, 2, 4, 128, 1), "f32", True, 16, False, False),
    # shapes that take the TMA-staged kernels (channels a multiple of 32, d_state 16)
    # (the backward's TMA kernel takes groups of a multiple of 32 channels and chunks of a
    # multiple of 16 tokens; a 24-token chunk runs its general kernels)
    ("tma_f32_ragged_multiseg", (2, 300, 64, 1, 16, 1), "f32", False, 64, False, False),
    ("tma_bf16_softplus", (3, 520, 128, 1, 16, 1), "bf16", False, 128, True, False),
    ("tma_chunk24_tile8", (1, 200, 32, 1, 16, 1), "f32", False, 24, False, False),
    ("tma_groups", (2, 100, 64, 1, 16, 2), "bf16", False, 32, False, False),
    ("tma_groups64_chunk48", (2, 200, 128, 1, 16, 2), "bf16", False, 48, False, False),
    ("tma_f32_pieces", (2, 333, 64, 1, 16, 1), "f32", False, 208, True, False),
    # Mamba-2 form (one A per head) with several heads per channel block, two groups
    ("mamba2_f32_heads", (2, 200, 16, 8, 32, 2), "f32", True, 32, False, False),
    # ... bf16 with softplus(dt + dt_bias)
    ("mamba2_bf16_softplus", (2, 160, 8, 16, 64, 1), "bf16", True, 32, True, False),
    # Mamba-2 form on the head-tiled forward: head_dim 64, d_state 128, two groups, 4 segments
    ("mh_f32_groups_segments", (2, 200, 4, 64, 128, 2), "f32", True, 32, False, False),
    # ... bf16 with softplus, head_dim 128 (two blocks per head)
    ("mh_bf16_softplus_p128", (1, 100, 8, 128, 128, 1), "bf16", True, 16, True, False),
    # TMA forward with fp32 I/O and one A per channel (head_dim 1), softplus, several segments
    ("tma_f32_scalar_a_softplus", (2, 400, 64, 1, 16, 1), "f32", True, 32, True, False),
    # TMA forward, bf16, one A per channel, d_state 64 (16 states x 4 threads per channel)
    ("tma_bf16_scalar_a_n64", (3, 130, 32, 1, 64, 1), "bf16", True, 16, False, False),
]


def _inputs(shape, io, scalar_a, softplus, seed):
    ns, L, H, P, N, G = shape
    inp = random_scan_inputs(ns, L, H, P, N, n_group=G, io=io, scalar_a=scalar_a, seed=seed,
                             dt_raw=softplus, has_z=not scalar_a, has_D=not scalar_a)
    if softplus:
        inp["dt_bias"] = torch.linspace(-0.5, 0.5, H).float()
    return inp


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_scan_forward_parity(case):
    name, shape, io, scalar_a, chunk, softplus, with_ids = case
    inp = _inputs(shape, io, scalar_a, softplus, seed=zlib.crc32(name.encode()) % 1000)
    ids, rows = None, 0
    if with_ids:
        rows = shape[0] + 2
        inp["s0"] = torch.randn(rows, shape[2], shape[3], shape[4]).float()
        ids = torch.tensor([rows - 1, 0, rows - 1][:shape[0]], dtype=torch.int32)
    y, st, ck = gpu_fwd(inp, chunk, softplus, ids, rows)
    yo, so, co = oracle_fwd(inp, chunk, softplus, ids, rows)
    t = tol(io, grad=False)
    assert_close("y", y, yo, t)
    assert_close("state_out", st, so, t)
    assert_close("ckpt", ck, co, t)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_scan_backward_parity(case):
    name, shape, io, scalar_a, chunk, softplus, with_ids = case
    inp = _inputs(shape, io, scalar_a, softplus, seed=zlib.crc32(name.encode()) % 1000 + 1)
    ids, rows = None, 0
    if with_ids:
        rows = shape[0] + 2
        inp["s0"] = torch.randn(rows, shape[2], shape[3], shape[4]).float()
        ids = torch.tensor([rows - 1, 0, rows - 1][:shape[0]], dtype=torch.int32)
    _, _, ck = gpu_fwd(inp, chunk, softplus, ids, rows)
    g = gpu_bwd(inp, chunk, ckpt=ck, softplus=softplus, ids=ids, state_rows=rows)
    o = oracle_bwd(inp, chunk, softplus, ids, rows)
    t = tol(io, grad=True)
    for k in GRADS:
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], t)
    assert binding.ssm_scan_status(g["_ws"]) == 0


THRESHOLD_SHAPES = [  # (ns, L, H, P, N, G), one A per head
    ((2, 96, 64, 1, 16, 1), False),     # Mamba-1 layout: the TMA kernels
    ((1, 80, 4, 64, 128, 1), True),     # Mamba-2 form: the head-tiled kernels
]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape_sa", THRESHOLD_SHAPES, ids=["mamba1", "mamba2"])
def test_softplus_threshold_parity(io, shape_sa):
    """dt biases near 20 put the softplus pre-activations of some channels on both sides of the
    threshold (identity and derivative 1 above it) and make their decays tiny; forward and
    gradients match the oracle."""
    shape, scalar_a = shape_sa
    inp = _inputs(shape, io, scalar_a, True, seed=97)
    H = shape[2]
    inp["dt_bias"] = torch.tensor([(20.2, 19.8, 0.1, 20.6)[c % 4] for c in range(H)]).float()
    pre = inp["dt"].float() + inp["dt_bias"]
    assert bool((pre > 20).any()) and bool(((pre <= 20) & (inp["dt_bias"] > 19)).any())
    y, st, ck = gpu_fwd(inp, 32, True)
    yo, so, co = oracle_fwd(inp, 32, True)
    t = tol(io, grad=False)
    assert_close("y", y, yo, t)
    assert_close("state_out", st, so, t)
    g = gpu_bwd(inp, 32, ckpt=ck, softplus=True)
    o = oracle_bwd(inp, 32, True)
    t = tol(io, grad=True)
    for k in GRADS:
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], t)
    assert binding.ssm_scan_status(g["_ws"]) == 0


# Enough (sequence, 32-channel block) chains to fill a 152-SM GPU without time segments (40 x 32
# = 1280 chains, 4 resident blocks per SM): the backward then runs resident blocks over (chain,
# chunk) units, last chunk first, each handing its chunk's start adjoint to the unit of the
# chunk before it.  Ragged last chunk.  22 x 32 = 704 chains fill 3/4 of the 608 resident
# blocks but not all: also persistent, with some blocks waiting on the flag of a chunk still in
# progress.  The dB/dC reduction items share the unit queue: chunk counts 2 and 3 put all of
# them at its end, 4, 5 and 10 interleave them with the units of earlier chunks (10: a ragged
# last chunk and two 32-token items per chunk).
PERSIST_CASES = [
    ("persist_bf16", (40, 100, 1024, 1, 16, 1), "bf16", 32, False),
    ("persist_f32_softplus", (24, 72, 1024, 1, 16, 1), "f32", 16, True),
    ("persist_partial_bf16", (22, 100, 1024, 1, 16, 1), "bf16", 32, False),
    ("persist_pieces_bf16", (24, 300, 1024, 1, 16, 1), "bf16", 144, False),
    ("persist_two_chunks_bf16", (40, 64, 1024, 1, 16, 1), "bf16", 32, False),
    ("persist_ten_chunks_bf16", (24, 600, 1024, 1, 16, 1), "bf16", 64, False),
]


@pytest.mark.parametrize("case", PERSIST_CASES, ids=[c[0] for c in PERSIST_CASES])
def test_persistent_backward_parity_and_determinism(case):
    name, shape, io, chunk, softplus = case
    inp = _inputs(shape, io, False, softplus, seed=zlib.crc32(name.encode()) % 1000)
    _, _, ck = gpu_fwd(inp, chunk, softplus)
    g = gpu_bwd(inp, chunk, ckpt=ck, softplus=softplus)
    o = oracle_bwd(inp, chunk, softplus)
    t = tol(io, grad=True)
    for k in GRADS:
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], t)
    assert binding.ssm_scan_status(g["_ws"]) == 0
    g2 = gpu_bwd(inp, chunk, ckpt=ck, softplus=softplus)
    for k in GRADS:
        if g.get(k) is not None:
            assert torch.equal(g[k], g2[k]), k


def test_persistent_backward_ids_without_final_state_gradient():
    """The persistent path seeds the last chunk with zero when no final-state gradient is given
    and sums d_s0 over the sequences that share an initial-state row."""
    ns, L, H = 24, 80, 1024
    inp = _inputs((ns, L, H, 1, 16, 1), "bf16", False, False, seed=41)
    rows = 3
    inp["s0"] = 0.5 * torch.randn(rows, H, 1, 16)
    ids = torch.tensor([i % rows for i in range(ns)], dtype=torch.int32)
    _, _, ck = gpu_fwd(inp, 32, ids=ids, state_rows=rows)
    g = gpu_bwd(inp, 32, ckpt=ck, ids=ids, state_rows=rows, d_state_out=False)
    o = oracle_bwd(inp, 32, ids=ids, state_rows=rows, d_state_out=False)
    for k in GRADS:
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], tol("bf16", grad=True))
    assert binding.ssm_scan_status(g["_ws"]) == 0


def test_misaligned_inputs_fall_back_to_general_kernels():
    inp = _inputs((2, 150, 64, 1, 16, 1), "f32", False, False, seed=11)
    # x one element past a 16-byte boundary: the TMA paths cannot take it
    buf = torch.empty(inp["x"].numel() + 1)
    buf[1:] = inp["x"].reshape(-1)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    xbuf = buf.cuda()
    x_mis = xbuf[1:].view_as(inp["x"])
    assert x_mis.data_ptr() % 16 != 0
    y, st, ck = binding.ssm_scan_fwd(x_mis, d["dt"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     s0=d["s0"], chunk=32)
    yo, so, co = oracle_fwd(inp, 32)
    assert_close("y", y, yo, 1e-4)
    assert_close("ckpt", ck, co, 1e-4)
    g = binding.ssm_scan_bwd(x_mis, d["dt"], d["A"], d["B"], d["C"], d["dy"], D=d["D"], z=d["z"],
                             s0=d["s0"], ckpt=ck, d_state_out=d["d_state_out"], chunk=32)
    o = oracle_bwd(inp, 32)
    for k in ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_z"):
        assert_close(k, g[k], o[k], 1e-3)


def test_backward_without_checkpoints_recomputes():
    inp = _inputs((2, 200, 8, 1, 16, 1), "f32", False, False, seed=5)
    g1 = gpu_bwd(inp, 32, ckpt=None)
    _, _, ck = gpu_fwd(inp, 32)
    g2 = gpu_bwd(inp, 32, ckpt=ck)
    for k in ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0"):
        assert torch.equal(g1[k], g2[k]), k


def test_backward_is_bitwise_deterministic():
    inp = _inputs((2, 700, 40, 1, 16, 1), "f32", False, False, seed=6)
    _, _, ck = gpu_fwd(inp, 64)
    g1 = gpu_bwd(inp, 64, ckpt=ck)
    g2 = gpu_bwd(inp, 64, ckpt=ck)
    for k in ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0"):
        assert torch.equal(g1[k], g2[k]), k


def test_zero_upstream_gives_zero_gradients():
    inp = _inputs((2, 90, 8, 1, 16, 1), "f32", False, False, seed=7)
    inp["dy"] = torch.zeros_like(inp["dy"])
    g = gpu_bwd(inp, 32, d_state_out=False)
    for k in ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0"):
        assert not torch.any(g[k]), k


def test_bad_id_is_reported_not_read():
    inp = _inputs((2, 20, 4, 1, 16, 1), "f32", False, False, seed=8)
    inp["s0"] = torch.randn(2, 4, 1, 16)
    ids = torch.tensor([1, 7], dtype=torch.int32)  # 7 is outside [0, 2)
    shape = binding.scan_shape(inp["x"], inp["dt"], inp["A"], inp["B"], inp["s0"], 16)
    ws = torch.empty(binding.ssm_scan_workspace_size(shape, False), dtype=torch.uint8,
                     device="cuda")
    d = {k: v.cuda() for k, v in inp.items() if torch.is_tensor(v)}
    y, _, _ = binding.ssm_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                   s0=d["s0"], ids=ids.cuda(), chunk=16, state_rows=2, ws=ws)
    assert binding.ssm_scan_status(ws) == binding.SSM_ERR_INVALID_ARG
    # the bad row reads as a zero initial state
    inp0 = dict(inp)
    inp0["s0"] = None
    y0, _, _ = oracle_fwd(inp0, 16)
    assert_close("y[seq 1]", y[1], y0[1], 1e-4)


def test_ggml_packing_roundtrip():
    inp = _inputs((2, 5, 3, 2, 4, 1), "f32", True, False, seed=9)
    y, st, _ = gpu_fwd(inp, 256)
    packed = binding.pack_scan_result(y, st)
    assert packed.numel() == inp["x"].numel() + 2 * 3 * 2 * 4
    assert torch.equal(packed[: y.numel()].view_as(y), y)


# ---- full-size benchmark workloads ---------------------------------------------------------

def _workload_inputs(name):
    w = workload(name)
    inp = make_inputs(w, grad_seed_state=True)
    if inp["x"] is None:  # the conv prelude produces x; the scan parity needs only its shape
        g = torch.Generator().manual_seed(w.seed + 7)
        inp["x"] = torch.randn(w.n_seqs, w.n_tok, w.n_head, w.head_dim, generator=g).to(w.torch_io)
    return w, inp


@pytest.mark.parametrize("name", ["mamba1_layer_f32_b8_l1024_d512_n16"])
def test_workload_full_parity(name):
    w, inp = _workload_inputs(name)
    y, st, ck = gpu_fwd(inp, w.chunk)
    yo, so, co = oracle_fwd(inp, w.chunk)
    assert_close("y", y, yo, tol(w.io, False))
    assert_close("state_out", st, so, tol(w.io, False))
    assert_close("ckpt", ck, co, tol(w.io, False))
    g = gpu_bwd(inp, w.chunk, ckpt=ck)
    o = oracle_bwd(inp, w.chunk)
    for k in GRADS:
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], tol(w.io, True))


def test_mamba2_scan_forward_sampled_heads():
    w, inp = _workload_inputs("mamba2_scan_f32_b4_l2048_h24_p64_n128")
    y, st, ck = gpu_fwd(inp, w.chunk)
    heads = [0, 11, 23]
    sub = dict(inp)
    for k in ("x", "dt"):
        sub[k] = inp[k][:, :, heads]
    sub["A"] = inp["A"][heads]
    sub["s0"] = inp["s0"][:, heads]
    sub["D"] = sub["z"] = None
    yo, so, co = oracle_fwd(sub, w.chunk)
    assert_close("y", y[:, :, heads], yo, tol(w.io, False))
    assert_close("state_out", st[:, heads], so, tol(w.io, False))
    assert_close("ckpt", ck[:, :, heads], co, tol(w.io, False))


@pytest.mark.parametrize("name", ["mamba1_long_bf16_b1_l16384_d2048_n16",
                                  "mamba1_train_bf16_b16_l2048_d1536_n16"])
def test_workload_full_size_sampled_channels(name):
    w, inp = _workload_inputs(name)
    D = w.n_head
    idx = torch.tensor(sorted({0, 1, 31, 32, 127, D // 2, D - 2, D - 1}), dtype=torch.long)
    y, st, ck = gpu_fwd(inp, w.chunk)
    sub = channel_subset(inp, idx)
    yo, so, co = oracle_fwd(sub, w.chunk)
    assert_close("y", y[:, :, idx], yo, tol(w.io, False))
    assert_close("state_out", st[:, idx], so, tol(w.io, False))
    assert_close("ckpt", ck[:, :, idx], co, tol(w.io, False))
    # dense upstream gradient: every per-channel gradient of the sampled channels
    g = gpu_bwd(inp, w.chunk, ckpt=ck)
    o = oracle_bwd(sub, w.chunk)
    for k in ("d_x", "d_dt", "d_z"):
        assert_close(k, g[k][:, :, idx], o[k], tol(w.io, True))
    assert_close("d_A", g["d_A"][idx], o["d_A"], tol(w.io, True))
    assert_close("d_D", g["d_D"][idx], o["d_D"], tol(w.io, True))
    assert_close("d_s0", g["d_s0"][:, idx], o["d_s0"], tol(w.io, True))
    # upstream gradient only on the sampled channels: dB and dC reduce to the subset's sums
    sparse = dict(inp)
    mask = torch.zeros(D, dtype=torch.bool)
    mask[idx] = True
    sparse["dy"] = torch.where(mask[None, None, :, None], inp["dy"], torch.zeros_like(inp["dy"]))
    sparse["d_state_out"] = torch.where(mask[None, :, None, None], inp["d_state_out"],
                                        torch.zeros_like(inp["d_state_out"]))
    gs = gpu_bwd(sparse, w.chunk, ckpt=ck)
    os_ = oracle_bwd(channel_subset(sparse, idx), w.chunk)
    assert_close("d_B", gs["d_B"], os_["d_B"], tol(w.io, True))
    assert_close("d_C", gs["d_C"], os_["d_C"], tol(w.io, True))


@pytest.mark.parametrize("shape,io,scalar_a", [
    ((1, 40, 4, 1, 512, 1), "f32", False),     # the forward's largest d_state, per-state A
    ((2, 33, 2, 4, 512, 2), "bf16", True),     # ... one A per head, groups, bf16
])
def test_scan_forward_largest_d_state(shape, io, scalar_a):
    """d_state at SSM_MAX_D_STATE (512): the general forward, ragged tokens, against the oracle."""
    inp = _inputs(shape, io, scalar_a, False, seed=17)
    y, st, ck = gpu_fwd(inp, 16)
    yo, so, co = oracle_fwd(inp, 16)
    t = tol(io, grad=False)
    assert_close("y", y, yo, t)
    assert_close("state_out", st, so, t)
    assert_close("ckpt", ck, co, t)


def test_scan_backward_largest_d_state():
    """d_state at SSM_MAX_D_STATE_BWD (128) with per-state A (the general backward kernels)."""
    inp = _inputs((2, 45, 3, 2, 128, 1), "f32", False, False, seed=19)
    _, _, ck = gpu_fwd(inp, 16)
    g = gpu_bwd(inp, 16, ckpt=ck)
    o = oracle_bwd(inp, 16)
    for k in GRADS:
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], tol("f32", grad=True))

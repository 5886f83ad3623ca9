"""Pins of the oracle's scan forward to things other than itself.

- a worked example computed by hand (tests/golden/scan_hand_l3_n1.json);
- constant inputs: the geometric series h_t = a^{t+1} h0 + u (1 - a^{t+1}) / (1 - a);
- delta = 0 keeps the state; zero x and zero s0 give zero outputs (ggmlR "the ssm_scan views
  read back the halves they point at");
- scipy.signal.lfilter (a library IIR filter) for a constant decay and varying input;
- the explicit sum h_t = sum_s exp(A (S_t - S_s)) u_s + exp(A S_t) h0 with cumulative sums of
  delta (pins which delta each decay uses);
- balanced-tree (associative) composition equals the sequential loop;
- checkpoints at any interval equal the full-history states;
- scalar-A form equals the per-state form with A broadcast; groups map head h to h / (H/G);
- ids pick the start row; softplus mode equals feeding torch's softplus(dt + bias).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.signal
import torch

import oracle
from oracle import ScanDims
from bwd_ssm_conv_gb300.workloads import random_scan_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(v):
    return float(eval(v, {"ln2": math.log(2.0)})) if isinstance(v, str) else float(v)


def _load_hand():
    with open(os.path.join(GOLDEN, "scan_hand_l3_n1.json")) as f:
        g = json.load(f)
    i = {k: np.array([_ev(v) for v in vals]) for k, vals in g["inputs"].items()}
    e = {k: np.array([_ev(v) for v in vals]) for k, vals in g["expected"].items()}
    return i, e


def _all_states(dims, inp, **kw):
    """States h_t for every t, from checkpoints every token plus the final state."""
    d1 = ScanDims(**{**dims.__dict__, "chunk": 1})
    y, st, ck = oracle.scan_fwd(d1, **kw)
    # ck[b][t] = state at the start of token t = h_{t-1}; shift by one and append state_out
    return np.concatenate([ck[:, 1:], st[:, None]], axis=1), y


def test_hand_worked_example_forward():
    i, e = _load_hand()
    dims = ScanDims(1, 3, 1, 1, 1, chunk=2)
    y, st, ck = oracle.scan_fwd(dims, x=i["x"].reshape(1, 3, 1, 1), dt=i["dt"].reshape(1, 3, 1),
                                A=i["A"].reshape(1, 1), B=i["B"].reshape(1, 3, 1, 1),
                                C=i["C"].reshape(1, 3, 1, 1), D=i["D"], s0=i["s0"].reshape(1, 1, 1, 1))
    np.testing.assert_allclose(y.ravel(), e["y"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(st.ravel(), e["state_out"], rtol=1e-14)
    # checkpoints: state at the start of chunk 0 (= s0) and of chunk 1 (= h after token 1)
    np.testing.assert_allclose(ck.ravel(), [1.0, -0.75], rtol=1e-14)


@pytest.mark.parametrize("gate", [False, True])
def test_constant_inputs_geometric_series(gate):
    L, H, N = 40, 3, 5
    rng = np.random.default_rng(1)
    delta = 0.07
    A = -rng.uniform(0.5, 3.0, (H, N))
    xv = rng.normal(size=H)
    Bv, Cv = rng.normal(size=N), rng.normal(size=N)
    D = rng.normal(size=H)
    h0 = rng.normal(size=(1, H, 1, N))
    zv = rng.normal(size=H)
    x = np.broadcast_to(xv[None, None, :, None], (1, L, H, 1))
    dt = np.full((1, L, H), delta)
    B = np.broadcast_to(Bv, (1, L, 1, N))
    C = np.broadcast_to(Cv, (1, L, 1, N))
    z = np.broadcast_to(zv[None, None, :, None], (1, L, H, 1)) if gate else None
    y, st, _ = oracle.scan_fwd(ScanDims(1, L, H, 1, N), x=x, dt=dt, A=A, B=B, C=C, D=D, z=z, s0=h0)
    t = np.arange(L)[:, None, None]                     # [L, 1, 1]
    a = np.exp(delta * A)[None]                         # [1, H, N]
    u = (delta * xv[:, None] * Bv[None, :])[None]       # [1, H, N]
    h = a ** (t + 1) * h0[0, :, 0][None] + u * (1 - a ** (t + 1)) / (1 - a)
    y_ref = (h * Cv).sum(-1) + D * xv                   # [L, H]
    if gate:
        y_ref = y_ref * zv / (1 + np.exp(-zv))
    np.testing.assert_allclose(y[0, :, :, 0], y_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(st[0, :, 0], h[-1], rtol=1e-11, atol=1e-12)


def test_zero_delta_keeps_state():
    d = random_scan_inputs(2, 7, 3, 2, 4, seed=2)
    dt = np.zeros((2, 7, 3))
    y, st, _ = oracle.scan_fwd(ScanDims(2, 7, 3, 2, 4), x=d["x"], dt=dt, A=d["A"], B=d["B"],
                               C=d["C"], D=d["D"], s0=d["s0"])
    s0 = d["s0"].double().numpy()
    np.testing.assert_array_equal(st, s0)
    ypre = np.einsum("bthpn,bthpn->bthp", np.broadcast_to(s0[:, None], (2, 7, 3, 2, 4)),
                     np.broadcast_to(d["C"].double().numpy()[:, :, :, None, :], (2, 7, 3, 2, 4)))
    ypre = ypre + d["D"].double().numpy().reshape(3, 2) * d["x"].double().numpy()
    np.testing.assert_allclose(y, ypre, rtol=1e-13, atol=1e-13)


def test_zero_x_and_state_give_zero():
    d = random_scan_inputs(2, 9, 2, 3, 4, seed=3)
    y, st, ck = oracle.scan_fwd(ScanDims(2, 9, 2, 3, 4, chunk=4), x=np.zeros((2, 9, 2, 3)),
                                dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], D=d["D"], z=d["z"])
    assert not y.any() and not st.any() and not ck.any()


def test_lfilter_constant_decay_varying_input():
    L, N = 50, 3
    rng = np.random.default_rng(4)
    delta, A = 0.2, np.array([[-0.3, -1.0, -2.5]])
    x = rng.normal(size=(1, L, 1, 1))
    B = rng.normal(size=(1, L, 1, N))
    h0 = rng.normal(size=(1, 1, 1, N))
    dims = ScanDims(1, L, 1, 1, N)
    states, _ = _all_states(dims, None, x=x, dt=np.full((1, L, 1), delta), A=A, B=B,
                            C=np.zeros((1, L, 1, N)), s0=h0)
    for n in range(N):
        a = math.exp(delta * A[0, n])
        u = delta * x[0, :, 0, 0] * B[0, :, 0, n]
        ref, _ = scipy.signal.lfilter([1.0], [1.0, -a], u, zi=[a * h0[0, 0, 0, n]])
        np.testing.assert_allclose(states[0, :, 0, 0, n], ref, rtol=1e-12, atol=1e-13)


def test_explicit_sum_time_varying_decay():
    d = random_scan_inputs(1, 20, 2, 1, 3, seed=5)
    dims = ScanDims(1, 20, 2, 1, 3)
    states, _ = _all_states(dims, None, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"],
                            s0=d["s0"])
    x, dt, A, B = (d[k].double().numpy() for k in ("x", "dt", "A", "B"))
    s0 = d["s0"].double().numpy()
    S = np.cumsum(dt[0], axis=0)  # [L, H]: S_t = sum_{r<=t} delta_r
    for h in range(2):
        for n in range(3):
            for t in range(20):
                acc = math.exp(A[h, n] * S[t, h]) * s0[0, h, 0, n]
                for s in range(t + 1):
                    acc += (math.exp(A[h, n] * (S[t, h] - S[s, h])) * dt[0, s, h] * x[0, s, h, 0]
                            * B[0, s, 0, n])
                assert abs(states[0, t, h, 0, n] - acc) < 1e-12 * max(1.0, abs(acc))


@pytest.mark.parametrize("L", [1, 2, 7, 33, 64])
def test_tree_composition_equals_sequential(L):
    d = random_scan_inputs(2, L, 3, 2, 4, n_group=1, seed=L)
    dims = ScanDims(2, L, 3, 2, 4)
    seq, _ = _all_states(dims, None, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"],
                         s0=d["s0"])
    tree = oracle.scan_states_assoc(dims, d["x"], d["dt"], d["A"], d["B"], s0=d["s0"])
    np.testing.assert_allclose(tree, seq, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 100])
def test_checkpoints_equal_full_history(chunk):
    d = random_scan_inputs(2, 64, 2, 1, 4, seed=6)
    dims = ScanDims(2, 64, 2, 1, 4, chunk=chunk)
    full, y_full = _all_states(dims, None, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"],
                               D=d["D"], z=d["z"], s0=d["s0"])
    y, st, ck = oracle.scan_fwd(dims, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"],
                                D=d["D"], z=d["z"], s0=d["s0"])
    np.testing.assert_array_equal(y, y_full)
    s0 = d["s0"].double().numpy()
    for c in range(dims.n_chunks):
        ref = s0 if c == 0 else full[:, c * chunk - 1]
        np.testing.assert_array_equal(ck[:, c], ref)


def test_scalar_a_equals_broadcast_per_state_a():
    d = random_scan_inputs(2, 12, 3, 4, 5, scalar_a=True, seed=7)
    A = d["A"].double().numpy()
    kw = dict(x=d["x"], dt=d["dt"], B=d["B"], C=d["C"], D=d["D"], z=d["z"], s0=d["s0"])
    y1, s1, _ = oracle.scan_fwd(ScanDims(2, 12, 3, 4, 5, a_per_state=0), A=A, **kw)
    y2, s2, _ = oracle.scan_fwd(ScanDims(2, 12, 3, 4, 5, a_per_state=1),
                                A=np.repeat(A[:, None], 5, axis=1), **kw)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(s1, s2)


def test_groups_map_heads_to_h_over_heads_per_group():
    H, G = 4, 2
    d = random_scan_inputs(1, 10, H, 2, 3, n_group=G, seed=8)
    y, st, _ = oracle.scan_fwd(ScanDims(1, 10, H, 2, 3, n_group=G), x=d["x"], dt=d["dt"],
                               A=d["A"], B=d["B"], C=d["C"], D=d["D"], z=d["z"], s0=d["s0"])
    hpg = H // G
    for g in range(G):
        hs = slice(g * hpg, (g + 1) * hpg)
        yg, sg, _ = oracle.scan_fwd(
            ScanDims(1, 10, hpg, 2, 3, n_group=1), x=d["x"][:, :, hs], dt=d["dt"][:, :, hs],
            A=d["A"][hs], B=d["B"][:, :, g:g + 1], C=d["C"][:, :, g:g + 1],
            D=d["D"].view(H, 2)[hs].reshape(-1), z=d["z"][:, :, hs], s0=d["s0"][:, hs])
        np.testing.assert_array_equal(y[:, :, hs], yg)
        np.testing.assert_array_equal(st[:, hs], sg)


def test_ids_select_start_rows():
    d = random_scan_inputs(3, 8, 2, 1, 4, seed=9)
    rows = torch.randn(5, 2, 1, 4, generator=torch.Generator().manual_seed(1)).double()
    ids = np.array([4, 0, 2], dtype=np.int32)
    kw = dict(x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], D=d["D"], z=d["z"])
    y1, s1, _ = oracle.scan_fwd(ScanDims(3, 8, 2, 1, 4, state_rows=5), s0=rows, ids=ids, **kw)
    y2, s2, _ = oracle.scan_fwd(ScanDims(3, 8, 2, 1, 4), s0=rows[ids], **kw)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(s1, s2)


def test_softplus_mode_equals_torch_softplus_inputs():
    d = random_scan_inputs(2, 9, 3, 1, 4, seed=10, dt_raw=True)
    bias = np.array([0.3, -0.7, 21.5])  # the last head crosses the threshold of 20
    dt_raw = d["dt"].double()
    delta = torch.nn.functional.softplus(dt_raw + torch.tensor(bias)).numpy()
    kw = dict(x=d["x"], A=d["A"], B=d["B"], C=d["C"], D=d["D"], z=d["z"], s0=d["s0"])
    y1, s1, _ = oracle.scan_fwd(ScanDims(2, 9, 3, 1, 4, dt_softplus=1), dt=dt_raw, dt_bias=bias,
                                **kw)
    y2, s2, _ = oracle.scan_fwd(ScanDims(2, 9, 3, 1, 4), dt=delta, **kw)
    np.testing.assert_allclose(y1, y2, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(s1, s2, rtol=1e-14, atol=1e-14)


def test_ggml_packing_sizes():
    # ggmlR "ggml_ssm_scan packs outputs and states into one flat tensor": nelements(x) +
    # d_state*head_dim*n_head*n_seqs
    dims = ScanDims(2, 2, 3, 2, 4)
    d = random_scan_inputs(2, 2, 3, 2, 4, seed=0)
    y, st, _ = oracle.scan_fwd(dims, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"])
    assert y.size + st.size == d["x"].numel() + 4 * 2 * 3 * 2

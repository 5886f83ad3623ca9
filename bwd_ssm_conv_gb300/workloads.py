"""Seeded synthetic workloads for the selective scan and its conv1d prelude.

This module only draws random inputs with the shapes and value distributions of the
five benchmark configurations (and of arbitrary small test shapes).  It performs none of
the scan's or the conv's arithmetic, and both the CUDA path's tests and the oracle's tests
draw from it, so the two always see the same bytes.

Recipe (per configuration, ``seed = 1000 + index`` unless given):
  * conv input ``sx`` [n_s][d][K-1+L]: a zero (K-1)-column prefix (zero initial conv state)
    followed by N(0,1) samples; conv weight ``c`` [d][K] ~ U(-0.5, 0.5); no conv bias.
  * ``z``, ``B``, ``C``, ``dy`` ~ N(0,1).
  * ``dt``: per channel (per head in the scalar-A form) u = exp(U(ln 1e-3, ln 1e-1)),
    dt = softplus(0.5 N(0,1) + log(expm1(u))) -- positive, centred near u.
  * ``A = -exp(A_log)`` with ``A_log[d][n] = log(n+1)``, i.e. A[d][n] = -(n+1).
    Scalar-A (Mamba-2) form: A[h] = -exp(U(log 1, log 16)).
  * ``D = 1``; ``h0 = 0`` except in the scalar-A configuration where s0 ~ N(0, 0.1^2).
  * bf16 configurations round every activation once (round-to-nearest-even) on the host;
    parameters and states stay fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_seqs: int
    n_tok: int
    n_head: int          # d_inner for the Mamba-1 form
    head_dim: int = 1
    d_state: int = 16
    n_group: int = 1
    d_conv: int = 4      # 0: no conv prelude (x drawn directly)
    io: str = "f32"      # "f32" | "bf16"
    has_z: bool = True
    has_D: bool = True
    scalar_a: bool = False
    chunk: int = 256
    nonzero_s0: bool = False
    fwd_only: bool = False
    seed: int = 1000

    @property
    def channels(self) -> int:
        return self.n_head * self.head_dim

    @property
    def tokens(self) -> int:
        return self.n_seqs * self.n_tok

    @property
    def io_bytes(self) -> int:
        return 2 if self.io == "bf16" else 4

    @property
    def torch_io(self):
        return torch.bfloat16 if self.io == "bf16" else torch.float32

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the benchmark, in order (`bench.py --config I` picks one by position).
WORKLOADS = [
    Workload("mamba1_tiny_f32_b1_l64_d16_n4", 1, 64, 16, d_state=4, io="f32", seed=1000),
    Workload("mamba1_layer_f32_b8_l1024_d512_n16", 8, 1024, 512, d_state=16, io="f32", seed=1001),
    Workload("mamba2_scan_f32_b4_l2048_h24_p64_n128", 4, 2048, 24, head_dim=64, d_state=128,
             d_conv=0, io="f32", has_z=False, has_D=False, scalar_a=True, nonzero_s0=True,
             fwd_only=True, seed=1002),
    Workload("mamba1_long_bf16_b1_l16384_d2048_n16", 1, 16384, 2048, d_state=16, io="bf16",
             chunk=256, seed=1003),
    Workload("mamba1_train_bf16_b16_l2048_d1536_n16", 16, 2048, 1536, d_state=16, io="bf16",
             chunk=256, seed=1004),
]


BY_NAME = {w.name: w for w in WORKLOADS}


def workload(name: str) -> Workload:
    """The benchmark workload of that name (KeyError for an unknown name)."""
    return BY_NAME[name]


def _round_io(t: torch.Tensor, io: str) -> torch.Tensor:
    """Round once to the I/O dtype (RNE for bf16); returns a tensor OF that dtype."""
    return t.to(torch.bfloat16) if io == "bf16" else t.to(torch.float32)


def make_inputs(w: Workload, seed: int | None = None, grad_seed_state: bool = False) -> dict:
    """Draw every input of one fwd+bwd step on the CPU.

    Returns a dict of CPU tensors: activations in the I/O dtype, parameters fp32.
    Keys: sx (or None), c, x (None when the conv prelude produces it), dt, A, B, C, D, z, s0,
    dy, d_state_out.  ``d_state_out`` is None unless ``grad_seed_state``.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    ns, L, H, P, N, G, K = w.n_seqs, w.n_tok, w.n_head, w.head_dim, w.d_state, w.n_group, w.d_conv
    ch = H * P
    out: dict = {}

    if K > 0:
        body = torch.randn(ns, ch, L, generator=g)
        sx = torch.cat([torch.zeros(ns, ch, K - 1), body], dim=2)
        out["sx"] = _round_io(sx, w.io)
        out["c"] = (torch.rand(ch, K, generator=g) - 0.5).float()
        out["x"] = None
    else:
        out["sx"] = None
        out["c"] = None
        out["x"] = _round_io(torch.randn(ns, L, H, P, generator=g), w.io)

    # dt: per-channel (per-head) centre u, log-uniform in [1e-3, 1e-1]
    lo, hi = math.log(1e-3), math.log(1e-1)
    u = torch.exp(lo + (hi - lo) * torch.rand(H, generator=g))
    inv_sp = torch.log(torch.expm1(u))
    dt = torch.nn.functional.softplus(0.5 * torch.randn(ns, L, H, generator=g) + inv_sp)
    out["dt"] = _round_io(dt, w.io)

    if w.scalar_a:
        out["A"] = (-torch.exp(math.log(16.0) * torch.rand(H, generator=g))).float()
    else:
        a_log = torch.log(torch.arange(1, N + 1, dtype=torch.float32)).expand(H, N)
        out["A"] = (-torch.exp(a_log)).contiguous().float()

    out["B"] = _round_io(torch.randn(ns, L, G, N, generator=g), w.io)
    out["C"] = _round_io(torch.randn(ns, L, G, N, generator=g), w.io)
    out["D"] = torch.ones(ch, dtype=torch.float32) if w.has_D else None
    out["z"] = _round_io(torch.randn(ns, L, H, P, generator=g), w.io) if w.has_z else None
    if w.nonzero_s0:
        out["s0"] = (0.1 * torch.randn(ns, H, P, N, generator=g)).float()
    else:
        out["s0"] = None
    out["dy"] = _round_io(torch.randn(ns, L, H, P, generator=g), w.io)
    if grad_seed_state:
        out["d_state_out"] = torch.randn(ns, H, P, N, generator=g).float()
    else:
        out["d_state_out"] = None
    return out


def random_scan_inputs(n_seqs, n_tok, n_head, head_dim, d_state, n_group=1, io="f32",
                       scalar_a=False, has_z=True, has_D=True, s0=True, seed=0,
                       dt_raw=False) -> dict:
    """Small arbitrary-shape scan inputs for tests (same distributions as the workloads).

    ``dt_raw``: draw dt ~ U(-1, 1) (a raw pre-softplus value, as in ggmlR's scan gradcheck)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    ns, L, H, P, N, G = n_seqs, n_tok, n_head, head_dim, d_state, n_group
    d = {}
    d["x"] = _round_io(torch.randn(ns, L, H, P, generator=g), io)
    if dt_raw:
        d["dt"] = _round_io(2 * torch.rand(ns, L, H, generator=g) - 1, io)
    else:
        lo, hi = math.log(1e-3), math.log(1e-1)
        u = torch.exp(lo + (hi - lo) * torch.rand(H, generator=g))
        d["dt"] = _round_io(torch.nn.functional.softplus(
            0.5 * torch.randn(ns, L, H, generator=g) + torch.log(torch.expm1(u))), io)
    if scalar_a:
        d["A"] = (-torch.exp(math.log(16.0) * torch.rand(H, generator=g))).float()
    else:
        d["A"] = (-(0.5 + 2 * torch.rand(H, N, generator=g)) *
                  torch.arange(1, N + 1, dtype=torch.float32)).float()
    d["B"] = _round_io(torch.randn(ns, L, G, N, generator=g), io)
    d["C"] = _round_io(torch.randn(ns, L, G, N, generator=g), io)
    d["D"] = torch.randn(H * P, generator=g).float() if has_D else None
    d["z"] = _round_io(torch.randn(ns, L, H, P, generator=g), io) if has_z else None
    d["s0"] = (0.5 * torch.randn(ns, H, P, N, generator=g)).float() if s0 else None
    d["dy"] = _round_io(torch.randn(ns, L, H, P, generator=g), io)
    d["d_state_out"] = torch.randn(ns, H, P, N, generator=g).float()
    return d


def random_conv_inputs(n_s, d_inner, n_t, d_conv, io="f32", bias=False, seed=0) -> dict:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    d = {}
    d["sx"] = _round_io(torch.randn(n_s, d_inner, n_t + d_conv - 1, generator=g), io)
    d["c"] = (torch.rand(d_inner, d_conv, generator=g) - 0.5).float()
    d["bias"] = (0.5 * torch.randn(d_inner, generator=g)).float() if bias else None
    d["dout"] = _round_io(torch.randn(n_s, n_t, d_inner, generator=g), io)
    return d

"""Seeded synthetic inputs for the fused conv1d + KDA verify-decode path.

This module only draws random numbers with the shapes, dtypes and
distributions of the workloads; it performs none of the method's arithmetic
(no convolution, no gate, no recurrence).  It is the one module that both the
CPU oracle tests and the CUDA path consume, so that the two are fed exactly
the same bits.

Tensor layout (all dense, row-major, contiguous):

    mixed_qkv   act  [N, T, dim]         dim = 2*H*K + HV*V, channels q | k | v
    conv_w      act  [dim, W]            tap W-1 multiplies the newest token
    conv_state  act  [N, dim, W-1]       index 0 is the oldest raw input
    A_log       f32  [HV]                softplus gate only
    dt_bias     f32  [HV, K]             softplus gate only
    a           act  [N, T, HV, K]       gate input (safe gate: the log-decay)
    b           act  [N, T, HV]          beta logit
    S0          f32  [N, HV, K, V]       persistent recurrent state (read-only)

"act" is float32 for the tiny workload and bfloat16 elsewhere.  Normal
distributions are written N(mean, std): the second number is the standard
deviation.  Draws happen in the fixed order of ``_DRAW_ORDER`` from one
``torch.Generator`` on the CPU, so a (workload, seed) pair always yields the
same tensors on any machine.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Iterator, Optional

import torch

GATE_SOFTPLUS = "softplus"
GATE_SAFE = "safe"


@dataclasses.dataclass(frozen=True)
class Shape:
    N: int
    T: int
    H: int
    HV: int
    K: int = 128
    V: int = 128
    W: int = 4
    act: str = "bf16"  # "bf16" or "f32"

    @property
    def dim(self) -> int:
        return 2 * self.H * self.K + self.HV * self.V

    @property
    def G(self) -> int:
        return self.HV // self.H

    @property
    def head_steps(self) -> int:
        return self.N * self.T * self.HV

    @property
    def act_bytes(self) -> int:
        return 4 if self.act == "f32" else 2

    @property
    def torch_act(self) -> torch.dtype:
        return torch.float32 if self.act == "f32" else torch.bfloat16

    def algorithmic_bytes(self, gate: str = "softplus") -> int:
        """Bytes the method itself must move once per call.

        S0 read once, every per-token state snapshot written once, the packed
        inputs read once, conv_state read and written once, the conv-window
        snapshots and the output written once, the small parameters read once
        (A_log and dt_bias only under the softplus gate, which reads them).
        """
        N, T, HV, K, V, W = self.N, self.T, self.HV, self.K, self.V, self.W
        dim, ab = self.dim, self.act_bytes
        state = 4 * N * HV * K * V * (1 + T)
        acts = ab * (N * T * dim + 2 * N * dim * (W - 1) + N * T * dim * (W - 1)
                     + N * T * HV * K + N * T * HV + N * T * HV * V + W * dim)
        params = 4 * HV * (1 + K) if gate == "softplus" else 0
        return state + acts + params

    def label(self) -> str:
        return (f"N{self.N}_T{self.T}_H{self.H}_HV{self.HV}_K{self.K}_V{self.V}"
                f"_{self.act}")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    gate: str
    seed: int
    s0_std: float
    # gate input distribution: ("normal", std) or ("uniform", lo, hi)
    a_dist: tuple = ("normal", 1.0)
    # plant these values into `a` at every `plant_stride`-th element so that
    # the large-argument softplus branch is certainly taken
    plant: tuple = ()
    plant_stride: int = 4096


# The five configurations of the verify-decode workload.
TINY = Workload("tiny_fp32_n2_t2_h2", Shape(2, 2, 2, 2, 32, 32, 4, "f32"),
                GATE_SOFTPLUS, seed=0, s0_std=0.1)
DECODE = Workload("decode_bf16_n16_t4_h16", Shape(16, 4, 16, 16),
                  GATE_SOFTPLUS, seed=1, s0_std=0.05)
GVA = Workload("gva_bf16_n64_t4_h8_hv32_safe", Shape(64, 4, 8, 32),
               GATE_SAFE, seed=2, s0_std=0.05, a_dist=("uniform", -5.0, 0.0))
LARGE = Workload("large_bf16_n256_t4_h32", Shape(256, 4, 32, 32),
                 GATE_SOFTPLUS, seed=3, s0_std=0.05, a_dist=("normal", 4.0),
                 plant=(25.0, 100.0))

WORKLOADS: Dict[str, Workload] = {w.name: w for w in (TINY, DECODE, GVA, LARGE)}

SWEEP_T = (1, 2, 3, 4, 8)
SWEEP_N = (1, 8, 32, 128, 512)
SWEEP_HEADS = ((16, 16), (16, 32), (32, 64))
SWEEP_GATES = (GATE_SOFTPLUS, GATE_SAFE)


def sweep() -> Iterator[Workload]:
    """The 150-point T x N x (H, HV) x gate sweep, seeds 100 + point index."""
    idx = 0
    for T in SWEEP_T:
        for N in SWEEP_N:
            for H, HV in SWEEP_HEADS:
                for gate in SWEEP_GATES:
                    a_dist = ("uniform", -5.0, 0.0) if gate == GATE_SAFE else ("normal", 1.0)
                    yield Workload(f"sweep_T{T}_N{N}_H{H}_HV{HV}_{gate}",
                                   Shape(N, T, H, HV), gate, seed=100 + idx,
                                   s0_std=0.05, a_dist=a_dist)
                    idx += 1


def custom(N: int, T: int, H: int, HV: int, K: int = 128, V: int = 128,
           act: str = "bf16", gate: str = GATE_SOFTPLUS, seed: int = 0,
           s0_std: float = 0.05) -> Workload:
    """An ad-hoc workload with the decode distributions (tests, edge cases)."""
    a_dist = ("uniform", -5.0, 0.0) if gate == GATE_SAFE else ("normal", 1.0)
    return Workload(f"custom_{Shape(N, T, H, HV, K, V, 4, act).label()}_{gate}",
                    Shape(N, T, H, HV, K, V, 4, act), gate, seed=seed,
                    s0_std=s0_std, a_dist=a_dist)


_DRAW_ORDER = ("mixed_qkv", "conv_state", "conv_w", "a", "b", "S0", "A_log", "dt_bias")


def make_inputs(wl: Workload, device: str = "cpu") -> Dict[str, Optional[torch.Tensor]]:
    """Draw the inputs of one call.  Values never depend on `device`: the
    draws always happen on the CPU and are copied afterwards."""
    s = wl.shape
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed)
    act = s.torch_act
    dim = s.dim

    def normal(shape, std=1.0):
        return torch.randn(shape, generator=g, dtype=torch.float32).mul_(std)

    def uniform(shape, lo, hi):
        return torch.rand(shape, generator=g, dtype=torch.float32).mul_(hi - lo).add_(lo)

    out: Dict[str, Optional[torch.Tensor]] = {}
    for name in _DRAW_ORDER:
        if name == "mixed_qkv":
            out[name] = normal((s.N, s.T, dim)).to(act)
        elif name == "conv_state":
            out[name] = normal((s.N, dim, s.W - 1)).to(act)
        elif name == "conv_w":
            out[name] = uniform((dim, s.W), -0.5, 0.5).to(act)
        elif name == "a":
            shape = (s.N, s.T, s.HV, s.K)
            if wl.a_dist[0] == "normal":
                a = normal(shape, wl.a_dist[1])
            else:
                a = uniform(shape, wl.a_dist[1], wl.a_dist[2])
            if wl.plant:
                flat = a.view(-1)
                for j, val in enumerate(wl.plant):
                    flat[j * (wl.plant_stride // max(1, len(wl.plant)))::wl.plant_stride] = val
            out[name] = a.to(act)
        elif name == "b":
            out[name] = normal((s.N, s.T, s.HV)).to(act)
        elif name == "S0":
            out[name] = normal((s.N, s.HV, s.K, s.V), wl.s0_std)
        elif name == "A_log":
            v = uniform((s.HV,), 0.0, math.log(16.0))
            out[name] = v if wl.gate == GATE_SOFTPLUS else None
        elif name == "dt_bias":
            v = uniform((s.HV, s.K), -1.0, 1.0)
            out[name] = v if wl.gate == GATE_SOFTPLUS else None
    if device != "cpu":
        out = {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    return out


def make_inputs_on_device(wl: Workload, device) -> Dict[str, Optional[torch.Tensor]]:
    """Inputs with the same shapes, dtypes and distributions drawn directly on
    `device` by its own seeded generator: fast for large timing-only runs, but
    the values differ from `make_inputs` (never use them for parity)."""
    s = wl.shape
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed)
    act = s.torch_act
    f32 = dict(generator=g, dtype=torch.float32, device=device)

    def uni(shape, lo, hi):
        return torch.rand(shape, **f32).mul_(hi - lo).add_(lo)

    out: Dict[str, Optional[torch.Tensor]] = {
        "mixed_qkv": torch.randn((s.N, s.T, s.dim), **f32).to(act),
        "conv_state": torch.randn((s.N, s.dim, s.W - 1), **f32).to(act),
        "conv_w": uni((s.dim, s.W), -0.5, 0.5).to(act),
    }
    shape = (s.N, s.T, s.HV, s.K)
    a = (torch.randn(shape, **f32).mul_(wl.a_dist[1]) if wl.a_dist[0] == "normal"
         else uni(shape, wl.a_dist[1], wl.a_dist[2]))
    if wl.plant:
        flat = a.view(-1)
        for j, val in enumerate(wl.plant):
            flat[j * (wl.plant_stride // max(1, len(wl.plant)))::wl.plant_stride] = val
    out["a"] = a.to(act)
    out["b"] = torch.randn((s.N, s.T, s.HV), **f32).to(act)
    out["S0"] = torch.randn((s.N, s.HV, s.K, s.V), **f32).mul_(wl.s0_std)
    sp = wl.gate == GATE_SOFTPLUS
    out["A_log"] = uni((s.HV,), 0.0, math.log(16.0)) if sp else None
    out["dt_bias"] = uni((s.HV, s.K), -1.0, 1.0) if sp else None
    return out


def empty_outputs(wl: Workload, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Uninitialised output buffers of the right shapes and dtypes."""
    s = wl.shape
    return {
        "o": torch.empty((s.N, s.T, s.HV, s.V), dtype=s.torch_act, device=device),
        "inter_ssm": torch.empty((s.N, s.T, s.HV, s.K, s.V), dtype=torch.float32, device=device),
        "conv_snapshots": torch.empty((s.N, s.T, s.dim, s.W - 1), dtype=s.torch_act, device=device),
    }

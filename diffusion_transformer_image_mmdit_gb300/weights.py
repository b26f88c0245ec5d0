"""Device copies of block weights: from host arrays (tests) or drawn on the
GPU (benchmark).  Marshalling only: weights stay as drawn, bf16 linears with
fp32 biases and fp32 RMSNorm gains."""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from .api import CondWeights, DoubleWeights, LinearDev, SingleWeights, StepWeights


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=torch.bfloat16)


def _f32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def linear_from_host(w: np.ndarray, b: Optional[np.ndarray], device="cuda") -> LinearDev:
    return LinearDev(_bf16(w, device), None if b is None else _f32(b, device))


def double_from_host(p: dict, device="cuda") -> DoubleWeights:
    L = lambda s, n: linear_from_host(p[s][n + "_w"], p[s][n + "_b"], device)
    return DoubleWeights(mod=[L("txt", "mod"), L("img", "mod")], qkv=[L("txt", "qkv"), L("img", "qkv")],
                         proj=[L("txt", "proj"), L("img", "proj")], mlp_in=[L("txt", "mlp_in"), L("img", "mlp_in")],
                         mlp_out=[L("txt", "mlp_out"), L("img", "mlp_out")],
                         q_norm=[_f32(p["txt"]["q_norm"], device), _f32(p["img"]["q_norm"], device)],
                         k_norm=[_f32(p["txt"]["k_norm"], device), _f32(p["img"]["k_norm"], device)])


def single_from_host(p: dict, device="cuda") -> SingleWeights:
    L = lambda n: linear_from_host(p[n + "_w"], p[n + "_b"], device)
    return SingleWeights(L("mod"), L("lin1"), L("lin2"), _f32(p["q_norm"], device), _f32(p["k_norm"], device))


def step_from_host(p: dict, device="cuda") -> StepWeights:
    return StepWeights(linear_from_host(p["t_w1"], p["t_b1"], device),
                       linear_from_host(p["t_w2"], p["t_b2"], device),
                       linear_from_host(p["img_in_w"], p["img_in_b"], device),
                       linear_from_host(p["final_mod_w"], p["final_mod_b"], device),
                       linear_from_host(p["final_w"], p["final_b"], device),
                       [double_from_host(d, device) for d in p["double"]],
                       [single_from_host(s, device) for s in p["single"]])


def cond_from_host(p: dict, device="cuda") -> CondWeights:
    L = lambda w, b: linear_from_host(p[w], p[b], device)
    return CondWeights(L("txt_in_w", "txt_in_b"), L("g_w1", "g_b1"), L("g_w2", "g_b2"), L("y_w1", "y_b1"),
                       L("y_w2", "y_b2"))


# ------------------------------------------------------------------ drawn on the GPU
class DeviceDraw:
    """Seeded N(mean, std) draws on the GPU (torch.Generator), for workloads too
    large to draw on the host.  Linear weights and biases N(0, 0.02) in bf16 /
    fp32, RMSNorm gains 1 + N(0, 0.02)."""

    def __init__(self, seed: int = 0, device="cuda"):
        self.g = torch.Generator(device=device)
        self.g.manual_seed(seed)
        self.device = device

    def normal(self, shape, std=1.0, mean=0.0, dtype=torch.float32) -> torch.Tensor:
        t = torch.empty(shape, dtype=torch.float32, device=self.device)
        t.normal_(mean, std, generator=self.g)
        return t.to(dtype)

    def linear(self, n_out: int, n_in: int) -> LinearDev:
        w = self.normal((n_out, n_in), 0.02, dtype=torch.bfloat16)
        b = self.normal((n_out,), 0.02).to(torch.bfloat16).float()
        return LinearDev(w, b)

    def gain(self, d: int) -> torch.Tensor:
        return self.normal((d,), 0.02, 1.0)

    def double(self, D: int, d: int, Dm: int, swiglu: bool = False) -> DoubleWeights:
        mk = lambda n_out, n_in: [self.linear(n_out, n_in) for _ in range(2)]
        return DoubleWeights(mk(6 * D, D), mk(3 * D, D), mk(D, D), mk((2 if swiglu else 1) * Dm, D), mk(D, Dm),
                             [self.gain(d), self.gain(d)], [self.gain(d), self.gain(d)])

    def single(self, D: int, d: int, Dm: int, swiglu: bool = False) -> SingleWeights:
        return SingleWeights(self.linear(3 * D, D), self.linear(3 * D + (2 if swiglu else 1) * Dm, D),
                             self.linear(D, D + Dm), self.gain(d), self.gain(d))

    def step(self, D: int, d: int, Dm: int, C_lat: int, t_dim: int, n_double: int, n_single: int,
             swiglu: bool = False) -> StepWeights:
        return StepWeights(self.linear(D, t_dim), self.linear(D, D), self.linear(D, C_lat), self.linear(2 * D, D),
                           self.linear(C_lat, D), [self.double(D, d, Dm, swiglu) for _ in range(n_double)],
                           [self.single(D, d, Dm, swiglu) for _ in range(n_single)])

    def cond(self, D: int, t_dim: int, C_txt: int, C_pool: int) -> CondWeights:
        return CondWeights(self.linear(D, C_txt), self.linear(D, t_dim), self.linear(D, D), self.linear(D, C_pool),
                           self.linear(D, D))

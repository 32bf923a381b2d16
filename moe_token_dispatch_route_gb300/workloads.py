"""Seeded synthetic workloads for the MoE dispatch + grouped-GEMM path.

This module only draws random inputs; it holds none of the routing, dispatch
or GEMM arithmetic.  Both the CUDA path and the CPU oracle take their inputs
from here.

Every workload is a Mixture-of-Experts up-projection layer:
  T tokens of width d (x, bf16), E experts with top-k routing, expert weights
  W[E][d][N] (bf16), R simulated expert ranks (E % R == 0).
x ~ N(0, 1); the router matrix W_r [d, E] and the expert weights ~ N(0, 1/d),
all rounded to bf16 with round-to-nearest-even.  Router logits are the input
of the routing step: L = fp32(x @ W_r summed in fp64) + bias, one rounding to
fp32, then the fp32 bias added in fp32.

Seeds: x uses `seed`, W_r `seed + 1`, W `seed + 2`, the bias draw `seed + 3`.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    N: int
    R: int = 1
    bias: str = "none"   # "none" | "zipf" | "hot4"
    note: str = ""

    @property
    def S(self) -> int:
        return self.T * self.k

    @property
    def flops(self) -> float:
        """2 * S * d * N: the grouped GEMM's multiply-adds, the only FLOPs of the path."""
        return 2.0 * self.S * self.d * self.N

    def describe(self) -> dict:
        return {"workload": self.name, "T": self.T, "d": self.d, "E": self.E, "k": self.k,
                "N": self.N, "ranks": self.R, "router_bias": self.bias}


WORKLOADS = {
    "tiny": Workload("tiny", 256, 512, 8, 2, 1024, 1, "none",
                     "tiny MoE up-projection"),
    "mixtral": Workload("mixtral", 8192, 4096, 8, 2, 14336, 1, "none",
                        "Mixtral-shaped up-projection, near-uniform load"),
    "finegrained": Workload("finegrained", 16384, 2048, 64, 4, 1408, 1, "zipf",
                            "fine-grained MoE, Zipf(s=1.1) expert load, some experts empty"),
    "deepseek_v3": Workload("deepseek_v3", 4096, 7168, 256, 8, 2048, 16, "none",
                            "DeepSeek-V3-shaped layer over 16 simulated rank buffers"),
    "decode": Workload("decode", 64, 4096, 128, 8, 1536, 1, "hot4",
                       "decode-sized batch, half the routing mass on 4 hot experts"),
}


def custom(name: str, T: int, d: int, E: int, k: int, N: int, R: int = 1, bias: str = "none") -> Workload:
    return Workload(name, T, d, E, k, N, R, bias)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def router_bias(wl: Workload, seed: int = 0) -> torch.Tensor:
    """fp32 [E] router bias for the workload's load pattern.

    zipf: expert at popularity rank r (a seeded random permutation decides which
      expert has which rank) gets ln(p_r), p_r proportional to (r+1)^-1.1; the 4
      least popular experts get -30 so that they surely receive no token.
    hot4: 4 seeded experts get +16 (the other logits are ~N(0,1)), so each
      token's top-k holds all four: half the routing mass at k=8.
    """
    E = wl.E
    b = torch.zeros(E, dtype=torch.float32)
    if wl.bias == "none":
        return b
    order = torch.randperm(E, generator=_gen(seed + 3))
    if wl.bias == "zipf":
        ranks = np.arange(1, E + 1, dtype=np.float64)
        p = ranks ** -1.1
        p /= p.sum()
        lp = np.log(p)
        if E > 4:
            lp[-4:] = -30.0
        b[order] = torch.from_numpy(lp.astype(np.float32))
        return b
    if wl.bias == "hot4":
        b[order[:4]] = 16.0
        return b
    raise ValueError(wl.bias)


def hot_experts(wl: Workload, seed: int = 0) -> list[int]:
    order = torch.randperm(wl.E, generator=_gen(seed + 3))
    return sorted(int(e) for e in order[:4])


def make_x(wl: Workload, seed: int = 0) -> torch.Tensor:
    return torch.randn(wl.T, wl.d, generator=_gen(seed)).to(torch.bfloat16)


def make_router(wl: Workload, seed: int = 0) -> torch.Tensor:
    return (torch.randn(wl.d, wl.E, generator=_gen(seed + 1)) / math.sqrt(wl.d)).to(torch.bfloat16)


def make_logits(x: torch.Tensor, W_r: torch.Tensor, bias: torch.Tensor) -> torch.Tensor:
    """Router logits (input preparation, not part of the timed path):
    fp64 product of the bf16 values, rounded once to fp32, plus the fp32 bias."""
    L = (x.double() @ W_r.double()).to(torch.float32)
    return (L + bias.to(torch.float32)).contiguous()


def make_weights(wl: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    """Expert weights W [E, d, N] bf16, drawn expert by expert on `device`."""
    dev = torch.device(device)
    g = _gen(seed + 2, dev)
    W = torch.empty(wl.E, wl.d, wl.N, dtype=torch.bfloat16, device=dev)
    scale = 1.0 / math.sqrt(wl.d)
    for e in range(wl.E):
        W[e] = (torch.randn(wl.d, wl.N, generator=g, device=dev) * scale).to(torch.bfloat16)
    return W


def _normal_bf16(shape, scale: float, seed: int, device) -> torch.Tensor:
    dev = torch.device(device)
    g = _gen(seed, dev)
    out = torch.empty(*shape, dtype=torch.bfloat16, device=dev)
    for e in range(shape[0]):  # one slice at a time: no fp32 copy of the whole tensor
        out[e] = (torch.randn(*shape[1:], generator=g, device=dev) * scale).to(torch.bfloat16)
    return out


def make_ffn_weights(wl: Workload, F: int, seed: int = 0, device="cpu"):
    """Gated expert FFN weights, bf16: W1 [E, d, 2F] ~ N(0, 1/d) with the gate
    projection in columns [0, F) and the up projection in [F, 2F) (seed + 4), and
    the down projection W2 [E, F, d] ~ N(0, 1/F) (seed + 5)."""
    W1 = _normal_bf16((wl.E, wl.d, 2 * F), 1.0 / math.sqrt(wl.d), seed + 4, device)
    W2 = _normal_bf16((wl.E, F, wl.d), 1.0 / math.sqrt(F), seed + 5, device)
    return W1, W2


def make_rows(S: int, width: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Rows already in destination order for the grouped GEMM alone: bf16 [S, width]
    ~ N(0, 1/4) (the spread of silu(g) * u for g, u ~ N(0, 1)), seed + 6."""
    dev = torch.device(device)
    g = _gen(seed + 6, dev)
    out = torch.empty(S, width, dtype=torch.bfloat16, device=dev)
    for r0 in range(0, S, 1024):  # blocks of rows: no fp32 copy of the whole tensor
        r1 = min(S, r0 + 1024)
        out[r0:r1] = (torch.randn(r1 - r0, width, generator=g, device=dev) * 0.5).to(torch.bfloat16)
    return out


def make_inputs(wl: Workload, seed: int = 0, w_device="cpu", with_weights: bool = True) -> dict:
    """All inputs of one step: x, W_r, bias, logits on the host; W on `w_device`."""
    x = make_x(wl, seed)
    W_r = make_router(wl, seed)
    bias = router_bias(wl, seed)
    logits = make_logits(x, W_r, bias)
    out = {"x": x, "W_r": W_r, "bias": bias, "logits": logits}
    if with_weights:
        out["W"] = make_weights(wl, seed, w_device)
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

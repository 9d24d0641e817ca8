"""Seeded synthetic inputs for the chunked gated delta rule.

This module holds only the input recipe (distributions, shapes, seeds) and
none of the method's arithmetic; both the device path and the fp64 oracle
read the values it produces.

Recipe (the workloads the pages train on are synthetic-data runs of a
Qwen3-Next-shaped GDN layer: 16 key heads shared by 32 value heads, head dim
128, chunk 128; PR "Fuse the Gated Delta Net inter-chunk scan into a Pallas
TPU kernel", section "Performance"):
  q, k ~ N(0, 1), then L2-normalised per token and head, rounded to bf16 (RNE)
  v    ~ N(0, 1), bf16
  beta = sigmoid(N(0, 1)), fp32
  g    = -softplus(N(0, 1) + shift), fp32 (log-gate per token and value head)
  h0   ~ N(0, h0_std^2) fp32 per value head (absent when h0_std == 0)
  dO   ~ N(0, 1) bf16 and dhT ~ N(0, 0.1^2) fp32 (backward workloads)

Host generation (numpy) draws, for each batch row b and block of 65,536
tokens, from default_rng([seed, b, block]) in the order q, k, v, beta-logit,
g-logit, dO; h0 and dhT come from default_rng([seed, 1 << 20]).  Device
generation (torch, for the million-token sizes where host generation takes
minutes) follows the same distributions with torch's CUDA generator seeded
per block; its values differ from the host stream, and every consumer reads
the generated tensors themselves.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

TOKEN_BLOCK = 1 << 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hk: int
    Hv: int
    dk: int = 128
    dv: int = 128
    chunk: int = 128
    gate_shift: float = 0.0
    h0_std: float = 0.0
    seed: int = 0
    n_segments: int = 0  # 0: let the library choose
    backward: bool = False

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, by what they are.
WORKLOADS = {
    "tiny_t1024": Workload("tiny_t1024", B=1, T=1024, Hk=2, Hv=2),
    "layer_t4096": Workload("layer_t4096", B=1, T=4096, Hk=16, Hv=32,
                            gate_shift=1.0, h0_std=0.1, backward=True),
    "batched_b2_t8192": Workload("batched_b2_t8192", B=2, T=8192, Hk=16, Hv=32,
                                 backward=True),
    "long_t262144": Workload("long_t262144", B=1, T=262144, Hk=16, Hv=32,
                             h0_std=0.1, n_segments=148, backward=True),
    "million_t1048576": Workload("million_t1048576", B=1, T=1048576, Hk=16, Hv=32,
                                 gate_shift=3.0, n_segments=148),
    # the slow-decay reading of the million-token workload (g ~ -0.05 per token)
    "million_t1048576_slow": Workload("million_t1048576_slow", B=1, T=1048576, Hk=16,
                                      Hv=32, gate_shift=-3.0, h0_std=0.1, n_segments=148),
}


@dataclasses.dataclass
class Inputs:
    """Tensors of one workload.  bf16 tensors are torch.bfloat16."""
    wl: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    dO: Optional[torch.Tensor] = None
    dhT: Optional[torch.Tensor] = None

    def to(self, device) -> "Inputs":
        f = lambda x: None if x is None else x.to(device)
        return Inputs(self.wl, f(self.q), f(self.k), f(self.v), f(self.g), f(self.beta),
                      f(self.h0), f(self.dO), f(self.dhT))

    def bits(self, name: str) -> np.ndarray:
        """bf16 tensor as a host uint16 array of its bit patterns."""
        x = getattr(self, name)
        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    def f32(self, name: str) -> Optional[np.ndarray]:
        x = getattr(self, name)
        return None if x is None else x.detach().cpu().contiguous().numpy().astype(np.float32)


def _softplus(x):
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def _to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def make_host(wl: Workload, backward: Optional[bool] = None) -> Inputs:
    """Generate on the host with numpy (bit-reproducible on any machine)."""
    bwd = wl.backward if backward is None else backward
    B, T, Hk, Hv, dk, dv = wl.B, wl.T, wl.Hk, wl.Hv, wl.dk, wl.dv
    q = np.empty((B, T, Hk, dk), np.float32)
    k = np.empty((B, T, Hk, dk), np.float32)
    v = np.empty((B, T, Hv, dv), np.float32)
    g = np.empty((B, T, Hv), np.float32)
    beta = np.empty((B, T, Hv), np.float32)
    dO = np.empty((B, T, Hv, dv), np.float32) if bwd else None
    for b in range(B):
        for blk, t0 in enumerate(range(0, T, TOKEN_BLOCK)):
            t1 = min(T, t0 + TOKEN_BLOCK)
            n = t1 - t0
            rng = np.random.default_rng([wl.seed, b, blk])
            q[b, t0:t1] = _unit_rows(rng.standard_normal((n, Hk, dk)))
            k[b, t0:t1] = _unit_rows(rng.standard_normal((n, Hk, dk)))
            v[b, t0:t1] = rng.standard_normal((n, Hv, dv))
            bl = rng.standard_normal((n, Hv))
            gl = rng.standard_normal((n, Hv))
            beta[b, t0:t1] = 1.0 / (1.0 + np.exp(-bl))
            g[b, t0:t1] = -_softplus(gl + wl.gate_shift)
            if bwd:
                dO[b, t0:t1] = rng.standard_normal((n, Hv, dv))
    srng = np.random.default_rng([wl.seed, 1 << 20])
    h0 = srng.standard_normal((B, Hv, dk, dv)) * wl.h0_std
    dhT = srng.standard_normal((B, Hv, dk, dv)) * 0.1
    return Inputs(
        wl, _to_bf16(q), _to_bf16(k), _to_bf16(v),
        torch.from_numpy(g), torch.from_numpy(beta),
        torch.from_numpy(h0.astype(np.float32)) if wl.h0_std > 0 else None,
        _to_bf16(dO) if bwd else None,
        torch.from_numpy(dhT.astype(np.float32)) if bwd else None)


def make_device(wl: Workload, device, backward: Optional[bool] = None) -> Inputs:
    """Generate directly on a device with torch (fast at million-token sizes)."""
    bwd = wl.backward if backward is None else backward
    B, T, Hk, Hv, dk, dv = wl.B, wl.T, wl.Hk, wl.Hv, wl.dk, wl.dv
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    bf = torch.bfloat16
    q = torch.empty((B, T, Hk, dk), dtype=bf, device=dev)
    k = torch.empty_like(q)
    v = torch.empty((B, T, Hv, dv), dtype=bf, device=dev)
    g = torch.empty((B, T, Hv), dtype=torch.float32, device=dev)
    beta = torch.empty_like(g)
    dO = torch.empty_like(v) if bwd else None
    for b in range(B):
        for blk, t0 in enumerate(range(0, T, TOKEN_BLOCK)):
            t1 = min(T, t0 + TOKEN_BLOCK)
            n = t1 - t0
            gen.manual_seed((wl.seed * 1_000_003 + b) * 65_537 + blk)
            r = lambda *s: torch.randn(*s, generator=gen, device=dev, dtype=torch.float32)
            x = r(n, Hk, dk)
            q[b, t0:t1] = (x / x.norm(dim=-1, keepdim=True)).to(bf)
            x = r(n, Hk, dk)
            k[b, t0:t1] = (x / x.norm(dim=-1, keepdim=True)).to(bf)
            v[b, t0:t1] = r(n, Hv, dv).to(bf)
            beta[b, t0:t1] = torch.sigmoid(r(n, Hv))
            g[b, t0:t1] = -torch.nn.functional.softplus(r(n, Hv) + wl.gate_shift)
            if bwd:
                dO[b, t0:t1] = r(n, Hv, dv).to(bf)
    gen.manual_seed(wl.seed * 1_000_003 + 999_983)
    h0 = (torch.randn((B, Hv, dk, dv), generator=gen, device=dev) * wl.h0_std
          if wl.h0_std > 0 else None)
    dhT = torch.randn((B, Hv, dk, dv), generator=gen, device=dev) * 0.1 if bwd else None
    return Inputs(wl, q, k, v, g, beta, h0, dO, dhT)


@dataclasses.dataclass
class LayerInputs:
    """Raw inputs of one GatedDeltaNet layer's use of the rule: q, k
    unnormalised, a and b the gate logits (g = -softplus(a), beta =
    sigmoid(b)), z the output gate, and the backward's cotangents."""
    wl: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    a: torch.Tensor
    b: torch.Tensor
    z: torch.Tensor
    h0: Optional[torch.Tensor]
    dy: torch.Tensor
    dhT: torch.Tensor

    def to(self, device) -> "LayerInputs":
        f = lambda x: None if x is None else x.to(device)
        return LayerInputs(self.wl, f(self.q), f(self.k), f(self.v), f(self.a), f(self.b),
                           f(self.z), f(self.h0), f(self.dy), f(self.dhT))


def make_layer_host(wl: Workload, qk_scale: float = 3.0) -> LayerInputs:
    """Raw layer inputs on the host: q, k ~ N(0, qk_scale^2) (not normalised),
    v, z, dy ~ N(0, 1) (bf16), a ~ N(gate_shift, 1) and b ~ N(0, 1) (fp32
    logits), h0 ~ N(0, h0_std^2), dhT ~ N(0, 0.1^2); one default_rng([seed, 7])
    stream in that order."""
    B, T, Hk, Hv, dk, dv = wl.B, wl.T, wl.Hk, wl.Hv, wl.dk, wl.dv
    rng = np.random.default_rng([wl.seed, 7])
    q = rng.standard_normal((B, T, Hk, dk)) * qk_scale
    k = rng.standard_normal((B, T, Hk, dk)) * qk_scale
    v = rng.standard_normal((B, T, Hv, dv))
    a = rng.standard_normal((B, T, Hv)) + wl.gate_shift
    b = rng.standard_normal((B, T, Hv))
    z = rng.standard_normal((B, T, Hv, dv))
    h0 = rng.standard_normal((B, Hv, dk, dv)) * wl.h0_std
    dy = rng.standard_normal((B, T, Hv, dv))
    dhT = rng.standard_normal((B, Hv, dk, dv)) * 0.1
    f32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32))
    return LayerInputs(wl, _to_bf16(q), _to_bf16(k), _to_bf16(v), f32(a), f32(b), _to_bf16(z),
                       f32(h0) if wl.h0_std > 0 else None, _to_bf16(dy), f32(dhT))


__all__ = ["Workload", "WORKLOADS", "Inputs", "make_host", "make_device", "LayerInputs",
           "make_layer_host"]

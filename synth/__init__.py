"""Seeded synthetic inputs for the fused gated-GLU + quantisation path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no activation, no scale, no encoding).  Both the CUDA
path's tests/bench and the CPU oracle consume what it makes: inputs are drawn
once (on the device for large shapes) and the oracle sees a host copy of the
very same bf16 bytes.

Workloads (shapes and value distributions of the pages' benchmarks; no
dataset or trained weight is involved):
  * swiglu_128     : gate, up [128, 128] ~ N(0,1)
  * swiglu_4096    : gate, up, dY [4096, 7168] ~ N(0,1)
  * geglu_8192     : gate, up [8192, N] ~ N(0,1), dY ~ 0.1 N(0,1),
                     N in {11008, 14336, 18944, 29568}
  * geglu_nvfp4    : X [M, 32768] ~ 2 N(0,1), gate/up interleaved by column
                     pairs, M in {784, 968}
  * swiglu_131072  : gate, up, dY [131072, 8192] ~ N(0,1) with 0.1 % of the
                     elements of each tensor set to +-60
Seeds: gate 1000+c, up 2000+c, dY 3000+c, spike mask 4000+c (c = workload
index 0..4), plus an optional offset (per rank, per repeat).
"""
from __future__ import annotations

import dataclasses

import torch

WORKLOADS = ("swiglu_128", "swiglu_4096", "geglu_8192", "geglu_nvfp4", "swiglu_131072")


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    index: int
    M: int
    N: int
    interleaved: bool = False
    scale: float = 1.0
    dy_scale: float = 1.0
    spikes: bool = False


def spec(name: str, M: int | None = None, N: int | None = None) -> Spec:
    if name == "swiglu_128":
        return Spec(name, 0, M or 128, N or 128)
    if name == "swiglu_4096":
        return Spec(name, 1, M or 4096, N or 7168)
    if name == "geglu_8192":
        return Spec(name, 2, M or 8192, N or 14336, dy_scale=0.1)
    if name == "geglu_nvfp4":
        return Spec(name, 3, M or 784, N or 16384, interleaved=True, scale=2.0)
    if name == "swiglu_131072":
        return Spec(name, 4, M or 131072, N or 8192, spikes=True)
    raise KeyError(name)


_CHUNK = 1 << 26  # elements drawn per generator call (bounds temporary memory)


def _normal_bf16(shape, seed: int, scale: float, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - s)
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        flat[s:s + n].copy_(x)  # fp32 -> bf16, round to nearest even
    return out


def _add_spikes(t: torch.Tensor, seed: int, value: float = 60.0, rate: float = 1e-3) -> None:
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    flat = t.view(-1)
    for s in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - s)
        r = torch.rand(n, generator=g, device=t.device)
        sgn = torch.rand(n, generator=g, device=t.device)
        mask = r < rate
        vals = torch.where(sgn < 0.5, torch.full_like(r, -value), torch.full_like(r, value))
        seg = flat[s:s + n]
        seg[mask] = vals[mask].to(torch.bfloat16)


def make(sp: Spec, device="cpu", with_dy: bool = False, seed_offset: int = 0) -> dict:
    """Draw the inputs of one workload.  Returns bf16 tensors:
    split layout: {"gate": [M,N], "up": [M,N], "dy": [M,N]?};
    interleaved:  {"x": [M,2N], "dy": [M,N]?}."""
    c = sp.index
    off = seed_offset
    res = {}
    if sp.interleaved:
        res["x"] = _normal_bf16((sp.M, 2 * sp.N), 1000 + c + off, sp.scale, device)
        if sp.spikes:
            _add_spikes(res["x"], 4000 + c + off)
    else:
        res["gate"] = _normal_bf16((sp.M, sp.N), 1000 + c + off, sp.scale, device)
        res["up"] = _normal_bf16((sp.M, sp.N), 2000 + c + off, sp.scale, device)
        if sp.spikes:
            _add_spikes(res["gate"], 4000 + c + off)
            _add_spikes(res["up"], 4100 + c + off)
    if with_dy:
        res["dy"] = _normal_bf16((sp.M, sp.N), 3000 + c + off, sp.dy_scale, device)
        if sp.spikes:
            _add_spikes(res["dy"], 4200 + c + off)
    return res


def to_host_bits(t: torch.Tensor):
    """A host numpy uint16 copy of a bf16 tensor's bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")

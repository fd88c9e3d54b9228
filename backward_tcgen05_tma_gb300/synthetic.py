"""Seeded synthetic inputs for the SwiGLU MLP (shared by the tests, the oracle
checks and the benchmark).

This module draws random numbers and nothing else: it holds none of the MLP's
arithmetic.  Two generators:

* ``counter_normal`` -- a counter-based stream, value i of (seed, tensor id)
  is a pure function of those three integers: SplitMix64 (Steele, Lea and
  Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014; state
  advanced by the golden-ratio increment, then the 64-bit finaliser) gives two
  uniforms in (0, 1], and the Box-Muller transform turns them into a standard
  normal.  It is stable across numpy/torch versions and machines, so small
  stored cases can be regenerated anywhere.  numpy, vectorised; used up to a
  few tens of millions of elements.
* ``device_normal`` -- torch's seeded generator on the target device, for the
  full-size workloads (hundreds of millions of elements) where the counter
  stream would be slow on the host.  Both sides of a comparison still get the
  same bytes because they are drawn once and copied.

Distributions follow the workloads' recipe: X ~ N(0, 1); Wg, Wu ~ N(0, 1/D);
Wd ~ N(0, 1/H) (the second parameter is the variance); dY ~ N(0, 1e-2), or
N(0, 1) for the tiny fp32 case.  Values are drawn in fp64 (counter) or fp32
(device), scaled by the standard deviation and cast once to the storage type
by torch.
"""
from __future__ import annotations

import math

import numpy as np

# tensor ids of the counter streams
TID_X, TID_WG, TID_WU, TID_WD, TID_DY = 0, 1, 2, 3, 4

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _splitmix64(state: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser applied to (state + gamma); uint64 arithmetic wraps."""
    z = state + _GAMMA
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def counter_uniform(seed: int, tid: int, n: int, offset: int = 0) -> np.ndarray:
    """n uniforms in (0, 1]: element i uses SplitMix64 state
    base + (offset + i) * gamma, with base = splitmix64(seed * 2^8 + tid)."""
    with np.errstate(over="ignore"):
        base = _splitmix64(np.array([(seed << 8) + tid], dtype=np.uint64))[0]
        idx = np.arange(offset, offset + n, dtype=np.uint64)
        bits = _splitmix64(base + idx * _GAMMA)
    return ((bits >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def counter_normal(seed: int, tid: int, n: int) -> np.ndarray:
    """n standard normals (fp64) from the counter stream: Box-Muller on the
    uniform pair (2i, 2i + 1)."""
    u = counter_uniform(seed, tid, 2 * n)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def counter_grid(seed: int, tid: int, n: int, half: int, scale: float) -> np.ndarray:
    """n values k * scale with k uniform on the integers {-half, ..., half}."""
    u = counter_uniform(seed, tid, n)
    k = np.minimum(np.floor((1.0 - u) * (2 * half + 1)), 2 * half) - half
    return k * scale


def _torch_dtype(name: str):
    import torch
    return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[name]


def dy_std_for(dtype: str) -> float:
    """dY ~ N(0, 1) in the fp32 tiny case, N(0, 1e-2) (std 0.1) otherwise."""
    return 1.0 if dtype == "f32" else 0.1


def make_inputs(M: int, D: int, H: int, dtype: str = "bf16", seed: int = 0,
                dy_std: float | None = None, device: str = "cpu", kind: str = "counter"):
    """Synthetic X [M,D], Wg/Wu [H,D], Wd [D,H], dY [M,D] as torch tensors of
    the storage dtype on ``device``.  Also returns Wgu = [Wg; Wu] ([2H, D]).

    kind="counter": counter stream (host, stable);  kind="device": torch's
    generator on ``device``;  kind="grid": exact-accumulation inputs on a coarse
    dyadic grid (X in {-4..4}/4, Wg/Wu/Wd in {-8..8}/64, dY in {-4..4}/64),
    for which every fp32 partial sum of the contractions is exact.
    """
    import torch
    tdt = _torch_dtype(dtype)
    if dy_std is None:
        dy_std = dy_std_for(dtype)
    shapes = {TID_X: (M, D), TID_WG: (H, D), TID_WU: (H, D), TID_WD: (D, H), TID_DY: (M, D)}
    stds = {TID_X: 1.0, TID_WG: D ** -0.5, TID_WU: D ** -0.5, TID_WD: H ** -0.5, TID_DY: dy_std}
    out = {}
    for tid, shape in shapes.items():
        n = shape[0] * shape[1]
        if kind == "counter":
            v = counter_normal(seed, tid, n) * stds[tid]
            t = torch.from_numpy(v.reshape(shape)).to(tdt).to(device)
        elif kind == "grid":
            if tid == TID_X:
                v = counter_grid(seed, tid, n, 4, 0.25)
            elif tid == TID_DY:
                v = counter_grid(seed, tid, n, 4, 1.0 / 64)
            else:
                v = counter_grid(seed, tid, n, 8, 1.0 / 64)
            t = torch.from_numpy(v.reshape(shape)).to(tdt).to(device)
        elif kind == "device":
            t = device_normal(shape, stds[tid], dtype, seed, tid, device)
        else:
            raise ValueError(kind)
        out[{TID_X: "X", TID_WG: "Wg", TID_WU: "Wu", TID_WD: "Wd", TID_DY: "dY"}[tid]] = t
    out["Wgu"] = torch.cat([out["Wg"], out["Wu"]], dim=0).contiguous()
    return out


def device_normal(shape, std: float, dtype: str, seed: int, tid: int, device: str):
    """N(0, std^2) drawn by torch's generator on ``device`` (fp32), cast once."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + tid)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(_torch_dtype(dtype))

"""Seeded synthetic inputs for the TSP layer.

This module is the only code shared by the CUDA path's tests/benchmark and the
fp64 oracle's tests.  It holds none of the layer's arithmetic: it draws
normal variates from a counter-based generator and rounds them to the storage
dtype, nothing else.

Generator (stated here so each side could re-implement it):

* splitmix64 mix:  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
                   z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
  (all arithmetic modulo 2**64).
* A stream with seed ``s0`` yields, for counter i = 0, 1, ..., the value
  ``mix(s0 + (i + 1) * 0x9E3779B97F4A7C15)`` -- the classic splitmix64
  sequence started from state ``s0``.
* Tensor ``k`` of a workload with base seed ``seed`` uses the stream seed
  ``mix(seed * 1000 + k + 0x9E3779B97F4A7C15)`` (the first splitmix64 output
  of state ``seed * 1000 + k``).  Tensor ids: x=0, W_Q=1, W_K=2, W_V=3,
  W_O=4, W_gate=5, W_up=6, W_down=7, dY=8.
* Normals by Box-Muller on consecutive pairs (u1, u2):
  u1 = ((z1 >> 11) + 1) * 2**-53 in (0, 1],  u2 = (z2 >> 11) * 2**-53,
  n0 = sqrt(-2 ln u1) cos(2 pi u2),  n1 = sqrt(-2 ln u1) sin(2 pi u2).
* Values are scaled by ``std`` in fp64 and rounded once, round-to-nearest-
  even, to the storage dtype (bf16 or fp32).  Both sides consume the rounded
  values, so any error measured afterwards is computation, not input rounding.

Workload distributions follow the layer definition used throughout:
x ~ N(0, 1); every weight ~ N(0, 1/fan_in) with fan_in = hidden for
W_Q, W_K, W_V, W_O, W_gate, W_up and fan_in = ffn for W_down; dY ~ N(0, 1).
"""

from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

TENSOR_IDS = {"x": 0, "Wq": 1, "Wk": 2, "Wv": 3, "Wo": 4, "Wg": 5, "Wu": 6, "Wd": 7, "dY": 8}


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def stream_seed(seed: int, k: int) -> int:
    s = np.array([(seed * 1000 + k) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    with np.errstate(over="ignore"):
        return int(_mix(s + GOLDEN)[0])


def uniform_u64(s0: int, start: int, n: int) -> np.ndarray:
    """Counter outputs ``start .. start+n-1`` of the splitmix64 stream ``s0``."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(s0) + i * GOLDEN)


def normals(s0: int, n: int) -> np.ndarray:
    """``n`` standard normal fp64 variates from stream ``s0`` (Box-Muller)."""
    out = np.empty(n, dtype=np.float64)
    npairs = (n + 1) // 2
    scale = 2.0 ** -53
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        z = uniform_u64(s0, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
        u1 = ((z[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * scale
        u2 = (z[:, 1] >> np.uint64(11)).astype(np.float64) * scale
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        pair = np.empty((p1 - p0, 2), dtype=np.float64)
        pair[:, 0] = r * np.cos(t)
        pair[:, 1] = r * np.sin(t)
        flat = pair.reshape(-1)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = flat[: hi - lo]
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values RNE to the nearest bf16; returns fp64 holding them.

    Rounds directly on the fp64 bit pattern (52 -> 7 mantissa bits), so there
    is no double rounding through fp32.  Inputs here are finite and inside the
    normal bf16 range (or zero).
    """
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    drop = np.uint64(45)
    lsb = (b >> drop) & np.uint64(1)
    with np.errstate(over="ignore"):
        b = (b + (np.uint64((1 << 44) - 1) + lsb)) & ~np.uint64((1 << 45) - 1)
    return b.view(np.float64)


def bf16_bits(x_rounded: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of values already rounded by ``round_bf16``."""
    f = np.ascontiguousarray(x_rounded, dtype=np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def tensor(name: str, shape, std: float, dtype: str, seed: int = 0) -> np.ndarray:
    """One seeded tensor, fp64 array holding values exactly representable in ``dtype``."""
    n = int(np.prod(shape))
    v = normals(stream_seed(seed, TENSOR_IDS[name]), n) * std
    if dtype == "bf16":
        v = round_bf16(v)
    elif dtype == "f32":
        v = v.astype(np.float32).astype(np.float64)
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    return v.reshape(shape)


def layer_inputs(cfg, seed: int = 0, with_dy: bool = False, only=None) -> dict:
    """All inputs of one TSP layer workload as fp64 arrays (values rounded to ``cfg.dtype``).

    Canonical weight layout, row-vector convention y = x @ W:
    Wq, Wo: [h, h]; Wk, Wv: [h, hk] (hk = K/V heads * head_dim, h unless the
    workload uses grouped-query attention); Wg, Wu: [h, F]; Wd: [F, h];
    x (and dY): [B, S, h].
    """
    h, F = cfg.hidden, cfg.ffn
    hk = cfg.kv_hidden
    spec = {
        "x": ((cfg.batch, cfg.seq, h), 1.0),
        "Wq": ((h, h), h ** -0.5),
        "Wk": ((h, hk), h ** -0.5),
        "Wv": ((h, hk), h ** -0.5),
        "Wo": ((h, h), h ** -0.5),
        "Wg": ((h, F), h ** -0.5),
        "Wu": ((h, F), h ** -0.5),
        "Wd": ((F, h), F ** -0.5),
    }
    if with_dy:
        spec["dY"] = ((cfg.batch, cfg.seq, h), 1.0)
    names = list(spec) if only is None else list(only)
    return {k: tensor(k, spec[k][0], spec[k][1], cfg.dtype, seed) for k in names}


# ---------------------------------------------------------------------------
# The same generator in torch int64 arithmetic, for filling large benchmark
# inputs directly in device memory.  Integer steps are identical to the numpy
# version (modulo-2**64 wrap-around, logical shifts emulated with masks); the
# fp64 log/cos/sin of the device may differ from the host's libm in the last
# ulp, so tests that compare against the oracle draw their inputs with the
# numpy functions above and copy them to the device.
# ---------------------------------------------------------------------------

def _i64(u: int) -> int:
    u &= 0xFFFFFFFFFFFFFFFF
    return u - (1 << 64) if u >= (1 << 63) else u


def _mix_torch(z):
    import torch  # noqa: F401  (torch is the caller's dependency here)
    z = z ^ ((z >> 30) & ((1 << 34) - 1))
    z = z * _i64(0xBF58476D1CE4E5B9)
    z = z ^ ((z >> 27) & ((1 << 37) - 1))
    z = z * _i64(0x94D049BB133111EB)
    return z ^ ((z >> 31) & ((1 << 33) - 1))


def normals_torch(s0: int, n: int, device):
    import torch
    out = torch.empty(n, dtype=torch.float64, device=device)
    npairs = (n + 1) // 2
    chunk = 1 << 24
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        i = torch.arange(2 * p0 + 1, 2 * p1 + 1, dtype=torch.int64, device=device)
        z = _mix_torch(i * _i64(int(GOLDEN)) + _i64(s0)).view(-1, 2)
        u1 = (((z[:, 0] >> 11) & ((1 << 53) - 1)).to(torch.float64) + 1.0) * 2.0 ** -53
        u2 = ((z[:, 1] >> 11) & ((1 << 53) - 1)).to(torch.float64) * 2.0 ** -53
        r = torch.sqrt(-2.0 * torch.log(u1))
        t = 2.0 * torch.pi * u2
        pair = torch.stack([r * torch.cos(t), r * torch.sin(t)], dim=1).view(-1)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = pair[: hi - lo]
    return out


def tensor_torch(name: str, shape, std: float, dtype: str, seed: int = 0, device="cuda"):
    """Like ``tensor`` but produced by torch on ``device``, returned in the storage dtype."""
    import torch
    n = 1
    for s in shape:
        n *= int(s)
    v = normals_torch(stream_seed(seed, TENSOR_IDS[name]), n, device) * std
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return v.to(tdt).view(*shape)

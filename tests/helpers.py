"""Shared test helpers: device transfer of seeded inputs and error metrics."""
import numpy as np

try:
    import torch
except ImportError:  # pragma: no cover
    torch = None

BF16_TOL = 2e-2  # relative Frobenius error, bf16 operands with fp32 accumulation
F32_TOL = 1e-4   # normwise max relative error, fp32


def to_dev(a, dtype: str, device="cuda"):
    """fp64 array holding values exact in `dtype` -> device tensor of that dtype (bit-exact)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.to(device)


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_frob(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def max_rel(got, ref):
    """max |g - r| / max |r| (normwise max relative error)."""
    return float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))


def check(got, ref, dtype: str, what: str):
    if dtype == "bf16":
        e = rel_frob(got, ref)
        print(f"PARITY {what}: relative Frobenius {e:.3e} (bound {BF16_TOL})")
        assert e <= BF16_TOL, f"{what}: relative Frobenius error {e:.3e} > {BF16_TOL}"
    else:
        e = max_rel(got, ref)
        print(f"PARITY {what}: max relative {e:.3e} (bound {F32_TOL})")
        assert e <= F32_TOL, f"{what}: max relative error {e:.3e} > {F32_TOL}"
    return e

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


# ---- canary guard bands ---------------------------------------------------------
# With compute-sanitizer unavailable, out-of-bounds writes are caught by placing
# each output (and each workspace) inside a larger device buffer whose bytes
# before and after it hold a fixed pattern; after the call the pattern must be
# intact.  64 KiB on each side covers more than one 128-row tile of any row
# width these tests use past either end.
GUARD_BYTES = 64 << 10


class Guarded:
    """A device tensor of `shape`/`dtype` (`.t`) with guard bands on both sides.

    The tensor itself starts filled with `fill` (NaN by default for floating
    types, so an element the call never writes also shows up in the parity
    checks); `check()` asserts the guard bands still hold their pattern.
    """

    def __init__(self, shape, dtype, device="cuda", fill="nan"):
        import torch

        esz = torch.empty((), dtype=dtype).element_size()
        n = 1
        for d in shape:
            n *= int(d)
        self.nbytes = n * esz
        total = 2 * GUARD_BYTES + self.nbytes
        idx = torch.arange(GUARD_BYTES, device=device, dtype=torch.int64)
        self.head = ((idx * 37 + 11) % 251).to(torch.uint8)
        self.tail = ((idx * 53 + 7) % 241).to(torch.uint8)
        self.buf = torch.empty(total, dtype=torch.uint8, device=device)
        self.buf[:GUARD_BYTES] = self.head
        self.buf[GUARD_BYTES + self.nbytes:] = self.tail
        self.t = self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(tuple(shape))
        if fill == "nan" and dtype.is_floating_point:
            self.t.fill_(float("nan"))
        elif fill is not None and fill != "nan":
            self.t.fill_(fill)

    def check(self, what: str = "") -> None:
        import torch

        if self.buf.is_cuda:
            torch.cuda.synchronize(self.buf.device)
        head = torch.equal(self.buf[:GUARD_BYTES], self.head)
        tail = torch.equal(self.buf[GUARD_BYTES + self.nbytes:], self.tail)
        assert head and tail, f"{what}: bytes written outside the tensor (guard before intact: {head}, after: {tail})"


def guarded_like(t, fill="nan"):
    return Guarded(t.shape, t.dtype, device=t.device, fill=fill)


def guarded_workspace(tsp, plan, batch, op):
    """A workspace of tsp_workspace_bytes(plan, batch, op) bytes (at least 16) with guard bands."""
    import torch

    return Guarded((max(16, tsp.tsp_workspace_bytes(plan, batch, op)),), torch.uint8, fill=None)


def guarded_packed(tsp, plan):
    """Packed-weight-shaped gradient buffers with guard bands: (PackedWeights view, [Guarded])."""
    ref = tsp.empty_packed(plan)
    gs = [guarded_like(getattr(ref, n)) for n in ("qkv", "o", "gate_up", "down")]
    del ref
    return tsp.PackedWeights(*(g.t for g in gs)), gs

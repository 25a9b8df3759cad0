"""Bit-exact parity of the layout kernels (zigzag permute, K/V gather, weight packing)."""
import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from oracle import tsp_oracle as O

from helpers import to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


CASES = [  # D, B, S, heads, head_dim, dtype
    (2, 1, 256, 4, 32, "f32"),
    (1, 2, 64, 2, 64, "f32"),
    (4, 2, 1024, 4, 128, "bf16"),
    (8, 1, 2048, 8, 128, "bf16"),
    (3, 2, 96, 3, 64, "bf16"),
    (2, 3, 40, 2, 128, "bf16"),
]


@pytest.mark.parametrize("D,B,S,H,dh,dt", CASES)
def test_zigzag_roundtrip_bit_exact(tsp, D, B, S, H, dh, dt):
    import torch

    h = H * dh
    plan = tsp.tsp_plan_create(D, S, h, H, dh, 128 * D, dt)
    x_np = synth.tensor("x", (B, S, h), 1.0, dt, seed=D * 100 + S)
    x = to_dev(x_np, dt)
    xz = torch.empty_like(x)
    tsp.tsp_zigzag_permute(plan, B, x, xz)
    back = torch.full_like(x, float("nan"))
    tsp.tsp_zigzag_unpermute(plan, B, xz, back)
    torch.cuda.synchronize()
    ref = O.zigzag_permute(x_np, D)  # [D, B, 2C, h]
    assert np.array_equal(to_np(xz).reshape(ref.shape), ref)
    assert torch.equal(back, x)


@pytest.mark.parametrize("D,B,S,H,dh,dt", CASES)
def test_kv_gather_bit_exact(tsp, D, B, S, H, dh, dt):
    import torch

    h = H * dh
    plan = tsp.tsp_plan_create(D, S, h, H, dh, 128 * D, dt)
    kz_np = synth.tensor("Wk", (D, B, S // D, h), 1.0, dt, seed=1)
    vz_np = synth.tensor("Wv", (D, B, S // D, h), 1.0, dt, seed=1)
    kz, vz = to_dev(kz_np, dt), to_dev(vz_np, dt)
    k = torch.empty(B, H, S, dh, dtype=kz.dtype, device="cuda")
    v = torch.empty_like(k)
    tsp.tsp_kv_gather(plan, B, kz, vz, k, v)
    torch.cuda.synchronize()
    for src, out in ((kz_np, k), (vz_np, v)):
        nat = O.zigzag_unpermute(src, D)  # [B, S, h]
        ref = nat.reshape(B, S, H, dh).transpose(0, 2, 1, 3)
        assert np.array_equal(to_np(out), ref)


@pytest.mark.parametrize("D,h,H,F,dt", [(2, 128, 4, 512, "f32"), (4, 512, 4, 768, "bf16"), (8, 1024, 8, 1024, "bf16")])
def test_pack_layout_and_roundtrip(tsp, D, h, H, F, dt):
    import torch

    dh = h // H
    plan = tsp.tsp_plan_create(D, 2 * D, h, H, dh, F, dt)
    shapes = {"Wq": (h, h), "Wk": (h, h), "Wv": (h, h), "Wo": (h, h), "Wg": (h, F), "Wu": (h, F), "Wd": (F, h)}
    canon_np = {k: synth.tensor(k, s, 1.0, dt, seed=7) for k, s in shapes.items()}
    canon = {k: to_dev(v, dt) for k, v in canon_np.items()}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    torch.cuda.synchronize()
    # expected packed layouts, built from the definitions in tsp.h
    hs = h // D
    qkv = np.concatenate([np.concatenate([canon_np[n][:, s * hs:(s + 1) * hs] for n in ("Wq", "Wk", "Wv")], 1)
                          for s in range(D)], 1).T
    gu = np.concatenate([np.concatenate([canon_np["Wg"][:, j * 128:(j + 1) * 128],
                                         canon_np["Wu"][:, j * 128:(j + 1) * 128]], 1) for j in range(F // 128)], 1).T
    assert np.array_equal(to_np(packed.qkv), qkv)
    assert np.array_equal(to_np(packed.o), canon_np["Wo"].T)
    assert np.array_equal(to_np(packed.gate_up), gu)
    assert np.array_equal(to_np(packed.down), canon_np["Wd"].T)
    back = {k: torch.empty_like(v) for k, v in canon.items()}
    tsp.tsp_unpack_weights(plan, packed, back)
    torch.cuda.synchronize()
    for k in canon:
        assert torch.equal(back[k], canon[k]), k


FULL_LAYOUT = [  # D, B, S, K/V heads, head_dim: the 16K-token x 2 and 64K-token workloads, and 8 K/V heads
    (8, 2, 16384, 32, 128),
    (8, 1, 65536, 32, 128),
    (8, 2, 16384, 8, 128),
]


@pytest.mark.parametrize("D,B,S,Hk,dh", FULL_LAYOUT)
def test_layout_full_size_bit_exact(tsp, D, B, S, Hk, dh):
    """Permute, unpermute and K/V gather at the full workload sizes (the launch
    configuration the benchmark times), every element compared with the
    oracle's zigzag position map applied by plain indexing."""
    import torch

    h = 32 * dh
    plan = tsp.tsp_plan_create_gqa(D, S, h, 32, Hk, dh, 128 * D, "bf16")
    gen = torch.Generator(device="cuda").manual_seed(D + S)
    x = torch.randn(B, S, h, generator=gen, device="cuda").to(torch.bfloat16)
    pos = torch.from_numpy(O.zigzag_positions(S, D).astype(np.int64)).to("cuda")  # [D, 2C]
    xz = torch.empty_like(x)
    tsp.tsp_zigzag_permute(plan, B, x, xz)
    back = torch.empty_like(x)
    tsp.tsp_zigzag_unpermute(plan, B, xz, back)
    torch.cuda.synchronize()
    want = x[:, pos.reshape(-1)].reshape(B, D, -1, h).transpose(0, 1)  # [D, B, 2C, h]
    assert torch.equal(xz.view(D, B, -1, h), want)
    assert torch.equal(back, x)
    del want, back
    hk = Hk * dh
    kz = torch.randn(B * S, hk, generator=gen, device="cuda").to(torch.bfloat16)
    vz = torch.randn(B * S, hk, generator=gen, device="cuda").to(torch.bfloat16)
    k = torch.empty(B, Hk, S, dh, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    tsp.tsp_kv_gather(plan, B, kz, vz, k, v)
    torch.cuda.synchronize()
    inv = torch.empty(S, dtype=torch.int64, device="cuda")  # natural position -> (rank, local index)
    inv[pos.reshape(-1)] = torch.arange(S, device="cuda")
    for src, out in ((kz, k), (vz, v)):
        zz = src.view(D, B, -1, hk).transpose(0, 1).reshape(B, S, hk)  # [B][rank-major zigzag][hk]
        nat = zz[:, inv]                                                 # natural order
        assert torch.equal(out, nat.view(B, S, Hk, dh).transpose(1, 2))

"""Grouped-query attention on the GPU against the fp64 oracle (small shapes).

Covers every attention kernel: fp32 (head_dim 32), the warp-MMA bf16 forward
(chunks that are not a multiple of 256), the tcgen05 forward and both tcgen05
backward kernels, with one, two and four query heads per K/V head.
"""
import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import LayerConfig
from oracle import tsp_oracle as O

from helpers import check, rel_frob, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def run(tsp, cfg, inp, backward=False, deterministic=0):
    import torch

    B = cfg.batch
    plan = tsp.plan_for(cfg)
    tsp.tsp_plan_set_deterministic(plan, deterministic)
    canon = {k: to_dev(inp[k], cfg.dtype) for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    x = to_dev(inp["x"], cfg.dtype)
    y = torch.empty_like(x)
    saved = torch.empty(tsp.tsp_saved_bytes(plan, B), dtype=torch.uint8, device="cuda") if backward else None
    tsp.tsp_layer_fwd(plan, B, x, packed, y, saved, tsp.workspace(plan, B, tsp.TSP_OP_LAYER_FWD))
    # attention piece with lse, on zigzag tokens
    xz = torch.empty_like(x)
    tsp.tsp_zigzag_permute(plan, B, x, xz)
    a = torch.empty_like(x)
    lse = torch.empty(B, cfg.heads, cfg.seq, dtype=torch.float32, device="cuda")
    tsp.tsp_attention_fwd(plan, B, xz, packed, a, lse, tsp.workspace(plan, B, tsp.TSP_OP_ATTENTION_FWD))
    out = {"Y": to_np(y), "A": O.zigzag_unpermute(to_np(a).reshape(cfg.D, B, -1, cfg.hidden), cfg.D),
           "lse": to_np(lse)}
    if backward:
        dy = to_dev(inp["dY"], cfg.dtype)
        dx = torch.empty_like(x)
        grads = tsp.empty_packed(plan)
        tsp.tsp_layer_bwd(plan, B, x, packed, saved, dy, dx, grads, tsp.workspace(plan, B, tsp.TSP_OP_LAYER_BWD))
        g = {k: torch.empty_like(v) for k, v in canon.items()}
        tsp.tsp_unpack_weights(plan, grads, g)
        out["dx"] = to_np(dx)
        out.update({"d" + k: to_np(v) for k, v in g.items()})
    tsp.tsp_sync_check()
    return out


FWD = [
    LayerConfig("gqa_f32_D2_s256_h128", D=2, batch=1, seq=256, hidden=128, heads=4, head_dim=32, ffn=512,
                dtype="f32", kv_heads=2),
    # chunk 160: the warp-MMA forward
    LayerConfig("gqa_bf16_D2_s640", D=2, batch=1, seq=640, hidden=512, heads=4, head_dim=128, ffn=512, dtype="bf16",
                kv_heads=2),
    # chunks of 256 / 512: the tcgen05 forward; 2 and 4 query heads per K/V head, and one K/V head
    LayerConfig("gqa_bf16_D2_b2_s1024", D=2, batch=2, seq=1024, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16", kv_heads=2),
    LayerConfig("gqa_bf16_D2_s2048_g4", D=2, batch=1, seq=2048, hidden=1024, heads=8, head_dim=128, ffn=1024,
                dtype="bf16", kv_heads=2),
    LayerConfig("gqa_bf16_D1_s1024_mqa", D=1, batch=1, seq=1024, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16", kv_heads=1),
    # chunks of 128: the tcgen05 forward on mirror pairs of 128-query tiles
    LayerConfig("gqa_bf16_D4_s1024_c128", D=4, batch=1, seq=1024, hidden=1024, heads=8, head_dim=128, ffn=1024,
                dtype="bf16", kv_heads=4),
]


@pytest.mark.parametrize("cfg", FWD, ids=lambda c: c.name)
def test_gqa_forward_matches_oracle(tsp, cfg):
    inp = synth.layer_inputs(cfg, seed=21)
    w = {k: inp[k] for k in tsp.CANONICAL}
    got = run(tsp, cfg, inp)
    ref = O.layer_fwd(inp["x"], w, cfg.heads)
    check(got["Y"], ref["Y"], cfg.dtype, f"{cfg.name} Y")
    check(got["A"], ref["A"], cfg.dtype, f"{cfg.name} A")
    assert np.max(np.abs(got["lse"] - ref["lse"])) < (2e-2 if cfg.dtype == "bf16" else 1e-4)


BWD = [
    LayerConfig("gqa_bwd_D2_b2_s1024", D=2, batch=2, seq=1024, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16", kv_heads=2),
    LayerConfig("gqa_bwd_D4_s2048_g2", D=4, batch=1, seq=2048, hidden=1024, heads=8, head_dim=128, ffn=1024,
                dtype="bf16", kv_heads=4),
    LayerConfig("gqa_bwd_D1_s512_g4", D=1, batch=1, seq=512, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16", kv_heads=1),
]


@pytest.mark.parametrize("det", [0, 1], ids=["fused", "split"])
@pytest.mark.parametrize("cfg", BWD, ids=lambda c: c.name)
def test_gqa_backward_matches_oracle(tsp, cfg, det):
    inp = synth.layer_inputs(cfg, seed=22, with_dy=True)
    w = {k: inp[k] for k in tsp.CANONICAL}
    got = run(tsp, cfg, inp, backward=True, deterministic=det)
    rdx, rg, ry = O.layer_bwd(inp["x"], w, cfg.heads, inp["dY"], return_y=True)
    check(got["Y"], ry, "bf16", f"{cfg.name} Y")
    check(got["dx"], rdx, "bf16", f"{cfg.name} dx")
    for k in tsp.CANONICAL:
        check(got["d" + k], rg[k], "bf16", f"{cfg.name} d{k}")


def test_gqa_agrees_across_D(tsp):
    base = LayerConfig("gqa_xD", D=1, batch=1, seq=2048, hidden=1024, heads=8, head_dim=128, ffn=1024, dtype="bf16",
                       kv_heads=4, backward=True)
    inp = synth.layer_inputs(base, seed=23, with_dy=True)
    outs = {D: run(tsp, base.with_(D=D), inp, backward=True) for D in (1, 2, 4)}
    for D in (2, 4):
        for k in ("Y", "dx", "dWk", "dWv", "dWq"):
            assert rel_frob(outs[D][k], outs[1][k]) <= 2e-2, (D, k)

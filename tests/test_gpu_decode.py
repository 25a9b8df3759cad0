"""Decode step on the GPU against the fp64 oracle.

The key/value cache holds seeded random values (any cache is a valid state);
rows after `pos` hold large sentinel values that would dominate the softmax
if a kernel read them.  Checked: the new token's output, the key and value it
appends at row `pos`, and that every other cache row is left untouched.
"""
import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import LayerConfig
from oracle import tsp_oracle as O

from helpers import Guarded, check, guarded_like, guarded_workspace, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def make_cache(cfg, pos, seed):
    """[B][Hk][S][dh] bf16 on the GPU between guard bands: N(0,1) rows < pos, sentinel 30.0 from pos on."""
    import torch

    gen = torch.Generator(device="cuda").manual_seed(seed)
    shape = (cfg.batch, cfg.kv_h, cfg.seq, cfg.head_dim)
    kg, vg = Guarded(shape, torch.bfloat16, fill=None), Guarded(shape, torch.bfloat16, fill=None)
    kg.t.copy_(torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16))
    vg.t.copy_(torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16))
    kg.t[:, :, pos:] = 30.0
    vg.t[:, :, pos:] = 30.0
    return kg, vg


def as_oracle_cache(c):
    """[B][Hk][S][dh] -> float32 [B][S][Hk*dh] (row = position), exact for bf16 values."""
    B, Hk, S, dh = c.shape
    return c.float().permute(0, 2, 1, 3).reshape(B, S, Hk * dh).cpu().numpy()


def run_decode(tsp, cfg, inp, x_new, pos, seed=5):
    """One decode step; the caches, the output and the workspace sit between guard bands."""
    plan = tsp.plan_for(cfg)
    canon = {k: to_dev(inp[k], "bf16") for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    kg, vg = make_cache(cfg, pos, seed)
    kc, vc = kg.t, vg.t
    k0, v0 = kc.clone(), vc.clone()
    xd = to_dev(x_new, "bf16")
    y = guarded_like(xd)
    ws = guarded_workspace(tsp, plan, cfg.batch, tsp.TSP_OP_DECODE)
    tsp.tsp_decode_step(plan, cfg.batch, pos, xd, packed, kc, vc, y.t, ws.t)
    tsp.tsp_sync_check()
    for g, what in ((kg, "k cache"), (vg, "v cache"), (y, "y_new"), (ws, "decode workspace")):
        g.check(f"{cfg.name} pos={pos} {what}")
    return to_np(y.t), kc, vc, k0, v0


def oracle_step(cfg, inp, x_new, k0, v0, pos):
    w = {k: inp[k] for k in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")}
    return O.decode_step(x_new, w, cfg.heads, as_oracle_cache(k0), as_oracle_cache(v0), pos)


def verify(cfg, got_y, kc, vc, k0, v0, ref, pos, label):
    Y, k_new, v_new = ref
    check(got_y, Y, "bf16", f"{label} y")
    B, Hk, S, dh = kc.shape
    for name, c, c0, r in (("k", kc, k0, k_new), ("v", vc, v0, v_new)):
        row = c[:, :, pos].float().reshape(B, Hk * dh).cpu().numpy()
        check(row, r, "bf16", f"{label} appended {name}")
        mask = np.ones(S, dtype=bool)
        mask[pos] = False
        assert np.array_equal(to_np(c[:, :, mask]), to_np(c0[:, :, mask])), f"{name} cache rows other than pos changed"


SMALL = [
    LayerConfig("dec_D2_s512_mha", D=2, batch=1, seq=512, hidden=512, heads=4, head_dim=128, ffn=512, dtype="bf16"),
    LayerConfig("dec_D2_b3_s512_gqa2", D=2, batch=3, seq=512, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16", kv_heads=2),
    LayerConfig("dec_D4_b2_s1024_g4", D=4, batch=2, seq=1024, hidden=1024, heads=8, head_dim=128, ffn=768,
                dtype="bf16", kv_heads=4),
    LayerConfig("dec_D2_b8_s512_g8", D=2, batch=8, seq=512, hidden=2048, heads=16, head_dim=128, ffn=512,
                dtype="bf16", kv_heads=2),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_decode_step_matches_oracle(tsp, cfg):
    inp = synth.layer_inputs(cfg, seed=41)
    x_all = synth.tensor("x", (cfg.batch, 8, cfg.hidden), 1.0, "bf16", 42)
    C = cfg.chunk
    for i, pos in enumerate(sorted({0, 1, C - 1, C, 2 * C + 5, cfg.seq // 2 + 3, cfg.seq - 1})):
        x_new = x_all[:, i % 8]
        y, kc, vc, k0, v0 = run_decode(tsp, cfg, inp, x_new, pos, seed=100 + i)
        ref = oracle_step(cfg, inp, x_new, k0, v0, pos)
        verify(cfg, y, kc, vc, k0, v0, ref, pos, f"{cfg.name} pos={pos}")


def test_decode_step_rejects_bad_arguments(tsp):
    import torch

    cfg = SMALL[0]
    plan = tsp.plan_for(cfg)
    packed = tsp.empty_packed(plan)
    x = torch.zeros(1, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, cfg.heads, cfg.seq, 128, dtype=torch.bfloat16, device="cuda")
    ws = tsp.workspace(plan, 1, tsp.TSP_OP_DECODE)
    for pos, batch in ((cfg.seq, 1), (-1, 1), (0, 9), (0, 0)):
        with pytest.raises(tsp.TspError) as ei:
            tsp.tsp_decode_step(plan, batch, pos, x, packed, kc, kc.clone(), x.clone(), ws)
        assert ei.value.status == tsp.TSP_ERR_INVALID_ARG
    with pytest.raises(tsp.TspError) as ei:
        tsp.tsp_decode_step(plan, 1, 0, x, packed, kc, kc.clone(), x.clone(), ws[:64])
    assert ei.value.status == tsp.TSP_ERR_WORKSPACE


FULL = [
    LayerConfig("bf16_decode_D8_b1_ctx131072_h4096", D=8, batch=1, seq=131072, hidden=4096, heads=32, head_dim=128,
                ffn=14336, dtype="bf16"),
    LayerConfig("bf16_decode_gqa8_D8_b4_ctx131072_h4096", D=8, batch=4, seq=131072, hidden=4096, heads=32,
                head_dim=128, ffn=14336, dtype="bf16", kv_heads=8),
]


@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_decode_full_context(tsp, cfg):
    """The 7B shape at a 128K-token cache: the last position and one in the middle of a chunk."""
    import torch

    inp = synth.layer_inputs(cfg, seed=43, only=tsp.CANONICAL)
    x_all = synth.tensor("x", (cfg.batch, 2, cfg.hidden), 1.0, "bf16", 44)
    for i, pos in enumerate((cfg.seq - 1, 5 * cfg.chunk + 1000)):
        y, kc, vc, k0, v0 = run_decode(tsp, cfg, inp, x_all[:, i], pos, seed=200 + i)
        ref = oracle_step(cfg, inp, x_all[:, i], k0, v0, pos)
        Y, k_new, v_new = ref
        check(y, Y, "bf16", f"{cfg.name} pos={pos} y")
        B, Hk, S, dh = kc.shape
        check(kc[:, :, pos].float().reshape(B, -1).cpu().numpy(), k_new, "bf16", "appended k")
        check(vc[:, :, pos].float().reshape(B, -1).cpu().numpy(), v_new, "bf16", "appended v")
        del kc, vc, k0, v0
        torch.cuda.empty_cache()


def test_decode_agrees_across_D(tsp):
    """The rank split of the cache only partitions the keys: D = 1, 2, 4 give the same step."""
    base = LayerConfig("dec_xD", D=1, batch=2, seq=1024, hidden=1024, heads=8, head_dim=128, ffn=512, dtype="bf16",
                       kv_heads=4)
    inp = synth.layer_inputs(base, seed=45)
    x_new = synth.tensor("x", (base.batch, base.hidden), 1.0, "bf16", 46)
    outs = {}
    for D in (1, 2, 4):
        y, kc, vc, _, _ = run_decode(tsp, base.with_(D=D), inp, x_new, 700, seed=300)
        outs[D] = (y, to_np(kc[:, :, 700]), to_np(vc[:, :, 700]))
    for D in (2, 4):
        assert np.array_equal(outs[D][1], outs[1][1]) and np.array_equal(outs[D][2], outs[1][2])  # same K/V row
        err = np.linalg.norm(outs[D][0] - outs[1][0]) / np.linalg.norm(outs[1][0])
        assert err <= 2e-2, (D, err)

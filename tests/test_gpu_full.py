"""Parity at the full workload sizes.

* 16K and 64K tokens (forward): the oracle evaluates sampled query rows
  exactly (K and V for every token, attention/W_O/MLP for the sampled rows):
  the first and last token of every zigzag chunk (so every rank and both of
  its chunks) plus seeded random rows.  Y and A on those rows must be within
  the bf16 relative-Frobenius bound.
* The same 16K-token layer recomputed with D = 1, 2, 4 must agree with D = 8
  over the whole output.
* 8K tokens forward + backward: the full fp64 oracle gradient (dx and all
  seven weight gradients) against the GPU.
* The same checks with grouped-query attention (8 K/V heads for 32 query
  heads) at 16K tokens (sampled rows) and 8K tokens (full backward).

Inputs are drawn by the seeded generator (torch integer recipe on the host)
once and handed to both sides.
"""
import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import (LAYER_7B_GQA8_S16K, LAYER_7B_S16K, LAYER_7B_S64K, TRAIN_7B_GQA8_S8K,
                                                  TRAIN_7B_S8K, TRAIN_7B_S16K)
from oracle import tsp_oracle as O

from helpers import check, rel_frob, to_np

pytestmark = pytest.mark.gpu

SHAPES = lambda h, F, hk: {"Wq": (h, h), "Wk": (h, hk), "Wv": (h, hk), "Wo": (h, h), "Wg": (h, F), "Wu": (h, F),
                           "Wd": (F, h)}


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def draw(cfg, with_dy=False):
    """bf16 host tensors of one workload (same values go to the GPU and, as fp64, to the oracle)."""
    h, F = cfg.hidden, cfg.ffn
    t = {k: synth.tensor_torch(k, s, (F if k == "Wd" else h) ** -0.5, "bf16", 0, "cpu")
         for k, s in SHAPES(h, F, cfg.kv_hidden).items()}
    t["x"] = synth.tensor_torch("x", (cfg.batch, cfg.seq, h), 1.0, "bf16", 0, "cpu")
    if with_dy:
        t["dY"] = synth.tensor_torch("dY", (cfg.batch, cfg.seq, h), 1.0, "bf16", 0, "cpu")
    return t


def sample_rows(cfg, n_random=224, seed=1):
    C = cfg.chunk
    rows = set()
    for c in range(2 * cfg.D):
        rows.add(c * C)
        rows.add(c * C + C - 1)
    rng = np.random.default_rng(seed)
    rows.update(rng.choice(cfg.seq, size=n_random, replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def gpu_forward(tsp, cfg, t, D=None):
    import torch

    D = D or cfg.D
    plan = tsp.plan_for(cfg.with_(D=D))
    canon = {k: t[k].cuda() for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    del canon
    x = t["x"].cuda()
    y = torch.empty_like(x)
    tsp.tsp_layer_fwd(plan, cfg.batch, x, packed, y, None, tsp.workspace(plan, cfg.batch, tsp.TSP_OP_LAYER_FWD))
    xz = torch.empty_like(x)
    tsp.tsp_zigzag_permute(plan, cfg.batch, x, xz)
    a = torch.empty_like(x)
    tsp.tsp_attention_fwd(plan, cfg.batch, xz, packed, a, None, tsp.workspace(plan, cfg.batch,
                                                                              tsp.TSP_OP_ATTENTION_FWD))
    az = torch.empty_like(x)
    tsp.tsp_zigzag_unpermute(plan, cfg.batch, a, az)
    tsp.tsp_sync_check()
    return y, az


@pytest.mark.parametrize("cfg", [LAYER_7B_S16K, LAYER_7B_S64K, LAYER_7B_GQA8_S16K], ids=lambda c: c.name)
def test_full_size_sampled_rows(tsp, cfg):
    t = draw(cfg)
    y, a = gpu_forward(tsp, cfg, t)
    rows = sample_rows(cfg)
    w = {k: t[k].double().numpy() for k in tsp.CANONICAL}
    x64 = t["x"].double().numpy()
    ref = O.layer_fwd(x64, w, cfg.heads, rows=rows)
    yr = y[:, torch_index(rows)].float().cpu().numpy()
    ar = a[:, torch_index(rows)].float().cpu().numpy()
    check(yr, ref["Y"], "bf16", f"{cfg.name} Y (sampled rows)")
    check(ar, ref["A"], "bf16", f"{cfg.name} A (sampled rows)")


def torch_index(rows):
    import torch

    return torch.from_numpy(rows).cuda()


def test_full_size_cross_D(tsp):
    cfg = LAYER_7B_S16K
    t = draw(cfg)
    y8, _ = gpu_forward(tsp, cfg, t)
    ref = to_np(y8)
    for D in (1, 2, 4):
        yD, _ = gpu_forward(tsp, cfg, t, D=D)
        assert rel_frob(to_np(yD), ref) <= 2e-2, D


@pytest.mark.parametrize("cfg", [TRAIN_7B_S8K, TRAIN_7B_GQA8_S8K], ids=lambda c: c.name)
def test_training_workload_backward(tsp, cfg):
    import torch

    t = draw(cfg, with_dy=True)
    B = cfg.batch
    plan = tsp.plan_for(cfg)
    canon = {k: t[k].cuda() for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    x, dy = t["x"].cuda(), t["dY"].cuda()
    y = torch.empty_like(x)
    saved = torch.empty(tsp.tsp_saved_bytes(plan, B), dtype=torch.uint8, device="cuda")
    tsp.tsp_layer_fwd(plan, B, x, packed, y, saved, tsp.workspace(plan, B, tsp.TSP_OP_LAYER_FWD))
    dx = torch.empty_like(x)
    grads = tsp.empty_packed(plan)
    tsp.tsp_layer_bwd(plan, B, x, packed, saved, dy, dx, grads, tsp.workspace(plan, B, tsp.TSP_OP_LAYER_BWD))
    g = {k: torch.empty_like(v) for k, v in canon.items()}
    tsp.tsp_unpack_weights(plan, grads, g)
    tsp.tsp_sync_check()
    w = {k: t[k].double().numpy() for k in tsp.CANONICAL}
    rdx, rg, ry = O.layer_bwd(t["x"].double().numpy(), w, cfg.heads, t["dY"].double().numpy(), return_y=True)
    check(to_np(y), ry, "bf16", f"{cfg.name} Y")
    check(to_np(dx), rdx, "bf16", f"{cfg.name} dx")
    for k in tsp.CANONICAL:
        check(to_np(g[k]), rg[k], "bf16", f"{cfg.name} d{k}")


def gpu_backward(tsp, cfg, t, D, deterministic=0):
    import torch

    B = cfg.batch
    plan = tsp.plan_for(cfg.with_(D=D))
    tsp.tsp_plan_set_deterministic(plan, deterministic)
    canon = {k: t[k].cuda() for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    x, dy = t["x"].cuda(), t["dY"].cuda()
    y = torch.empty_like(x)
    saved = torch.empty(tsp.tsp_saved_bytes(plan, B), dtype=torch.uint8, device="cuda")
    tsp.tsp_layer_fwd(plan, B, x, packed, y, saved, tsp.workspace(plan, B, tsp.TSP_OP_LAYER_FWD))
    dx = torch.empty_like(x)
    grads = tsp.empty_packed(plan)
    tsp.tsp_layer_bwd(plan, B, x, packed, saved, dy, dx, grads, tsp.workspace(plan, B, tsp.TSP_OP_LAYER_BWD))
    g = {k: torch.empty_like(v) for k, v in canon.items()}
    tsp.tsp_unpack_weights(plan, grads, g)
    tsp.tsp_sync_check()
    out = {"dx": to_np(dx)}
    out.update({k: to_np(v) for k, v in g.items()})
    del saved, packed, canon
    torch.cuda.empty_cache()
    return out


def test_backward_16k_tokens_agrees_across_D(tsp):
    """Backward at batch 2 x 16384 tokens: D = 2 and 4 against D = 8 on dx and every weight gradient.

    No fp64 reference at this size (its gradient would take hours); the
    D = 8 run itself is pinned at 8K tokens by test_training_workload_backward.
    """
    cfg = TRAIN_7B_S16K
    t = draw(cfg, with_dy=True)
    ref = gpu_backward(tsp, cfg, t, 8)
    for D in (2, 4):
        got = gpu_backward(tsp, cfg, t, D)
        for k in ref:
            e = rel_frob(got[k], ref[k])
            print(f"PARITY cross-D {D} vs 8 {k}: relative Frobenius {e:.3e}")
            assert e <= 2e-2, (D, k, e)


@pytest.mark.parametrize("cfg", [TRAIN_7B_S8K, TRAIN_7B_GQA8_S8K], ids=lambda c: c.name)
def test_training_workload_fused_vs_split(tsp, cfg):
    """The fused backward (dQ summed by fp32 reductions) against the split,
    bitwise-reproducible one at the full 8K-token training shape; both are
    pinned to the fp64 gradient by the tests above and on small shapes."""
    t = draw(cfg, with_dy=True)
    fused = gpu_backward(tsp, cfg, t, cfg.D, deterministic=0)
    split = gpu_backward(tsp, cfg, t, cfg.D, deterministic=1)
    for k in split:
        e = rel_frob(fused[k], split[k])
        print(f"PARITY {cfg.name} fused vs split {k}: relative Frobenius {e:.3e}")
        assert e <= 5e-3, (k, e)

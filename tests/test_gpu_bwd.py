"""Backward parity (dx and every weight gradient) against the fp64 oracle's exact gradient."""
import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import LayerConfig
from oracle import tsp_oracle as O

from helpers import Guarded, check, guarded_like, guarded_packed, guarded_workspace, rel_frob, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def run_bwd(tsp, cfg, inp, deterministic=0):
    """Forward (keeping activations) and backward; every output, the saved buffer and both
    workspaces sit between guard bands that must be intact afterwards."""
    import torch

    B = cfg.batch
    plan = tsp.tsp_plan_create(cfg.D, cfg.seq, cfg.hidden, cfg.heads, cfg.head_dim, cfg.ffn, cfg.dtype)
    tsp.tsp_plan_set_deterministic(plan, deterministic)
    canon = {k: to_dev(inp[k], cfg.dtype) for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    x = to_dev(inp["x"], cfg.dtype)
    dy = to_dev(inp["dY"], cfg.dtype)
    y = guarded_like(x)
    saved = Guarded((tsp.tsp_saved_bytes(plan, B),), torch.uint8, fill=None)
    wf = guarded_workspace(tsp, plan, B, tsp.TSP_OP_LAYER_FWD)
    tsp.tsp_layer_fwd(plan, B, x, packed, y.t, saved.t, wf.t)
    dx = guarded_like(x)
    grads, gguards = guarded_packed(tsp, plan)
    wb = guarded_workspace(tsp, plan, B, tsp.TSP_OP_LAYER_BWD)
    tsp.tsp_layer_bwd(plan, B, x, packed, saved.t, dy, dx.t, grads, wb.t)
    canon_g = {k: torch.empty_like(v) for k, v in canon.items()}
    tsp.tsp_unpack_weights(plan, grads, canon_g)
    tsp.tsp_sync_check()
    for g, what in ((y, "y"), (saved, "saved"), (wf, "forward workspace"), (dx, "dx"), (wb, "backward workspace"),
                    *zip(gguards, ("dW_qkv", "dW_o", "dW_gate_up", "dW_down"))):
        g.check(f"{cfg.name} {what}")
    return to_np(y.t), to_np(dx.t), {k: to_np(v) for k, v in canon_g.items()}


BWD_CASES = [
    LayerConfig("bwd_D2_s256", D=2, batch=1, seq=256, hidden=256, heads=2, head_dim=128, ffn=512, dtype="bf16"),
    # ragged: chunks of 80 queries, T = 320 tokens leaves a 64-row tail in every token-major GEMM
    LayerConfig("bwd_D2_s320", D=2, batch=1, seq=320, hidden=256, heads=2, head_dim=128, ffn=512, dtype="bf16"),
    LayerConfig("bwd_D4_b2_s1024", D=4, batch=2, seq=1024, hidden=512, heads=4, head_dim=128, ffn=768, dtype="bf16"),
    LayerConfig("bwd_D8_s2048", D=8, batch=1, seq=2048, hidden=1024, heads=8, head_dim=128, ffn=1024, dtype="bf16"),
    LayerConfig("bwd_D3_s1152", D=3, batch=1, seq=1152, hidden=768, heads=6, head_dim=128, ffn=1536, dtype="bf16"),
    # forward through the tcgen05 attention kernel (V saved transposed)
    LayerConfig("bwd_D2_b2_s1024", D=2, batch=2, seq=1024, hidden=256, heads=2, head_dim=128, ffn=512, dtype="bf16"),
    LayerConfig("bwd_D4_s2048", D=4, batch=1, seq=2048, hidden=512, heads=4, head_dim=128, ffn=768, dtype="bf16"),
]


def tc_case(cfg):
    """Chunks that are multiples of 128 take the tensor-core backward (fused or split)."""
    return (cfg.seq // (2 * cfg.D)) % 128 == 0


# (case, deterministic): the tensor-core cases run both backward algorithms
MODE_CASES = [(c, m) for c in BWD_CASES for m in ((0, 1) if tc_case(c) else (0,))]


@pytest.mark.parametrize("cfg,det", MODE_CASES, ids=lambda v: v.name if hasattr(v, "name") else f"det{v}")
def test_backward_matches_oracle(tsp, cfg, det):
    inp = synth.layer_inputs(cfg, seed=5, with_dy=True)
    w = {k: inp[k] for k in tsp.CANONICAL}
    y, dx, g = run_bwd(tsp, cfg, inp, deterministic=det)
    ref_y = O.layer_fwd(inp["x"], w, cfg.heads)["Y"]
    check(y, ref_y, "bf16", f"{cfg.name} Y")
    rdx, rg = O.layer_bwd(inp["x"], w, cfg.heads, inp["dY"])
    check(dx, rdx, "bf16", f"{cfg.name} dx")
    for k in tsp.CANONICAL:
        check(g[k], rg[k], "bf16", f"{cfg.name} d{k}")


DET_CFG = LayerConfig("det_D8_s4096", D=8, batch=1, seq=4096, hidden=1024, heads=8, head_dim=128, ffn=1024,
                      dtype="bf16")


def test_forward_and_backward_are_bitwise_deterministic(tsp):
    """With the split backward no kernel uses atomics, so repeated runs must
    agree bit for bit; a barrier or ordering race would show up here as
    run-to-run differences."""
    inp = synth.layer_inputs(DET_CFG, seed=9, with_dy=True)
    runs = [run_bwd(tsp, DET_CFG, inp, deterministic=1) for _ in range(3)]
    for y, dx, g in runs[1:]:
        assert np.array_equal(y, runs[0][0])
        assert np.array_equal(dx, runs[0][1])
        for k in g:
            assert np.array_equal(g[k], runs[0][2][k]), k


def test_fused_backward_repeats(tsp):
    """The fused backward sums dQ with fp32 reductions in varying order: what
    does not depend on dQ (Y, dK, dV and so dWk, dWv, and the MLP and output
    projection gradients) must still repeat bit for bit, dx and dWq only up
    to rounding; and the two algorithms must agree."""
    inp = synth.layer_inputs(DET_CFG, seed=9, with_dy=True)
    runs = [run_bwd(tsp, DET_CFG, inp, deterministic=0) for _ in range(3)]
    exact = ["Wk", "Wv", "Wo", "Wg", "Wu", "Wd"]
    for y, dx, g in runs[1:]:
        assert np.array_equal(y, runs[0][0])
        for k in exact:
            assert np.array_equal(g[k], runs[0][2][k]), k
        assert rel_frob(dx, runs[0][1]) <= 1e-3
        assert rel_frob(g["Wq"], runs[0][2]["Wq"]) <= 1e-3
    y1, dx1, g1 = run_bwd(tsp, DET_CFG, inp, deterministic=1)
    assert rel_frob(dx1, runs[0][1]) <= 5e-3
    for k in g1:
        e = rel_frob(g1[k], runs[0][2][k])
        print(f"PARITY fused vs split d{k}: relative Frobenius {e:.3e}")
        assert e <= 5e-3, (k, e)

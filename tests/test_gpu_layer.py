"""Layer-level parity of the CUDA path against the fp64 oracle (small and mid sizes).

Tolerances: fp32 plans, normwise max relative error <= 1e-4; bf16 plans,
relative Frobenius error <= 2e-2 per output tensor.  Outputs are checked both
with and without the residual (A, MLP, Y) so the residual cannot hide errors.
"""
import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import MID_BF16, TINY_F32, LayerConfig
from oracle import tsp_oracle as O

from helpers import Guarded, check, guarded_like, guarded_workspace, rel_frob, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def setup(tsp, cfg, inp=None, seed=0):
    import torch

    inp = inp if inp is not None else synth.layer_inputs(cfg, seed=seed)
    plan = tsp.tsp_plan_create(cfg.D, cfg.seq, cfg.hidden, cfg.heads, cfg.head_dim, cfg.ffn, cfg.dtype)
    canon = {k: to_dev(inp[k], cfg.dtype) for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    x = to_dev(inp["x"], cfg.dtype)
    return plan, packed, x, inp


def run_pieces(tsp, cfg, plan, packed, x):
    """Runs attention_fwd, gated_mlp_fwd and layer_fwd; returns natural-order A, MLP(H_ref-free), Y, lse.

    Every output and workspace sits between guard bands that must be intact afterwards."""
    import torch

    B = cfg.batch
    xz = guarded_like(x)
    tsp.tsp_zigzag_permute(plan, B, x, xz.t)
    a = guarded_like(x)
    lse = Guarded((B, cfg.heads, cfg.seq), torch.float32)
    wa = guarded_workspace(tsp, plan, B, tsp.TSP_OP_ATTENTION_FWD)
    tsp.tsp_attention_fwd(plan, B, xz.t, packed, a.t, lse.t, wa.t)
    y = guarded_like(x)
    wl = guarded_workspace(tsp, plan, B, tsp.TSP_OP_LAYER_FWD)
    tsp.tsp_layer_fwd(plan, B, x, packed, y.t, None, wl.t)
    tsp.tsp_sync_check()
    for g, what in ((xz, "xz"), (a, "a_out"), (lse, "lse"), (y, "y"), (wa, "attention workspace"),
                    (wl, "layer workspace")):
        g.check(f"{cfg.name} {what}")
    a_nat = O.zigzag_unpermute(to_np(a.t).reshape(cfg.D, B, -1, cfg.hidden), cfg.D)
    return a_nat, to_np(y.t), to_np(lse.t)


def mlp_piece(tsp, cfg, plan, packed, H_np):
    """gated_mlp_fwd on the given natural-order H (values exact in the plan dtype)."""
    B = cfg.batch
    Hd = to_dev(H_np, cfg.dtype)
    hz = guarded_like(Hd)
    tsp.tsp_zigzag_permute(plan, B, Hd, hz.t)
    m = guarded_like(Hd)
    wm = guarded_workspace(tsp, plan, B, tsp.TSP_OP_GATED_MLP_FWD)
    tsp.tsp_gated_mlp_fwd(plan, B, hz.t, packed, m.t, wm.t)
    tsp.tsp_sync_check()
    for g, what in ((hz, "hz"), (m, "m_out"), (wm, "mlp workspace")):
        g.check(f"{cfg.name} {what}")
    return O.zigzag_unpermute(to_np(m.t).reshape(cfg.D, B, -1, cfg.hidden), cfg.D)


def round_to(a, dtype):
    return synth.round_bf16(a) if dtype == "bf16" else a.astype(np.float32).astype(np.float64)


def full_check(tsp, cfg, seed=0):
    plan, packed, x, inp = setup(tsp, cfg, seed=seed)
    w = {k: inp[k] for k in tsp.CANONICAL}
    ref = O.layer_fwd(inp["x"], w, cfg.heads)
    a, y, lse = run_pieces(tsp, cfg, plan, packed, x)
    errs = {"A": check(a, ref["A"], cfg.dtype, f"{cfg.name} A"), "Y": check(y, ref["Y"], cfg.dtype, f"{cfg.name} Y")}
    # lse is fp32 in both paths; bf16 inputs to QK^T are exact, so it must be close
    assert np.max(np.abs(lse - ref["lse"])) < (2e-2 if cfg.dtype == "bf16" else 1e-4)
    Hr = round_to(ref["H"], cfg.dtype)
    mref = O.gated_mlp(Hr, w)
    errs["MLP"] = check(mlp_piece(tsp, cfg, plan, packed, Hr), mref, cfg.dtype, f"{cfg.name} MLP")
    return errs, y



def test_tiny_f32_matches_oracle(tsp):
    full_check(tsp, TINY_F32)


@pytest.mark.parametrize("D", [1, 4])
def test_tiny_f32_other_D(tsp, D):
    full_check(tsp, TINY_F32.with_(D=D, name=f"tiny_f32_D{D}"))


SMALL_BF16 = [
    # ragged query tiles (C = 80) and a ragged 64-row GEMM tail (T = 320)
    LayerConfig("bf16_D2_s320", D=2, batch=1, seq=320, hidden=256, heads=2, head_dim=128, ffn=512, dtype="bf16"),
    # several tiles in every GEMM dimension, two batches
    LayerConfig("bf16_D4_b2_s1024", D=4, batch=2, seq=1024, hidden=512, heads=4, head_dim=128, ffn=768, dtype="bf16"),
    # D = 8 with one head per shard; chunks of 128 queries: the tcgen05 attention on mirror pairs of 128-query tiles
    LayerConfig("bf16_D8_s2048", D=8, batch=1, seq=2048, hidden=1024, heads=8, head_dim=128, ffn=1024, dtype="bf16"),
    # chunks of 384 queries (three 128-query tiles): tcgen05 attention, tile mirror pairs, two sequences
    LayerConfig("bf16_D2_b2_s1536", D=2, batch=2, seq=1536, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16"),
    # odd D, chunk not a multiple of the 128-row query tile
    LayerConfig("bf16_D3_s1152", D=3, batch=1, seq=1152, hidden=768, heads=6, head_dim=128, ffn=1536, dtype="bf16"),
    # chunks of 256 and 512 queries: the tcgen05 attention kernel (256-query blocks)
    LayerConfig("bf16_D2_b2_s1024", D=2, batch=2, seq=1024, hidden=256, heads=2, head_dim=128, ffn=512, dtype="bf16"),
    LayerConfig("bf16_D4_s2048", D=4, batch=1, seq=2048, hidden=512, heads=4, head_dim=128, ffn=768, dtype="bf16"),
    LayerConfig("bf16_D1_s1536", D=1, batch=1, seq=1536, hidden=256, heads=2, head_dim=128, ffn=256, dtype="bf16"),
]


@pytest.mark.parametrize("cfg", SMALL_BF16, ids=lambda c: c.name)
def test_small_bf16_matches_oracle(tsp, cfg):
    full_check(tsp, cfg)


def test_mid_bf16_matches_oracle(tsp):
    full_check(tsp, MID_BF16)


def test_outputs_agree_across_D(tsp):
    base = LayerConfig("xD", D=1, batch=1, seq=2048, hidden=1024, heads=8, head_dim=128, ffn=1024, dtype="bf16")
    inp = synth.layer_inputs(base, seed=3)
    ys = {}
    for D in (1, 2, 4, 8):
        cfg = base.with_(D=D)
        plan, packed, x, _ = setup(tsp, cfg, inp=inp)
        _, y, _ = run_pieces(tsp, cfg, plan, packed, x)
        ys[D] = y
    for D in (2, 4, 8):
        assert rel_frob(ys[D], ys[1]) <= 2e-2


def test_attention_rescale_path_matches_oracle(tsp):
    """Scores that grow along the sequence, so that a row's maximum rises above its first key
    tile's by more than 2^8 (8 in log2 units): the tcgen05 softmax then leaves its common path
    (the two half-row warps vote on their pair barrier, read the row's maximum, rescale O in
    tensor memory and recompute P).  Built from the seeded inputs: x becomes x / 2 + c(p) u with u a
    fixed unit vector and c rising from -8 to 8 along the sequence, and W_K = W_Q, so every score
    gains c(i) c(j) |u W_Q|^2 / sqrt(dh): late keys win the late rows, early keys lose them (and
    the scores stay below 8, where the bf16 comparison is as tight as in the other tests)."""
    import torch

    cfg = LayerConfig("bf16_rescale_D2_s1024", D=2, batch=1, seq=1024, hidden=256, heads=2, head_dim=128,
                      ffn=512, dtype="bf16")
    inp = dict(synth.layer_inputs(cfg, seed=5))
    S, h, dh = cfg.seq, cfg.hidden, cfg.head_dim
    u = np.ones(h) / np.sqrt(h)
    c = 8.0 * (2.0 * np.arange(S) / (S - 1) - 1.0)
    inp["x"] = synth.round_bf16(0.5 * inp["x"] + c[None, :, None] * u[None, None, :])
    inp["Wk"] = inp["Wq"].copy()
    # the precondition, from fp64 scores: many rows' running max grows by > 8 (log2) after key tile 0
    x0 = inp["x"][0]
    Qm, Km = x0 @ inp["Wq"], x0 @ inp["Wk"]
    causal = np.tril(np.ones((S, S), dtype=bool))
    smax = 0.0
    for hd in range(cfg.heads):
        sl = slice(hd * dh, (hd + 1) * dh)
        s = (Qm[:, sl] @ Km[:, sl].T) / np.sqrt(dh)
        smax = max(smax, float(np.max(np.abs(s[causal]))))
        s2 = np.where(causal, s * np.log2(np.e), -np.inf)
        first, later = s2[:, :128].max(axis=1), s2[:, 128:].max(axis=1)
        assert int(np.sum(later > first + 8)) >= 64, "too few rows take the rescale path"
    plan, packed, x, _ = setup(tsp, cfg, inp=inp)
    w = {k: inp[k] for k in tsp.CANONICAL}
    ref = O.layer_fwd(inp["x"], w, cfg.heads)
    B = cfg.batch
    xz = guarded_like(x)
    tsp.tsp_zigzag_permute(plan, B, x, xz.t)
    a = guarded_like(x)
    lse = Guarded((B, cfg.heads, cfg.seq), torch.float32)
    wa = guarded_workspace(tsp, plan, B, tsp.TSP_OP_ATTENTION_FWD)
    tsp.tsp_attention_fwd(plan, B, xz.t, packed, a.t, lse.t, wa.t)
    tsp.tsp_sync_check()
    for g, what in ((a, "a_out"), (lse, "lse"), (wa, "attention workspace")):
        g.check(f"{cfg.name} {what}")
    a_nat = O.zigzag_unpermute(to_np(a.t).reshape(cfg.D, B, -1, cfg.hidden), cfg.D)
    check(a_nat, ref["A"], "bf16", f"{cfg.name} A")
    # Q and K are rounded to bf16 on the GPU (2^-8 relative each), so a score of size |s| moves by
    # up to about 2^-7 |s|, and the log-sum-exp by at most the largest such move
    assert smax < 8.0
    err = float(np.max(np.abs(to_np(lse.t) - ref["lse"])))
    print(f"PARITY {cfg.name} lse: max abs {err:.3e} (largest |score| {smax:.2f})")
    assert err <= 2 ** -7 * smax + 1e-2

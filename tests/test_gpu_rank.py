"""The per-rank TSP path on the GPU (tsp_rank_* through the C ABI).

* tsp_rank_extract_shard writes, bit for bit, the shard layouts include/tsp.h
  documents (built here from the oracle's shard definitions).
* The whole schedule (folded_tensor_sequence_gb300.tsp_rank.layer_fwd) run as
  D virtual ranks on one GPU -- one host thread and CUDA stream per rank, the
  broadcasts, the K/V all-gather and the MLP ring as stream-ordered copies --
  gives every rank's output rows; stitched together they must match the
  oracle (fp32: max relative 1e-4; bf16: relative Frobenius 2e-2) and the
  single-GPU tsp_layer_fwd (which sums the same shards in another order).
* At the 16K-token x 2, D = 8 workload (32 and 8 K/V heads) the stitched
  output is compared with tsp_layer_fwd over every element.  One rank's
  attention there runs with the key split (two CTAs per mirror pair and a
  log-sum-exp combine), as it does in every small tcgen05 case here.
* One rank's three calls write nothing outside their outputs and workspaces
  (guard bands) and produce finite values.
"""
import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import LAYER_7B_GQA8_S16K, LAYER_7B_S16K, LayerConfig
from oracle import tsp_oracle as O

from helpers import check, guarded_like, guarded_workspace, rel_frob, to_dev, to_np
from rank_oracle import pack_attention_shard, pack_mlp_shard

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


CASES = [
    # fp32 (SIMT GEMMs, fp32 attention)
    LayerConfig("rank_f32_D2_s256", D=2, batch=1, seq=256, hidden=128, heads=4, head_dim=32, ffn=512, dtype="f32"),
    # bf16, chunks of 256: tcgen05 attention of one rank's mirror block pairs
    LayerConfig("rank_bf16_D2_s1024", D=2, batch=1, seq=1024, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16"),
    # two sequences, D = 4, grouped-query attention (2 query heads per K/V head)
    LayerConfig("rank_bf16_D4_b2_s2048_gqa", D=4, batch=2, seq=2048, hidden=1024, heads=8, head_dim=128, ffn=1024,
                dtype="bf16", kv_heads=4),
    # chunks of 160 queries: the warp-MMA attention kernel with a ragged tile
    LayerConfig("rank_bf16_D2_s640", D=2, batch=1, seq=640, hidden=512, heads=4, head_dim=128, ffn=512,
                dtype="bf16"),
]


def _packed(tsp, plan, inp, dtype):
    canon = {k: to_dev(inp[k], dtype) for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    return packed


@pytest.mark.parametrize("cfg", CASES[:3], ids=lambda c: c.name)
def test_extract_shard_layout_bit_exact(tsp, cfg):
    import torch

    inp = synth.layer_inputs(cfg, seed=21, only=tsp.CANONICAL)
    plan = tsp.plan_for(cfg)
    packed = _packed(tsp, plan, inp, cfg.dtype)
    w = {k: inp[k] for k in tsp.CANONICAL}
    dt = plan.torch_dtype
    for kind, pack in ((tsp.TSP_SHARD_ATTENTION, pack_attention_shard), (tsp.TSP_SHARD_MLP, pack_mlp_shard)):
        nbytes = tsp.tsp_rank_shard_bytes(plan, kind)
        for s in range(cfg.D):
            want = pack(w, s, cfg.D)
            assert nbytes == want.size * (2 if cfg.dtype == "bf16" else 4)
            g = guarded_like(torch.empty(nbytes, dtype=torch.uint8, device="cuda"), fill=None)
            tsp.tsp_rank_extract_shard(plan, packed, s, kind, g.t)
            torch.cuda.synchronize()
            g.check(f"shard {s} kind {kind}")
            got = to_np(g.t.view(dt))
            assert np.array_equal(got, want), f"shard {s} kind {kind}"


def run_ranks(tsp, cfg, inp):
    """The schedule for every rank as D threads on this GPU; returns natural-order Y [B, S, h]."""
    import torch

    from folded_tensor_sequence_gb300 import tsp_rank

    plan = tsp.plan_for(cfg)
    packed = _packed(tsp, plan, inp, cfg.dtype)
    x = to_dev(inp["x"], cfg.dtype)
    xz = torch.empty_like(x)
    tsp.tsp_zigzag_permute(plan, cfg.batch, x, xz)
    torch.cuda.synchronize()
    D, L, h = cfg.D, cfg.batch * 2 * cfg.chunk, cfg.hidden
    xz_r = xz.view(D, L, h)

    def body(rank, comm):
        layer = tsp_rank.RankLayer(plan, rank, cfg.batch, stream=comm.stream)
        with torch.cuda.stream(comm.stream):
            attn_own, mlp_own = layer.own_shards(packed)
            y = tsp_rank.layer_fwd(comm, layer, xz_r[rank], attn_own, mlp_own)
            out = y.clone()
        return out

    ys = tsp_rank.run_local_ranks(D, body)
    torch.cuda.synchronize()
    yz = torch.stack(ys).view(x.shape)  # rank-major zigzag rows
    y = torch.empty_like(x)
    tsp.tsp_zigzag_unpermute(plan, cfg.batch, yz, y)
    torch.cuda.synchronize()
    return y, plan, packed, x


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_rank_schedule_matches_layer(tsp, cfg):
    import torch

    inp = synth.layer_inputs(cfg, seed=23)
    y, plan, packed, x = run_ranks(tsp, cfg, inp)
    w = {k: inp[k] for k in tsp.CANONICAL}
    ref = O.layer_fwd(inp["x"], w, cfg.heads)
    check(to_np(y), ref["Y"], cfg.dtype, f"{cfg.name} per-rank Y vs oracle")
    y1 = guarded_like(x)
    ws = guarded_workspace(tsp, plan, cfg.batch, tsp.TSP_OP_LAYER_FWD)
    tsp.tsp_layer_fwd(plan, cfg.batch, x, packed, y1.t, None, ws.t)
    tsp.tsp_sync_check()
    y1.check("tsp_layer_fwd y")
    e = rel_frob(to_np(y), to_np(y1.t))
    print(f"PARITY {cfg.name} per-rank vs tsp_layer_fwd: relative Frobenius {e:.3e}")
    assert e <= (1e-5 if cfg.dtype == "f32" else 2e-2)


def test_rank_entry_outputs_stay_in_bounds(tsp):
    """One rank's three calls with every output and workspace between guard bands."""
    import torch

    cfg = CASES[1]
    inp = synth.layer_inputs(cfg, seed=25)
    plan = tsp.plan_for(cfg)
    packed = _packed(tsp, plan, inp, cfg.dtype)
    D, L, h = cfg.D, cfg.batch * 2 * cfg.chunk, cfg.hidden
    hs, ks = h // D, cfg.kv_hidden // D
    x = torch.randn(L, h, device="cuda").to(torch.bfloat16)
    shard = torch.empty(tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_ATTENTION), dtype=torch.uint8, device="cuda")
    mshard = torch.empty(tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_MLP), dtype=torch.uint8, device="cuda")
    tsp.tsp_rank_extract_shard(plan, packed, 1, tsp.TSP_SHARD_ATTENTION, shard)
    tsp.tsp_rank_extract_shard(plan, packed, 1, tsp.TSP_SHARD_MLP, mshard)
    q = guarded_like(torch.empty(L, hs, dtype=torch.bfloat16, device="cuda"))
    kv = guarded_like(torch.empty(L, 2 * ks, dtype=torch.bfloat16, device="cuda"))
    tsp.tsp_rank_qkv(plan, cfg.batch, x, shard, q.t, kv.t)
    kv_all = kv.t.repeat(D, 1).view(D, L, 2 * ks)  # every rank's K/V: stand-in values, shapes are what matter
    hout = guarded_like(x)
    wa = guarded_workspace(tsp, plan, cfg.batch, tsp.TSP_OP_RANK_ATTENTION)
    tsp.tsp_rank_attention(plan, 1, cfg.batch, q.t, kv_all, shard, x, hout.t, wa.t)
    yout = guarded_like(x)
    wm = guarded_workspace(tsp, plan, cfg.batch, tsp.TSP_OP_RANK_MLP)
    tsp.tsp_rank_mlp(plan, cfg.batch, hout.t, mshard, hout.t, yout.t, wm.t)
    tsp.tsp_sync_check()
    for g, what in ((q, "q"), (kv, "kv"), (hout, "h_out"), (wa, "attention workspace"), (yout, "y_out"),
                    (wm, "mlp workspace")):
        g.check(what)
    for g in (q, kv, hout, yout):
        assert torch.isfinite(g.t.float()).all()


@pytest.mark.parametrize("cfg", [LAYER_7B_S16K, LAYER_7B_GQA8_S16K], ids=lambda c: c.name)
def test_rank_schedule_full_size_matches_layer(tsp, cfg):
    """D = 8 ranks, 2 x 16384 tokens, hidden 4096 (32 K/V heads, and 8): the stitched per-rank output
    against tsp_layer_fwd over every element (the layer itself is pinned to the oracle on sampled rows
    at this size)."""
    import torch

    h, F, hk = cfg.hidden, cfg.ffn, cfg.kv_hidden
    shapes = {"Wq": (h, h), "Wk": (h, hk), "Wv": (h, hk), "Wo": (h, h), "Wg": (h, F), "Wu": (h, F), "Wd": (F, h)}
    inp = {k: synth.tensor_torch(k, s, (F if k == "Wd" else h) ** -0.5, "bf16", 0, "cpu").double().numpy()
           for k, s in shapes.items()}
    inp["x"] = synth.tensor_torch("x", (cfg.batch, cfg.seq, h), 1.0, "bf16", 0, "cpu").double().numpy()
    y, plan, packed, x = run_ranks(tsp, cfg, inp)
    y1 = torch.empty_like(x)
    tsp.tsp_layer_fwd(plan, cfg.batch, x, packed, y1, None, tsp.workspace(plan, cfg.batch, tsp.TSP_OP_LAYER_FWD))
    tsp.tsp_sync_check()
    assert torch.isfinite(y.float()).all()
    e = float((y.float() - y1.float()).norm() / y1.float().norm())
    print(f"PARITY full-size per-rank vs tsp_layer_fwd: relative Frobenius {e:.3e}")
    assert e <= 2e-2


def test_rank_calls_without_residual(tsp):
    """resid NULL means 0: the attention and MLP steps store their product, equal to adding it to zeros."""
    import torch

    cfg = CASES[2]  # grouped-query attention, two sequences, tcgen05 attention with the key split
    inp = synth.layer_inputs(cfg, seed=27)
    plan = tsp.plan_for(cfg)
    packed = _packed(tsp, plan, inp, cfg.dtype)
    D, L, h = cfg.D, cfg.batch * 2 * cfg.chunk, cfg.hidden
    hs, ks = h // D, cfg.kv_hidden // D
    gen = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(L, h, generator=gen, device="cuda").to(torch.bfloat16)
    kv_all = torch.randn(D, L, 2 * ks, generator=gen, device="cuda").to(torch.bfloat16)
    shard = torch.empty(tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_ATTENTION), dtype=torch.uint8, device="cuda")
    mshard = torch.empty(tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_MLP), dtype=torch.uint8, device="cuda")
    tsp.tsp_rank_extract_shard(plan, packed, 2, tsp.TSP_SHARD_ATTENTION, shard)
    tsp.tsp_rank_extract_shard(plan, packed, 3, tsp.TSP_SHARD_MLP, mshard)
    q = torch.empty(L, hs, dtype=torch.bfloat16, device="cuda")
    kv = torch.empty(L, 2 * ks, dtype=torch.bfloat16, device="cuda")
    tsp.tsp_rank_qkv(plan, cfg.batch, x, shard, q, kv)
    wa = tsp.workspace(plan, cfg.batch, tsp.TSP_OP_RANK_ATTENTION)
    wm = tsp.workspace(plan, cfg.batch, tsp.TSP_OP_RANK_MLP)
    zeros = torch.zeros_like(x)
    for r in (0, D - 1):
        a0, a1 = torch.empty_like(x), torch.empty_like(x)
        tsp.tsp_rank_attention(plan, r, cfg.batch, q, kv_all, shard, None, a0, wa)
        tsp.tsp_rank_attention(plan, r, cfg.batch, q, kv_all, shard, zeros, a1, wa)
        m0, m1 = torch.empty_like(x), torch.empty_like(x)
        tsp.tsp_rank_mlp(plan, cfg.batch, x, mshard, None, m0, wm)
        tsp.tsp_rank_mlp(plan, cfg.batch, x, mshard, zeros, m1, wm)
        tsp.tsp_sync_check()
        assert torch.isfinite(a0.float()).all() and float(a0.float().abs().max()) > 0
        assert torch.equal(a0, a1), f"rank {r}: attention output with resid NULL differs from resid 0"
        assert torch.equal(m0, m1), f"rank {r}: MLP output with resid NULL differs from resid 0"

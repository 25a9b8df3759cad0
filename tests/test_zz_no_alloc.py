"""tsp_attention_fwd_static: the attention entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc at all -- a plug-in whose host application
owns every device allocation, or a latency-critical loop where an allocation
could synchronize the device -- so they cannot pass a workspace.  This entry
point takes its scratch from the library's static device array instead.  The
test calls it through the C ABI twice in a row (different inputs, so stale
contents of the shared array would show) and checks each result against
tsp_attention_fwd with a caller-allocated workspace.  Both run the same
deterministic kernels on the same inputs, so the outputs and the log-sum-exp
must be bit-identical.  Two shapes: chunks of 80 queries (the warp-MMA
attention kernel) and chunks of 256 (the tcgen05 attention kernel, which also
keeps V transposed in the scratch).  It also checks that a batch too large for
the static array is refused before anything runs.

The file name makes pytest collect it last.
"""
import ctypes

import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import LayerConfig

from helpers import to_dev

pytestmark = pytest.mark.gpu

CFGS = [
    # chunk 80: the warp-MMA attention kernel
    LayerConfig("static_D2_s320", D=2, batch=1, seq=320, hidden=256, heads=2, head_dim=128, ffn=512, dtype="bf16"),
    # chunk 256: the tcgen05 attention kernel (V^T in the scratch); 2 MiB of scratch
    LayerConfig("static_D2_s1024", D=2, batch=1, seq=1024, hidden=256, heads=2, head_dim=128, ffn=512,
                dtype="bf16"),
]


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: c.name)
def test_static_scratch_matches_workspace_path(tsp, cfg):
    import torch

    plan = tsp.tsp_plan_create(cfg.D, cfg.seq, cfg.hidden, cfg.heads, cfg.head_dim, cfg.ffn, "bf16")
    assert tsp.tsp_workspace_bytes(plan, cfg.batch, tsp.TSP_OP_ATTENTION_FWD) <= tsp.TSP_STATIC_SCRATCH_BYTES
    inp = synth.layer_inputs(cfg, seed=11)
    canon = {k: to_dev(inp[k], "bf16") for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    ws = tsp.workspace(plan, cfg.batch, tsp.TSP_OP_ATTENTION_FWD)
    L = tsp.lib()
    w = packed.c()
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((11, 12)):
        x = to_dev(synth.tensor("x", (cfg.batch, cfg.seq, cfg.hidden), 1.0, "bf16", seed=seed), "bf16")
        xz = torch.empty_like(x)
        tsp.tsp_zigzag_permute(plan, cfg.batch, x, xz)
        ref = torch.empty_like(x)
        ref_lse = torch.empty(cfg.batch, cfg.heads, cfg.seq, dtype=torch.float32, device="cuda")
        tsp.tsp_attention_fwd(plan, cfg.batch, xz, packed, ref, ref_lse, ws)
        got = torch.full_like(x, float("nan"))
        got_lse = torch.full_like(ref_lse, float("nan"))
        st = L.tsp_attention_fwd_static(plan.handle, cfg.batch, xz.data_ptr(), ctypes.byref(w), got.data_ptr(),
                                        got_lse.data_ptr(), stream)
        assert st == tsp.TSP_OK, tsp.tsp_last_error_message()
        tsp.tsp_sync_check()
        assert torch.equal(got, ref), f"call {call}: output differs from the workspace path"
        assert torch.equal(got_lse, ref_lse), f"call {call}: log-sum-exp differs from the workspace path"
        # and both are the layer's attention (the oracle check lives in the layer tests; this guards
        # against both paths being wrong the same way, e.g. an all-zero result)
        assert float(got.float().abs().max()) > 0


def test_static_scratch_rejects_oversized_batch(tsp):
    # hidden 4096 x 16384 tokens needs 512 MiB of scratch, far above the static array
    plan = tsp.tsp_plan_create(8, 16384, 4096, 32, 128, 14336, "bf16")
    L = tsp.lib()
    w = tsp._Weights(0x1000, 0x2000, 0x3000, 0x4000)
    st = L.tsp_attention_fwd_static(plan.handle, 1, 0x1000, ctypes.byref(w), 0x2000, None, None)
    assert st == tsp.TSP_ERR_WORKSPACE
    assert "static" in tsp.tsp_last_error_message()

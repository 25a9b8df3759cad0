"""tsp_attention_fwd_static: the attention entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc at all -- a plug-in whose host application
owns every device allocation, or a latency-critical loop where an allocation
could synchronize the device -- so they cannot pass a workspace.  This entry
point takes its scratch from the library's static device array instead.  The
test calls it through the C ABI twice in a row (different inputs, so stale
contents of the shared array would show) and checks each result against
tsp_attention_fwd with a caller-allocated workspace, within the bf16 tolerance
used by the other parity tests.  It also checks that a batch too large for the
static array is refused before anything runs.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

from folded_tensor_sequence_gb300 import synth
from folded_tensor_sequence_gb300.configs import LayerConfig

from helpers import BF16_TOL, rel_frob, to_dev, to_np

pytestmark = pytest.mark.gpu

CFG = LayerConfig("static_D2_s320", D=2, batch=1, seq=320, hidden=256, heads=2, head_dim=128, ffn=512,
                  dtype="bf16")


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def test_static_scratch_matches_workspace_path(tsp):
    import torch

    plan = tsp.tsp_plan_create(CFG.D, CFG.seq, CFG.hidden, CFG.heads, CFG.head_dim, CFG.ffn, "bf16")
    inp = synth.layer_inputs(CFG, seed=11)
    canon = {k: to_dev(inp[k], "bf16") for k in tsp.CANONICAL}
    packed = tsp.empty_packed(plan)
    tsp.tsp_pack_weights(plan, canon, packed)
    ws = tsp.workspace(plan, CFG.batch, tsp.TSP_OP_ATTENTION_FWD)
    L = tsp.lib()
    w = packed.c()
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((11, 12)):
        x = to_dev(synth.tensor("x", (CFG.batch, CFG.seq, CFG.hidden), 1.0, "bf16", seed=seed), "bf16")
        xz = torch.empty_like(x)
        tsp.tsp_zigzag_permute(plan, CFG.batch, x, xz)
        ref = torch.empty_like(x)
        ref_lse = torch.empty(CFG.batch, CFG.heads, CFG.seq, dtype=torch.float32, device="cuda")
        tsp.tsp_attention_fwd(plan, CFG.batch, xz, packed, ref, ref_lse, ws)
        got = torch.full_like(x, float("nan"))
        got_lse = torch.full_like(ref_lse, float("nan"))
        st = L.tsp_attention_fwd_static(plan.handle, CFG.batch, xz.data_ptr(), ctypes.byref(w), got.data_ptr(),
                                        got_lse.data_ptr(), stream)
        assert st == tsp.TSP_OK, tsp.tsp_last_error_message()
        tsp.tsp_sync_check()
        e = rel_frob(to_np(got), to_np(ref))
        assert e <= BF16_TOL, f"call {call}: relative Frobenius error {e:.3e}"
        assert np.max(np.abs(to_np(got_lse) - to_np(ref_lse))) <= 2e-2


def test_static_scratch_rejects_oversized_batch(tsp):
    # hidden 4096 x 16384 tokens needs 512 MiB of scratch, far above the static array
    plan = tsp.tsp_plan_create(8, 16384, 4096, 32, 128, 14336, "bf16")
    L = tsp.lib()
    w = tsp._Weights(0x1000, 0x2000, 0x3000, 0x4000)
    st = L.tsp_attention_fwd_static(plan.handle, 1, 0x1000, ctypes.byref(w), 0x2000, None, None)
    assert st == tsp.TSP_ERR_WORKSPACE
    assert "static" in tsp.tsp_last_error_message()

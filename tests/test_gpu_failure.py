"""Failure detection on the GPU without a fault: a bounded device wait gives up and is reported."""
import pytest

from folded_tensor_sequence_gb300.configs import LayerConfig

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def test_bounded_wait_reports_timeout_and_context_survives(tsp):
    import torch

    tsp.tsp_sync_check()  # clean start
    tsp.tsp_debug_wait_timeout(200000)  # 0.2 s on a barrier nothing signals
    with pytest.raises(tsp.TspError) as ei:
        tsp.tsp_sync_check()
    assert ei.value.status == tsp.TSP_ERR_TIMEOUT
    assert "kernel 4" in tsp.tsp_last_error_message()
    tsp.tsp_sync_check()  # the error word was cleared
    # the context still runs real work afterwards
    cfg = LayerConfig("after_timeout", D=2, batch=1, seq=256, hidden=256, heads=2, head_dim=128, ffn=512,
                      dtype="bf16")
    plan = tsp.tsp_plan_create(cfg.D, cfg.seq, cfg.hidden, cfg.heads, cfg.head_dim, cfg.ffn, "bf16")
    x = torch.randn(1, cfg.seq, cfg.hidden, device="cuda").to(torch.bfloat16)
    xz = torch.empty_like(x)
    back = torch.empty_like(x)
    tsp.tsp_zigzag_permute(plan, 1, x, xz)
    tsp.tsp_zigzag_unpermute(plan, 1, xz, back)
    tsp.tsp_sync_check()
    assert torch.equal(back, x)


def test_injected_host_failure_enqueues_nothing(tsp):
    import torch

    plan = tsp.tsp_plan_create(2, 256, 256, 2, 128, 512, "bf16")
    x = torch.randn(1, 256, 256, device="cuda").to(torch.bfloat16)
    xz = torch.zeros_like(x)
    tsp.tsp_debug_fail_next(tsp.TSP_ERR_CUDA, 1)
    with pytest.raises(tsp.TspError):
        tsp.tsp_zigzag_permute(plan, 1, x, xz)
    tsp.tsp_sync_check()
    assert torch.count_nonzero(xz) == 0  # the failed call wrote nothing

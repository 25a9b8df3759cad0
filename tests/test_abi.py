"""The C ABI library loads, exports every declared symbol, and validates on the host (no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tsp():
    import __graft_entry__ as g

    g.build()
    from folded_tensor_sequence_gb300 import tsp as T

    return T


def declared_symbols():
    with open(os.path.join(ROOT, "include", "tsp.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsp_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(tsp):
    names = declared_symbols()
    assert len(names) >= 17
    L = tsp.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(tsp.EXPORTS) == names


def test_plan_validation(tsp):
    p = tsp.tsp_plan_create(2, 256, 128, 4, 32, 512, "f32")
    assert p.handle
    bad = [
        (0, 256, 128, 4, 32, 512),      # D < 1
        (2, 250, 128, 4, 32, 512),      # seq % 2D
        (2, 256, 130, 4, 32, 512),      # hidden != heads*head_dim
        (3, 258, 128, 4, 32, 384),      # heads % D
        (2, 256, 96, 3, 32, 512),       # heads % D (3 % 2)
        (2, 256, 128, 4, 32, 500),      # ffn % 128
        (2, 256, 192, 4, 48, 512),      # head_dim not in {32,64,128}
    ]
    for args in bad:
        with pytest.raises(tsp.TspError) as ei:
            tsp.tsp_plan_create(*args, "f32")
        assert ei.value.status == tsp.TSP_ERR_INVALID_ARG
        assert tsp.tsp_last_error_message()


def test_workspace_sizes_are_consistent(tsp):
    p = tsp.tsp_plan_create(8, 16384, 4096, 32, 128, 14336, "bf16")
    T, h, F = 2 * 16384, 4096, 14336
    assert tsp.tsp_workspace_bytes(p, 2, tsp.TSP_OP_ATTENTION_FWD) >= 4 * T * h * 2
    assert tsp.tsp_workspace_bytes(p, 2, tsp.TSP_OP_GATED_MLP_FWD) >= 3 * T * F * 2
    saved = tsp.tsp_saved_bytes(p, 2)
    assert saved >= (6 * T * h + 3 * T * F) * 2 + 2 * 32 * 16384 * 4
    assert tsp.tsp_workspace_bytes(p, 2, tsp.TSP_OP_LAYER_FWD) >= saved + T * h * 2
    assert tsp.tsp_workspace_bytes(p, 2, tsp.TSP_OP_LAYER_BWD) > 0
    assert tsp.tsp_workspace_bytes(p, 0, tsp.TSP_OP_LAYER_FWD) == 0 or True
    assert tsp.lib().tsp_workspace_bytes(None, 2, 0) == 0


def test_status_strings(tsp):
    for s in range(6):
        assert tsp.tsp_status_string(s).startswith("TSP_")


def test_invalid_args_rejected_before_launch(tsp):
    p = tsp.tsp_plan_create(2, 256, 256, 2, 128, 512, "bf16")
    with pytest.raises(tsp.TspError) as ei:
        tsp.tsp_zigzag_permute(p, 1, None, None)
    assert ei.value.status == tsp.TSP_ERR_INVALID_ARG
    with pytest.raises(tsp.TspError) as ei:
        tsp.tsp_zigzag_permute(p, 1, 0x1003, 0x2000)  # misaligned
    assert ei.value.status == tsp.TSP_ERR_INVALID_ARG
    with pytest.raises(tsp.TspError) as ei:
        tsp.tsp_zigzag_permute(p, -1, 0x1000, 0x2000)
    assert ei.value.status == tsp.TSP_ERR_INVALID_ARG
    # workspace too small is reported before anything is enqueued
    L = tsp.lib()
    w = tsp._Weights(0x1000, 0x2000, 0x3000, 0x4000)
    st = L.tsp_layer_fwd(p.handle, 1, 0x1000, ctypes.byref(w), 0x2000, None, 0x5000, 16, None)
    assert st == tsp.TSP_ERR_WORKSPACE
    # bf16 shapes without a kernel are reported as unsupported
    p2 = tsp.tsp_plan_create(1, 256, 128, 1, 128, 512, "bf16")
    st = L.tsp_layer_fwd(p2.handle, 1, 0x1000, ctypes.byref(w), 0x2000, None, 0x5000, 1 << 40, None)
    assert st == tsp.TSP_ERR_UNSUPPORTED
    # the fp32 backward is not provided
    p3 = tsp.tsp_plan_create(2, 256, 128, 4, 32, 512, "f32")
    st = L.tsp_layer_bwd(p3.handle, 1, 0x1000, ctypes.byref(w), 0x2000, 0x3000, 0x4000, ctypes.byref(w), 0x5000,
                         1 << 40, None)
    assert st == tsp.TSP_ERR_UNSUPPORTED


def test_host_fault_injection(tsp):
    p = tsp.tsp_plan_create(2, 256, 256, 2, 128, 512, "bf16")
    tsp.tsp_debug_fail_next(tsp.TSP_ERR_CUDA, 2)
    for _ in range(2):
        with pytest.raises(tsp.TspError) as ei:
            tsp.tsp_zigzag_permute(p, 1, 0x1000, 0x2000)
        assert ei.value.status == tsp.TSP_ERR_CUDA
        assert "injected" in tsp.tsp_last_error_message()
    tsp.tsp_debug_fail_next(tsp.TSP_OK, 0)
    # disarmed: the next call is validated normally (NULL -> invalid arg)
    with pytest.raises(tsp.TspError) as ei:
        tsp.tsp_zigzag_permute(p, 1, None, None)
    assert ei.value.status == tsp.TSP_ERR_INVALID_ARG


def test_wait_probe_validates_on_host(tsp):
    L = tsp.lib()
    assert L.tsp_debug_wait_timeout(0, None) == tsp.TSP_ERR_INVALID_ARG
    assert L.tsp_debug_wait_timeout(20000000, None) == tsp.TSP_ERR_INVALID_ARG


def test_gqa_plan_validation_and_sizes(tsp):
    p = tsp.tsp_plan_create_gqa(8, 16384, 4096, 32, 8, 128, 14336, "bf16")
    assert p.kv_heads == 8 and p.kv_hidden == 1024
    mha = tsp.tsp_plan_create(8, 16384, 4096, 32, 128, 14336, "bf16")
    # K and V (and their gradients) shrink with the K/V head count
    assert tsp.tsp_saved_bytes(p, 2) < tsp.tsp_saved_bytes(mha, 2)
    assert tsp.tsp_workspace_bytes(p, 2, tsp.TSP_OP_LAYER_BWD) < tsp.tsp_workspace_bytes(mha, 2, tsp.TSP_OP_LAYER_BWD)
    # kv_heads == heads is the multi-head plan
    same = tsp.tsp_plan_create_gqa(8, 16384, 4096, 32, 32, 128, 14336, "bf16")
    assert tsp.tsp_saved_bytes(same, 2) == tsp.tsp_saved_bytes(mha, 2)
    bad = [
        (2, 1024, 512, 4, 3, 128, 512),   # kv_heads does not divide heads
        (4, 1024, 1024, 8, 2, 128, 512),  # kv_heads % D (a shard must own whole K/V heads)
        (2, 1024, 512, 4, 0, 128, 512),   # kv_heads < 1
    ]
    for args in bad:
        with pytest.raises(tsp.TspError) as ei:
            tsp.tsp_plan_create_gqa(*args, "bf16")
        assert ei.value.status == tsp.TSP_ERR_INVALID_ARG


def test_gqa_backward_needs_128_query_chunks(tsp):
    L = tsp.lib()
    w = tsp._Weights(0x1000, 0x2000, 0x3000, 0x4000)
    p = tsp.tsp_plan_create_gqa(2, 640, 512, 4, 2, 128, 512, "bf16")  # chunk 160
    st = L.tsp_layer_bwd(p.handle, 1, 0x1000, ctypes.byref(w), 0x2000, 0x3000, 0x4000, ctypes.byref(w), 0x5000,
                         1 << 40, None)
    assert st == tsp.TSP_ERR_UNSUPPORTED
    assert "grouped-query" in tsp.tsp_last_error_message()


def test_deterministic_setting(tsp):
    p = tsp.tsp_plan_create(8, 16384, 4096, 32, 128, 14336, "bf16")
    assert tsp.tsp_plan_get_deterministic(p) == 0  # fused backward by default
    tsp.tsp_plan_set_deterministic(p, 1)
    assert tsp.tsp_plan_get_deterministic(p) == 1
    for bad in (-1, 2, 7):
        with pytest.raises(tsp.TspError) as ei:
            tsp.tsp_plan_set_deterministic(p, bad)
        assert ei.value.status == tsp.TSP_ERR_INVALID_ARG
    assert tsp.tsp_plan_get_deterministic(p) == 1
    L = tsp.lib()
    assert L.tsp_plan_set_deterministic(None, 1) == tsp.TSP_ERR_INVALID_ARG
    assert L.tsp_plan_get_deterministic(None) == -1
    # the backward workspace holds the fp32 dQ accumulator (T x h x 4 bytes) either way
    T, h = 2 * 16384, 4096
    assert tsp.tsp_workspace_bytes(p, 2, tsp.TSP_OP_LAYER_BWD) >= T * h * 4


def test_empty_batch_is_a_no_op(tsp):
    """batch 0 (no tokens) is valid for every entry point that takes a batch of
    sequences: it returns TSP_OK without reading a pointer or touching the
    device (this runs without a GPU, with every pointer NULL).  Decode batches
    are 1..8 sequences and reject 0."""
    L = tsp.lib()
    for dt in ("bf16", "f32"):
        p = tsp.tsp_plan_create(2, 256, 256, 2, 128, 512, dt)
        h = p.handle
        assert L.tsp_zigzag_permute(h, 0, None, None, None) == tsp.TSP_OK
        assert L.tsp_zigzag_unpermute(h, 0, None, None, None) == tsp.TSP_OK
        assert L.tsp_kv_gather(h, 0, None, None, None, None, None) == tsp.TSP_OK
        assert L.tsp_attention_fwd(h, 0, None, None, None, None, None, 0, None) == tsp.TSP_OK
        assert L.tsp_attention_fwd_static(h, 0, None, None, None, None, None) == tsp.TSP_OK
        assert L.tsp_gated_mlp_fwd(h, 0, None, None, None, None, 0, None) == tsp.TSP_OK
        assert L.tsp_layer_fwd(h, 0, None, None, None, None, None, 0, None) == tsp.TSP_OK
        assert L.tsp_layer_bwd(h, 0, None, None, None, None, None, None, None, 0, None) == tsp.TSP_OK
        assert tsp.tsp_saved_bytes(p, 0) == 0
        for op in (tsp.TSP_OP_ATTENTION_FWD, tsp.TSP_OP_GATED_MLP_FWD, tsp.TSP_OP_LAYER_FWD, tsp.TSP_OP_LAYER_BWD):
            assert tsp.tsp_workspace_bytes(p, 0, op) == 0
        # a negative batch is still an error, on the static entry point too
        assert L.tsp_attention_fwd_static(h, -1, None, None, None, None, None) == tsp.TSP_ERR_INVALID_ARG
    p = tsp.tsp_plan_create(2, 256, 256, 2, 128, 512, "bf16")
    assert L.tsp_decode_step(p.handle, 0, 0, None, None, None, None, None, None, 0, None) == tsp.TSP_ERR_INVALID_ARG


def test_rank_shard_sizes_and_validation(tsp):
    """Shard sizes follow the documented layouts; bad ranks, shards, shapes and workspaces are refused
    on the host before anything is enqueued."""
    D, S, h, H, dh, F = 8, 16384, 4096, 32, 128, 14336
    p = tsp.tsp_plan_create(D, S, h, H, dh, F, "bf16")
    hs, fs = h // D, F // D
    assert tsp.tsp_rank_shard_bytes(p, tsp.TSP_SHARD_ATTENTION) == ((hs + 2 * hs) * h + h * hs) * 2
    assert tsp.tsp_rank_shard_bytes(p, tsp.TSP_SHARD_MLP) == (2 * fs * h + h * fs) * 2
    assert tsp.lib().tsp_rank_shard_bytes(None, 0) == 0
    g = tsp.tsp_plan_create_gqa(D, S, h, H, 8, dh, F, "bf16")
    assert tsp.tsp_rank_shard_bytes(g, tsp.TSP_SHARD_ATTENTION) == ((hs + 2 * 128) * h + h * hs) * 2
    # workspaces: K and V^T (V for the warp-MMA kernel) of the shard's heads over the whole sequence, and
    # the rank's attention output
    B = 2
    L = B * S // D
    assert tsp.tsp_workspace_bytes(p, B, tsp.TSP_OP_RANK_ATTENTION) >= (2 * B * S * hs + L * hs) * 2
    assert tsp.tsp_workspace_bytes(p, B, tsp.TSP_OP_RANK_MLP) >= L * fs * 2
    w = tsp._Weights(0x1000, 0x2000, 0x3000, 0x4000)
    L_ = tsp.lib()
    big = 1 << 40
    ws_ok = tsp.tsp_workspace_bytes(p, B, tsp.TSP_OP_RANK_ATTENTION)
    cases = [
        (L_.tsp_rank_attention(p.handle, D, B, 0x1000, 0x2000, 0x3000, None, 0x4000, 0x5000, big, None),
         tsp.TSP_ERR_INVALID_ARG),  # rank == D
        (L_.tsp_rank_attention(p.handle, -1, B, 0x1000, 0x2000, 0x3000, None, 0x4000, 0x5000, big, None),
         tsp.TSP_ERR_INVALID_ARG),
        (L_.tsp_rank_attention(p.handle, 0, B, 0x1000, 0x2000, 0x3000, None, 0x4000, 0x5000, ws_ok - 1, None),
         tsp.TSP_ERR_WORKSPACE),
        (L_.tsp_rank_attention(p.handle, 0, B, 0x1000, 0x2000, 0x3000, 0x3008, 0x4000, 0x5000, big, None),
         tsp.TSP_ERR_INVALID_ARG),  # misaligned resid
        (L_.tsp_rank_qkv(p.handle, B, 0x1000, None, 0x2000, 0x3000, None), tsp.TSP_ERR_INVALID_ARG),
        (L_.tsp_rank_mlp(p.handle, B, 0x1000, 0x2000, None, 0x3000, 0x4000, 0, None), tsp.TSP_ERR_WORKSPACE),
        (L_.tsp_rank_extract_shard(p.handle, ctypes.byref(w), D, 0, 0x5000, None), tsp.TSP_ERR_INVALID_ARG),
        (L_.tsp_rank_extract_shard(p.handle, ctypes.byref(w), 0, 7, 0x5000, None), tsp.TSP_ERR_INVALID_ARG),
    ]
    for got, want in cases:
        assert got == want, (got, want, tsp.tsp_last_error_message())
    # a shard must hold whole 128-column gate/up blocks: ffn / D = 1152 / 8 = 144
    odd = tsp.tsp_plan_create(8, 2048, 2048, 16, 128, 1152, "bf16")
    st = L_.tsp_rank_mlp(odd.handle, 1, 0x1000, 0x2000, None, 0x3000, 0x4000, big, None)
    assert st == tsp.TSP_ERR_UNSUPPORTED and "128" in tsp.tsp_last_error_message()
    # bf16 needs hidden / D % 256 == 0 (2048 / 16 = 128)
    narrow = tsp.tsp_plan_create(16, 4096, 2048, 16, 128, 4096, "bf16")
    st = L_.tsp_rank_qkv(narrow.handle, 1, 0x1000, 0x2000, 0x3000, 0x4000, None)
    assert st == tsp.TSP_ERR_UNSUPPORTED
    # an empty batch is a no-op that reads no pointer
    assert L_.tsp_rank_qkv(p.handle, 0, None, None, None, None, None) == tsp.TSP_OK
    assert L_.tsp_rank_attention(p.handle, 0, 0, None, None, None, None, None, None, 0, None) == tsp.TSP_OK
    assert L_.tsp_rank_mlp(p.handle, 0, None, None, None, None, None, 0, None) == tsp.TSP_OK

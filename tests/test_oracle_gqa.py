"""Pins of the oracle's grouped-query attention (no GPU).

Independent checks: (1) GQA equals multi-head attention whose K/V weights
repeat every K/V head's columns once per query head that reads it (an exact
identity, so fp64 agreement to rounding); (2) the GQA gradients are that
expanded model's gradients with the repeated copies summed; (3) central
finite differences; (4) the TSP-sharded schedule equals the plain layer.
"""
import numpy as np
import pytest

from oracle import tsp_oracle as O


def _weights(rng, h, hk, F):
    return {
        "Wq": rng.standard_normal((h, h)) / np.sqrt(h),
        "Wk": rng.standard_normal((h, hk)) / np.sqrt(h),
        "Wv": rng.standard_normal((h, hk)) / np.sqrt(h),
        "Wo": rng.standard_normal((h, h)) / np.sqrt(h),
        "Wg": rng.standard_normal((h, F)) / np.sqrt(h),
        "Wu": rng.standard_normal((h, F)) / np.sqrt(h),
        "Wd": rng.standard_normal((F, h)) / np.sqrt(F),
    }


def _expand(w, heads, kv_heads, dh):
    """Multi-head weights equal to the GQA ones: K/V head g copied into query heads g*grp .. (g+1)*grp-1."""
    grp = heads // kv_heads
    cols = np.concatenate([np.arange(e // grp * dh, (e // grp + 1) * dh) for e in range(heads)])
    we = dict(w)
    we["Wk"] = w["Wk"][:, cols]
    we["Wv"] = w["Wv"][:, cols]
    return we, cols


@pytest.mark.parametrize("heads,kv_heads", [(4, 2), (4, 1), (6, 3), (4, 4)])
def test_gqa_equals_expanded_multi_head(heads, kv_heads):
    rng = np.random.default_rng(11)
    dh, B, S, F = 4, 2, 12, 24
    h = heads * dh
    w = _weights(rng, h, kv_heads * dh, F)
    x = rng.standard_normal((B, S, h))
    we, _ = _expand(w, heads, kv_heads, dh)
    g, m = O.layer_fwd(x, w, heads), O.layer_fwd(x, we, heads)
    for k in ("A", "Y", "lse", "O"):
        np.testing.assert_allclose(g[k], m[k], rtol=1e-12, atol=1e-12)


def test_gqa_gradients_are_summed_expanded_gradients():
    rng = np.random.default_rng(12)
    heads, kv_heads, dh, B, S, F = 6, 2, 4, 1, 10, 16
    h = heads * dh
    w = _weights(rng, h, kv_heads * dh, F)
    x = rng.standard_normal((B, S, h))
    dY = rng.standard_normal((B, S, h))
    we, cols = _expand(w, heads, kv_heads, dh)
    dx, g = O.layer_bwd(x, w, heads, dY)
    dxe, ge = O.layer_bwd(x, we, heads, dY)
    np.testing.assert_allclose(dx, dxe, rtol=1e-11, atol=1e-11)
    for k in ("Wq", "Wo", "Wg", "Wu", "Wd"):
        np.testing.assert_allclose(g[k], ge[k], rtol=1e-11, atol=1e-11)
    for k in ("Wk", "Wv"):
        summed = np.zeros_like(w[k])
        np.add.at(summed.T, cols, ge[k].T)  # fold the copies back onto their K/V head's columns
        np.testing.assert_allclose(g[k], summed, rtol=1e-11, atol=1e-11)


def test_gqa_backward_matches_finite_differences():
    rng = np.random.default_rng(13)
    heads, kv_heads, dh, B, S, F = 4, 2, 2, 1, 6, 8
    h = heads * dh
    w = _weights(rng, h, kv_heads * dh, F)
    x = rng.standard_normal((B, S, h))
    dY = rng.standard_normal((B, S, h))
    dx, g = O.layer_bwd(x, w, heads, dY)

    def loss():
        return float(np.sum(O.layer_fwd(x, w, heads)["Y"] * dY))

    eps = 1e-6
    for name, arr, ref in (("x", x, dx), ("Wk", w["Wk"], g["Wk"]), ("Wv", w["Wv"], g["Wv"]), ("Wq", w["Wq"], g["Wq"])):
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            old = arr[i]
            arr[i] = old + eps
            lp = loss()
            arr[i] = old - eps
            lm = loss()
            arr[i] = old
            fd[i] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(fd - ref) / np.linalg.norm(ref)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("D", [1, 2, 4])
def test_gqa_sharded_schedule_equals_plain_layer(D):
    rng = np.random.default_rng(14)
    heads, kv_heads, dh, B, S, F = 8, 4, 4, 2, 16, 32
    h = heads * dh
    w = _weights(rng, h, kv_heads * dh, F)
    x = rng.standard_normal((B, S, h))
    ref = O.layer_fwd(x, w, heads)
    got = O.tsp_layer_fwd_sharded(x, w, heads, D)
    for k in ("A", "Y"):
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-12, atol=1e-12)


def test_gqa_shard_needs_kv_heads_divisible_by_D():
    rng = np.random.default_rng(15)
    heads, kv_heads, dh = 8, 2, 4
    w = _weights(rng, heads * dh, kv_heads * dh, 16)
    with pytest.raises(ValueError):
        O.tsp_layer_fwd_sharded(rng.standard_normal((1, 16, heads * dh)), w, heads, 4)


def test_gqa_cuts_the_kv_gather_volume():
    # K/V gather and K/V weight traffic scale with the K/V width; multi-head is the special case hk = h
    B, S, h, F, D = 1, 131072, 4096, 16384, 8
    mha = O.forward_comm_elements(B, S, h, F, D, "tsp")
    assert O.forward_comm_elements(B, S, h, F, D, "tsp", kv_hidden=h) == mha
    gqa = O.forward_comm_elements(B, S, h, F, D, "tsp", kv_hidden=h // 4)
    kv_saved = 2 * B * S * (h - h // 4) * (D - 1) / D
    w_saved = (D - 1) * (2 * h * (h - h // 4) // D)
    assert mha - gqa == pytest.approx(kv_saved + w_saved)

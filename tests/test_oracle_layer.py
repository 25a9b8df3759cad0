"""Pins of the oracle's attention, MLP, full layer and TSP schedule (no GPU).

The brute-force functions below are written independently of the oracle:
pure-Python loops, math.exp, no max subtraction, no numpy matmul.
"""
import math

import numpy as np
import pytest

from oracle import tsp_oracle as O


def _rand_w(rng, h, F, scale=1.0):
    return {
        "Wq": rng.standard_normal((h, h)) * scale / math.sqrt(h),
        "Wk": rng.standard_normal((h, h)) * scale / math.sqrt(h),
        "Wv": rng.standard_normal((h, h)) / math.sqrt(h),
        "Wo": rng.standard_normal((h, h)) / math.sqrt(h),
        "Wg": rng.standard_normal((h, F)) / math.sqrt(h),
        "Wu": rng.standard_normal((h, F)) / math.sqrt(h),
        "Wd": rng.standard_normal((F, h)) / math.sqrt(F),
    }


def _mv(vec, mat):  # row vector times matrix, loops
    return [sum(vec[i] * mat[i][j] for i in range(len(vec))) for j in range(len(mat[0]))]


def _brute_attention(Q, K, V, heads):
    S, h = len(Q), len(Q[0])
    dh = h // heads
    out = [[0.0] * h for _ in range(S)]
    lse = [[0.0] * S for _ in range(heads)]
    for e in range(heads):
        for i in range(S):
            ws = []
            for j in range(i + 1):
                dot = sum(Q[i][e * dh + d] * K[j][e * dh + d] for d in range(dh))
                ws.append(math.exp(dot / math.sqrt(dh)))
            z = sum(ws)
            lse[e][i] = math.log(z)
            for d in range(dh):
                out[i][e * dh + d] = sum(ws[j] / z * V[j][e * dh + d] for j in range(i + 1))
    return out, lse


def _brute_layer(x, w, heads):
    """Whole layer for one batch element, pure Python."""
    L = lambda a: a.tolist()
    Wq, Wk, Wv, Wo, Wg, Wu, Wd = (L(w[k]) for k in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd"))
    xs = L(x)
    Q = [_mv(t, Wq) for t in xs]
    K = [_mv(t, Wk) for t in xs]
    V = [_mv(t, Wv) for t in xs]
    att, _ = _brute_attention(Q, K, V, heads)
    A = [_mv(t, Wo) for t in att]
    H = [[a + b for a, b in zip(t, u)] for t, u in zip(xs, A)]
    mlp = []
    for t in H:
        g = _mv(t, Wg)
        u = _mv(t, Wu)
        m = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
        mlp.append(_mv(m, Wd))
    Y = [[a + b for a, b in zip(t, u)] for t, u in zip(H, mlp)]
    return np.array(A), np.array(H), np.array(mlp), np.array(Y)


@pytest.mark.parametrize("S,h,heads", [(1, 4, 1), (7, 6, 2), (12, 8, 4)])
def test_attention_matches_brute_force(S, h, heads):
    rng = np.random.default_rng(S * 100 + h)
    Q, K, V = (rng.standard_normal((S, h)) for _ in range(3))
    got, lse = O.causal_attention(Q, K, V, heads)
    ref, ref_lse = _brute_attention(Q.tolist(), K.tolist(), V.tolist(), heads)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(7)
    S, h, heads = 10, 8, 2
    Q = rng.standard_normal((S, h))
    V = rng.standard_normal((S, h))
    # all keys equal -> uniform weights over the visible prefix: O[i] = mean(v_0..v_i)
    K = np.tile(rng.standard_normal((1, h)), (S, 1))
    Oa, _ = O.causal_attention(Q, K, V, heads)
    means = np.cumsum(V, axis=0) / np.arange(1, S + 1)[:, None]
    assert np.allclose(Oa, means, rtol=0, atol=1e-13)
    # row 0 sees only itself
    K2 = rng.standard_normal((S, h))
    O2, _ = O.causal_attention(Q, K2, V, heads)
    assert np.array_equal(O2[0], V[0])
    # dh = 1 with huge logits selects the visible key with the largest score
    S3 = 9
    q = np.full((S3, 1), 1000.0)
    k = rng.permutation(S3).astype(float)[:, None]
    v = rng.standard_normal((S3, 1))
    O3, _ = O.causal_attention(q, k, v, 1)
    for i in range(S3):
        j = int(np.argmax(k[: i + 1, 0]))
        assert O3[i, 0] == pytest.approx(v[j, 0], abs=1e-12)


def test_attention_row_subset():
    rng = np.random.default_rng(3)
    Q, K, V = (rng.standard_normal((33, 8)) for _ in range(3))
    full, lse = O.causal_attention(Q, K, V, 2)
    rows = [0, 5, 17, 32]
    sub, lse_sub = O.causal_attention(Q, K, V, 2, rows=rows, row_block=3)
    assert np.allclose(sub, full[rows], atol=1e-14)
    assert np.allclose(lse_sub, lse[:, rows], atol=1e-14)


def test_layer_matches_brute_force():
    rng = np.random.default_rng(11)
    B, S, h, heads, F = 2, 6, 4, 2, 6
    x = rng.standard_normal((B, S, h))
    w = _rand_w(rng, h, F, scale=2.0)
    out = O.layer_fwd(x, w, heads)
    for b in range(B):
        A, H, mlp, Y = _brute_layer(x[b], w, heads)
        assert np.allclose(out["A"][b], A, rtol=1e-12, atol=1e-12)
        assert np.allclose(out["H"][b], H, rtol=1e-12, atol=1e-12)
        assert np.allclose(out["MLP"][b], mlp, rtol=1e-12, atol=1e-12)
        assert np.allclose(out["Y"][b], Y, rtol=1e-12, atol=1e-12)


def test_layer_rows_subset_equals_full():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 16, 8))
    w = _rand_w(rng, 8, 12)
    full = O.layer_fwd(x, w, 2)
    rows = [0, 3, 8, 15]
    sub = O.layer_fwd(x, w, 2, rows=rows)
    for k in ("A", "H", "MLP", "Y"):
        assert np.allclose(sub[k], full[k][:, rows], atol=1e-13)


def test_mlp_special_cases():
    assert O.silu(0.0) == 0.0
    assert O.silu_grad(0.0) == 0.5
    z = np.linspace(-6, 6, 25)
    eps = 1e-6
    fd = (O.silu(z + eps) - O.silu(z - eps)) / (2 * eps)
    assert np.allclose(O.silu_grad(z), fd, rtol=1e-8, atol=1e-9)
    # zero gate weights: M = 0, so the MLP adds nothing and Y = H
    rng = np.random.default_rng(2)
    x = rng.standard_normal((1, 8, 8))
    w = _rand_w(rng, 8, 16)
    w["Wg"] = np.zeros_like(w["Wg"])
    out = O.layer_fwd(x, w, 2)
    assert np.array_equal(out["MLP"], np.zeros_like(out["MLP"]))
    assert np.array_equal(out["Y"], out["H"])


@pytest.mark.parametrize("D", [1, 2, 4, 8])
def test_sharded_schedule_equals_unsharded(D):
    rng = np.random.default_rng(100 + D)
    B, S, h, heads, F = 2, 32, 16, 8, 24
    x = rng.standard_normal((B, S, h))
    w = _rand_w(rng, h, F)
    ref = O.layer_fwd(x, w, heads)
    got = O.tsp_layer_fwd_sharded(x, w, heads, D)
    for k in ("A", "H", "MLP", "Y"):
        err = np.linalg.norm(got[k] - ref[k]) / np.linalg.norm(ref[k])
        assert err <= 1e-12, (k, err)


def test_shards_tile_the_weights():
    rng = np.random.default_rng(9)
    w = _rand_w(rng, 16, 24)
    D = 4
    # column split then row split reassembles every weight exactly
    assert np.array_equal(np.concatenate([O.attention_shard(w, s, D)[0] for s in range(D)], 1), w["Wq"])
    assert np.array_equal(np.concatenate([O.attention_shard(w, s, D)[3] for s in range(D)], 0), w["Wo"])
    assert np.array_equal(np.concatenate([O.mlp_shard(w, j, D)[1] for j in range(D)], 1), w["Wu"])
    assert np.array_equal(np.concatenate([O.mlp_shard(w, j, D)[2] for j in range(D)], 0), w["Wd"])


def test_comm_break_even_is_8h():
    # with F = 4h the TSP forward volume equals TP's exactly at B*S = 8h
    for h in (1024, 4096, 8192):
        F = 4 * h
        for D in (2, 8):
            at = O.forward_comm_elements(1, 8 * h, h, F, D, "tsp")
            assert at == pytest.approx(O.forward_comm_elements(1, 8 * h, h, F, D, "tp"))
            assert O.forward_comm_elements(1, 16 * h, h, F, D, "tsp") < O.forward_comm_elements(1, 16 * h, h, F, D, "tp")
            assert O.forward_comm_elements(1, 4 * h, h, F, D, "tsp") > O.forward_comm_elements(1, 4 * h, h, F, D, "tp")

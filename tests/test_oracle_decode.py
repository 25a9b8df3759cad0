"""Pins of the oracle's decode step (no GPU).

(1) A decode step on an exact cache equals the last row of the full forward
over the same tokens; (2) decoding token by token from an empty cache
reproduces every row of the forward; (3) the rank-sharded attention with the
log-sum-exp merge equals the plain softmax row, for every position (chunk
edges included) and D; (4) special cases: pos = 0 attends only to itself.
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


@pytest.mark.parametrize("heads,kv_heads", [(4, 4), (4, 2)])
def test_decode_step_is_the_last_forward_row(heads, kv_heads):
    rng = np.random.default_rng(31)
    dh, B, S, F = 4, 2, 9, 24
    h = heads * dh
    w = _weights(rng, h, kv_heads * dh, F)
    x = rng.standard_normal((B, S, h))
    pos = S - 1
    Kc, Vc = x @ w["Wk"], x @ w["Wv"]  # exact cache of positions 0..S-1 (row pos is ignored)
    Y, k, v = O.decode_step(x[:, pos], w, heads, Kc, Vc, pos)
    ref = O.layer_fwd(x, w, heads)["Y"][:, pos]
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(k, Kc[:, pos], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(v, Vc[:, pos], rtol=1e-13, atol=1e-13)


def test_token_by_token_decoding_reproduces_the_forward():
    rng = np.random.default_rng(32)
    heads, kv_heads, dh, B, S, F = 4, 2, 4, 1, 7, 16
    h = heads * dh
    w = _weights(rng, h, kv_heads * dh, F)
    x = rng.standard_normal((B, S, h))
    Kc = np.zeros((B, S, kv_heads * dh))
    Vc = np.zeros_like(Kc)
    ys = []
    for p in range(S):
        Y, k, v = O.decode_step(x[:, p], w, heads, Kc, Vc, p)
        Kc[:, p], Vc[:, p] = k, v
        ys.append(Y)
    np.testing.assert_allclose(np.stack(ys, axis=1), O.layer_fwd(x, w, heads)["Y"], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("D", [1, 2, 4])
def test_rank_sharded_decode_attention_equals_softmax(D):
    rng = np.random.default_rng(33)
    heads, kv_heads, dh = 4, 2, 8
    h, S = heads * dh, 2 * D * 6
    K = rng.standard_normal((S, kv_heads * dh))
    V = rng.standard_normal((S, kv_heads * dh))
    C = S // (2 * D)
    positions = sorted({0, 1, C - 1, C, 2 * C - 1, S // 2, S - 2, S - 1})
    for pos in positions:
        q = rng.standard_normal(h) * 2.0
        Q = np.zeros((S, h))
        Q[pos] = q
        ref, _ = O.causal_attention(Q, K, V, heads, rows=[pos])
        got = O.decode_attention_by_rank(q, K, V, heads, pos, D)
        np.testing.assert_allclose(got, ref[0], rtol=1e-12, atol=1e-12)


def test_first_token_attends_only_to_itself():
    rng = np.random.default_rng(34)
    heads, dh, F = 2, 4, 8
    h = heads * dh
    w = _weights(rng, h, h, F)
    x = rng.standard_normal((1, h))
    Y, k, v = O.decode_step(x, w, heads, np.zeros((1, 4, h)), np.zeros((1, 4, h)), 0)
    Hm = x + v @ w["Wo"]  # softmax over a single key is 1: O = v
    np.testing.assert_allclose(Y, Hm + O.gated_mlp(Hm, w), rtol=1e-13, atol=1e-13)

"""Pins of the oracle's zigzag partition and causal balance (no GPU)."""
import os

import numpy as np
import pytest

from oracle import tsp_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln for ln in f.read().splitlines() if ln and not ln.startswith("#")]


def test_listing_D2_S8():
    pos = O.zigzag_positions(8, 2)
    for ln in _read("zigzag_D2_S8.txt"):
        r, rest = ln.split(":")
        assert pos[int(r)].tolist() == [int(t) for t in rest.split()]


@pytest.mark.parametrize("S,D", [(8, 1), (8, 2), (16, 4), (64, 8), (96, 3), (256, 2), (4096, 8)])
def test_bijection_and_local_sizes(S, D):
    pos = O.zigzag_positions(S, D)
    assert pos.shape == (D, S // D)  # every rank holds S/D tokens
    assert sorted(pos.ravel().tolist()) == list(range(S))
    C = S // (2 * D)
    for r in range(D):
        # rank r: chunk r ascending, then chunk 2D-1-r ascending
        assert pos[r, 0] == r * C and pos[r, C] == (2 * D - 1 - r) * C
        assert np.all(np.diff(pos[r, :C]) == 1) and np.all(np.diff(pos[r, C:]) == 1)


@pytest.mark.parametrize("S,D,B", [(16, 2, 2), (64, 4, 1), (128, 8, 3)])
def test_permute_unpermute_identity(S, D, B):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((B, S, 5))
    xz = O.zigzag_permute(x, D)
    assert xz.shape == (D, B, S // D, 5)
    assert np.array_equal(O.zigzag_unpermute(xz, D), x)
    # the permutation is a pure reindex: every value appears exactly where pos says
    pos = O.zigzag_positions(S, D)
    for r in range(D):
        assert np.array_equal(xz[r], x[:, pos[r]])


def _visits_brute(S, D):
    C = S // (2 * D)
    out = []
    for r in range(D):
        tot = 0
        for chunk in (r, 2 * D - 1 - r):
            for p in range(chunk * C, (chunk + 1) * C):
                tot += p + 1  # query p sees keys 0..p
        out.append(tot)
    return out


def test_causal_balance_closed_form():
    for ln in _read("causal_balance.txt"):
        D, S, v = (int(t) for t in ln.split())
        C = S // (2 * D)
        assert C * C * (2 * D - 1) + C * (C + 1) == v
        got = O.causal_key_visits_per_rank(S, D)
        assert got.tolist() == [v] * D
        if S <= 16384:
            assert _visits_brute(S, D) == [v] * D
        # the per-rank share is exactly 1/D of the causal triangle
        assert D * v == S * (S + 1) // 2


def test_tile_level_mirror_pairs_balanced():
    # q-tile g of size T (n tiles per chunk) needs g+1 key tiles; pairing g with its
    # mirror 2Dn-1-g (same rank) costs 2Dn+1 tiles for every pair.
    for D, n in [(2, 1), (4, 4), (8, 8), (8, 32)]:
        G = 2 * D * n
        costs = {(g + 1) + (G - 1 - g + 1) for g in range(G // 2)}
        assert costs == {G + 1}
        for g in range(G):
            c = g // n
            cm = (G - 1 - g) // n
            assert min(c, 2 * D - 1 - c) == min(cm, 2 * D - 1 - cm)  # same rank

"""Pin of the oracle's backward: central finite differences in fp64 (no GPU)."""
import numpy as np

from oracle import tsp_oracle as O


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(4)
    B, S, h, heads, F = 1, 8, 8, 2, 16
    x = rng.standard_normal((B, S, h))
    w = {
        "Wq": rng.standard_normal((h, h)) / np.sqrt(h),
        "Wk": rng.standard_normal((h, h)) / np.sqrt(h),
        "Wv": rng.standard_normal((h, h)) / np.sqrt(h),
        "Wo": rng.standard_normal((h, h)) / np.sqrt(h),
        "Wg": rng.standard_normal((h, F)) / np.sqrt(h),
        "Wu": rng.standard_normal((h, F)) / np.sqrt(h),
        "Wd": rng.standard_normal((F, h)) / np.sqrt(F),
    }
    dY = rng.standard_normal((B, S, h))
    dx, g = O.layer_bwd(x, w, heads, dY)

    def loss(xx, ww):
        return float(np.sum(O.layer_fwd(xx, ww, heads)["Y"] * dY))

    eps = 1e-6

    def fd_of(arr, setter):
        out = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = arr[i]
            arr[i] = old + eps
            lp = setter()
            arr[i] = old - eps
            lm = setter()
            arr[i] = old
            out[i] = (lp - lm) / (2 * eps)
        return out

    fdx = fd_of(x, lambda: loss(x, w))
    assert np.linalg.norm(fdx - dx) / np.linalg.norm(dx) < 1e-6
    for k in w:
        fdw = fd_of(w[k], lambda: loss(x, w))
        err = np.linalg.norm(fdw - g[k]) / np.linalg.norm(g[k])
        assert err < 1e-6, (k, err)


def test_backward_returns_forward_output():
    rng = np.random.default_rng(8)
    B, S, h, heads, F = 2, 6, 4, 2, 8
    x = rng.standard_normal((B, S, h))
    w = {k: rng.standard_normal(s) * 0.5 for k, s in
         {"Wq": (h, h), "Wk": (h, h), "Wv": (h, h), "Wo": (h, h), "Wg": (h, F), "Wu": (h, F), "Wd": (F, h)}.items()}
    dY = rng.standard_normal((B, S, h))
    dx, g, Y = O.layer_bwd(x, w, heads, dY, return_y=True)
    dx2, g2 = O.layer_bwd(x, w, heads, dY)
    assert np.allclose(Y, O.layer_fwd(x, w, heads)["Y"], rtol=1e-13, atol=1e-13)
    assert np.array_equal(dx, dx2) and all(np.array_equal(g[k], g2[k]) for k in g)

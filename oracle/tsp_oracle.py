"""fp64 CPU oracle of one TSP transformer layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's ``smoke()`` entry and the benchmark's CPU
baseline leg may import this module.  The CUDA library never calls it and it
never calls the CUDA library; the two share no code.  Inputs come from the
seeded generator (``folded_tensor_sequence_gb300.synth``) as fp64 arrays whose
values are already rounded to the storage dtype; this module does not import
it.

What it computes (plain definitions, fp64, numpy):

* The zigzag token partition: the sequence is cut into 2D equal chunks and
  virtual rank r holds chunk r followed by chunk 2D-1-r.  The TSP posts only
  name a "zigzag" reorder of K/V before FlashAttention (ai-trends.today,
  "Zyphra Introduces Tensor and Sequence Parallelism (TSP)", section "How to
  Fold a Book"; edge.aivizor.me TSP news post, paragraph on layer execution);
  the 2D-chunk rule is the load-balancing split the ring-attention section of
  the r007 "Распределенное обучение" chapter alludes to ("Параллелизм по
  контексту: Ring Attention против Ulysses").
* The unsharded layer, row-vector convention y = x W:
    Q = x Wq, K = x Wk, V = x Wv, per head causal softmax attention with scale
    1/sqrt(dh); A = concat_heads(O) Wo; H = x + A;
    M = SiLU(H Wg) * (H Wu); Y = H + M Wd.
  No norm, no bias, no positional term (the posts name only attention and the
  gated MLP with gate, up and down projections, "How to Fold a Book").
* Its exact gradient (``layer_bwd``).
* The same layer computed the TSP way (``tsp_layer_fwd_sharded``): iterate
  over attention weight shards, project every rank's local tokens, gather K/V
  into natural order, attend, accumulate the row-sharded W_O partial sums on
  the rank; then the gated-MLP ring where each rank starts from its own
  gate/up/down shard and accumulates partial outputs with no all-reduce
  ("How to Fold a Book").  Used only to check that the sharded schedule equals
  the plain definition (column split X[W1|W2] = [XW1|XW2] and row split
  XW = X1W1 + X2W2, r007 chapter, section "Тензорный параллелизм").
* Causal key-visit counts per rank and the forward communication-volume model
  behind the break-even B*S > 8h ("The Practicality of Trade-offs").
* A decode step against a key/value cache (``decode_step``) and its
  attention computed the TSP way over a cache sharded by the zigzag rule,
  with per-rank partial softmax results merged by log-sum-exp
  (``decode_attention_by_rank``).
* Grouped-query attention: K and V may have fewer heads than Q (Wk, Wv of
  shape [h, Hk*dh]); the r007 chapter names GQA, with the K/V head count
  often cut to 8, as what bounds a head-split degree ("Параллелизм по
  контексту: Ring Attention против Ulysses").  Reading where the pages are
  silent: query head e reads K/V head e // (H/Hk) (consecutive query heads
  share one K/V head), and a TSP shard owns H/D query heads and Hk/D K/V
  heads, so Hk must be divisible by D.  Hk = H is plain multi-head attention.

Readings where the pages are silent are stated next to each function.
Every function is pinned by tests/test_oracle_*.py against closed forms,
brute force and finite differences.
"""

from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# Zigzag partition
# ---------------------------------------------------------------------------

def zigzag_positions(S: int, D: int) -> np.ndarray:
    """pos[r, k] = global position of local token k on rank r.

    Chunk length C = S / (2D).  Local tokens 0..C-1 are chunk r, local tokens
    C..2C-1 are chunk 2D-1-r.
    """
    if S % (2 * D):
        raise ValueError("seq must be divisible by 2*D")
    C = S // (2 * D)
    pos = np.empty((D, 2 * C), dtype=np.int64)
    for r in range(D):
        pos[r, :C] = r * C + np.arange(C)
        pos[r, C:] = (2 * D - 1 - r) * C + np.arange(C)
    return pos


def zigzag_permute(x: np.ndarray, D: int) -> np.ndarray:
    """x [B, S, ...] natural order -> xz [D, B, 2C, ...] rank-major zigzag."""
    pos = zigzag_positions(x.shape[1], D)
    return np.stack([x[:, pos[r]] for r in range(D)], axis=0)


def zigzag_unpermute(xz: np.ndarray, D: int) -> np.ndarray:
    """Inverse of ``zigzag_permute``."""
    Dd, B, twoC = xz.shape[:3]
    S = D * twoC
    pos = zigzag_positions(S, D)
    x = np.empty((B, S) + xz.shape[3:], dtype=xz.dtype)
    for r in range(D):
        x[:, pos[r]] = xz[r]
    return x


def causal_key_visits_per_rank(S: int, D: int) -> np.ndarray:
    """Number of (query, key) pairs with key <= query that each rank's queries need."""
    pos = zigzag_positions(S, D)
    return (pos + 1).sum(axis=1)


# ---------------------------------------------------------------------------
# Layer pieces (plain definitions)
# ---------------------------------------------------------------------------

def silu(z):
    """SiLU(z) = z / (1 + exp(-z)); the gated MLP is SwiGLU."""
    return z / (1.0 + np.exp(-z))


def silu_grad(z):
    """d/dz SiLU(z) = sigma(z) * (1 + z * (1 - sigma(z)))."""
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def kv_head_slice(e: int, heads: int, kv_heads: int, dh: int) -> slice:
    """Columns of K/V read by query head e: K/V head e // (heads / kv_heads)."""
    if heads % kv_heads:
        raise ValueError("heads must be a multiple of kv_heads")
    g = e // (heads // kv_heads)
    return slice(g * dh, (g + 1) * dh)


def causal_attention(Q, K, V, heads: int, rows=None, row_block: int = 1024):
    """Causal softmax attention per head, natural positions.

    Q: [S, h] for one batch element (h = heads * dh); K, V: [S, Hk*dh] with
    Hk K/V heads (Hk = heads for multi-head attention, fewer for GQA).
    ``rows`` selects the query positions to evaluate (default: all).  Key j is
    visible to query i iff j <= i (global positions, diagonal included); scale
    1/sqrt(dh).  Returns (O [len(rows), h], lse [heads, len(rows)]) with lse
    the natural log-sum-exp of the scaled, masked scores.  Rows are processed
    in blocks only to bound memory; each row is computed on its own.
    """
    S, h = Q.shape
    dh = h // heads
    kv_heads = K.shape[1] // dh
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.zeros((len(rows), h))
    lse = np.zeros((heads, len(rows)))
    scale = 1.0 / math.sqrt(dh)
    keys = np.arange(S)
    for e in range(heads):
        sl = slice(e * dh, (e + 1) * dh)
        kv = kv_head_slice(e, heads, kv_heads, dh)
        for b0 in range(0, len(rows), row_block):
            rb = rows[b0:b0 + row_block]
            s = (Q[rb, sl] @ K[:, kv].T) * scale
            visible = keys[None, :] <= rb[:, None]
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1, keepdims=True)
            O[b0:b0 + len(rb), sl] = (p / l) @ V[:, kv]
            lse[e, b0:b0 + len(rb)] = (m + np.log(l))[:, 0]
    return O, lse


def gated_mlp(Hm, w):
    """SwiGLU MLP without the residual: (SiLU(H Wg) * (H Wu)) Wd, rows of H independent."""
    return (silu(Hm @ w["Wg"]) * (Hm @ w["Wu"])) @ w["Wd"]


def layer_fwd(x, w, heads: int, rows=None):
    """Unsharded layer forward in fp64.

    x: [B, S, h]; w: dict with Wq, Wo [h, h], Wk, Wv [h, Hk*dh] (Hk = heads
    unless the layer uses grouped-query attention), Wg, Wu [h, F], Wd [F, h].
    ``rows`` (optional) restricts every per-token output to those natural
    positions (K and V are still computed for all tokens, since attention needs
    them).  Returns dict of [B, R, .] arrays:
      A   = attention output after W_O, before the residual,
      H   = x + A,
      MLP = SiLU(H Wg) * (H Wu) @ Wd (before the residual),
      Y   = H + MLP,
    and ``lse`` [B, heads, R].
    """
    B, S, h = x.shape
    rows_arr = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    out = {k: [] for k in ("A", "H", "MLP", "Y", "O", "lse")}
    for b in range(B):
        xb = x[b]
        K = xb @ w["Wk"]
        V = xb @ w["Wv"]
        Q = np.zeros((S, h))
        Q[rows_arr] = xb[rows_arr] @ w["Wq"]
        O, lse = causal_attention(Q, K, V, heads, rows_arr)
        A = O @ w["Wo"]
        Hb = xb[rows_arr] + A
        mlp = gated_mlp(Hb, w)
        out["A"].append(A)
        out["H"].append(Hb)
        out["MLP"].append(mlp)
        out["Y"].append(Hb + mlp)
        out["O"].append(O)
        out["lse"].append(lse)
    return {k: np.stack(v) for k, v in out.items()}


def _head_probs(Q, K, sl, kv, scale, mask):
    """Causal softmax probabilities of one head (rows: queries, columns: keys);
    sl: the head's Q columns, kv: its K columns."""
    s = np.where(mask, (Q[:, sl] @ K[:, kv].T) * scale, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    return p / p.sum(axis=1, keepdims=True)


def layer_bwd(x, w, heads: int, dY, return_y: bool = False):
    """Exact gradient of ``layer_fwd``'s Y with respect to x and all weights, fp64.

    The posts do not describe the TSP backward; its plainest reading is the
    gradient of the same function (sharding changes placement and rounding,
    not values).  Steps, per batch element and head:
      dM = dY Wd^T; dWd = M^T dY; dG = dM * U * SiLU'(G); dU = dM * SiLU(G);
      dH = dY + dG Wg^T + dU Wu^T; dWg = H^T dG; dWu = H^T dU;
      dWo = O^T dH; dO = dH Wo^T; per head: dV = P^T dO, dP = dO V^T,
      dS = P * (dP - rowsum(dP * P)), dQ = dS K / sqrt(dh), dK = dS^T Q / sqrt(dh);
      dWq = x^T dQ (likewise K, V); dx = dH + dQ Wq^T + dK Wk^T + dV Wv^T.
    With grouped-query attention a K/V head's dK and dV are the sums over the
    query heads that read it.
    """
    B, S, h = x.shape
    dh = h // heads
    kv_heads = w["Wk"].shape[1] // dh
    scale = 1.0 / math.sqrt(dh)
    grads = {k: np.zeros_like(v) for k, v in w.items()}
    dx = np.zeros_like(x)
    Y = np.zeros_like(x) if return_y else None
    mask = np.tril(np.ones((S, S), dtype=bool))
    for b in range(B):
        xb = x[b]
        Q, K, V = xb @ w["Wq"], xb @ w["Wk"], xb @ w["Wv"]
        O = np.zeros((S, h))
        for e in range(heads):
            sl = slice(e * dh, (e + 1) * dh)
            kv = kv_head_slice(e, heads, kv_heads, dh)
            O[:, sl] = _head_probs(Q, K, sl, kv, scale, mask) @ V[:, kv]
        Hb = xb + O @ w["Wo"]
        G, U = Hb @ w["Wg"], Hb @ w["Wu"]
        M = silu(G) * U
        if return_y:
            Y[b] = Hb + M @ w["Wd"]
        dYb = dY[b]
        dM = dYb @ w["Wd"].T
        grads["Wd"] += M.T @ dYb
        dG = dM * U * silu_grad(G)
        dU = dM * silu(G)
        grads["Wg"] += Hb.T @ dG
        grads["Wu"] += Hb.T @ dU
        dH = dYb + dG @ w["Wg"].T + dU @ w["Wu"].T
        grads["Wo"] += O.T @ dH
        dO = dH @ w["Wo"].T
        dQ = np.zeros((S, h))
        dK = np.zeros_like(K)
        dV = np.zeros_like(V)
        for e in range(heads):
            sl = slice(e * dh, (e + 1) * dh)
            kv = kv_head_slice(e, heads, kv_heads, dh)
            p = _head_probs(Q, K, sl, kv, scale, mask)  # recomputed per head to bound memory
            dV[:, kv] += p.T @ dO[:, sl]
            dP = dO[:, sl] @ V[:, kv].T
            dS = p * (dP - (dP * p).sum(axis=1, keepdims=True))
            dQ[:, sl] = dS @ K[:, kv] * scale
            dK[:, kv] += dS.T @ Q[:, sl] * scale
        grads["Wq"] += xb.T @ dQ
        grads["Wk"] += xb.T @ dK
        grads["Wv"] += xb.T @ dV
        dx[b] = dH + dQ @ w["Wq"].T + dK @ w["Wk"].T + dV @ w["Wv"].T
    if return_y:
        return dx, grads, Y
    return dx, grads


# ---------------------------------------------------------------------------
# The layer computed the TSP way (checks the schedule's algebra)
# ---------------------------------------------------------------------------

def attention_shard(w, s: int, D: int):
    """Packed attention shard s: Q columns and W_O rows of query heads
    s*H/D .. (s+1)*H/D-1, K/V columns of K/V heads s*Hk/D .. (s+1)*Hk/D-1.

    Reading: attention weights are sharded by head (softmax needs whole rows,
    so a head cannot be split; bowenzhou.top "张量并行", 机制：行切与列切).
    With GQA the shard's query heads read exactly its own K/V heads, since
    consecutive query heads share a K/V head.
    """
    h, hk = w["Wq"].shape[0], w["Wk"].shape[1]
    lo, hi = s * h // D, (s + 1) * h // D
    klo, khi = s * hk // D, (s + 1) * hk // D
    return w["Wq"][:, lo:hi], w["Wk"][:, klo:khi], w["Wv"][:, klo:khi], w["Wo"][lo:hi, :]


def mlp_shard(w, j: int, D: int):
    """Gate/up columns and down rows j*F/D .. (j+1)*F/D-1 (column split then row split)."""
    F = w["Wg"].shape[1]
    lo, hi = j * F // D, (j + 1) * F // D
    return w["Wg"][:, lo:hi], w["Wu"][:, lo:hi], w["Wd"][lo:hi, :]


def tsp_layer_fwd_sharded(x, w, heads: int, D: int):
    """The layer as D ranks compute it under TSP, emulated in one address space.

    Rank r holds local tokens xz[r] (zigzag) and weight shard r.  Attention
    iterates over weight shards s; every rank projects its own tokens with
    shard s, the local K/V are gathered over all ranks and put back into
    natural order, each rank attends with its own queries, and multiplies by
    shard s's W_O rows, accumulating the partial output locally.  The MLP is a
    ring: at step t rank r holds shard (r - t) mod D, starting from its own,
    and accumulates SiLU(H Wg_j) * (H Wu_j) Wd_j with no all-reduce.
    Returns natural-order A, H, MLP, Y (same keys as ``layer_fwd``).
    """
    B, S, h = x.shape
    dh = h // heads
    kv_heads = w["Wk"].shape[1] // dh
    if heads % D or kv_heads % D or h % D or w["Wg"].shape[1] % D:
        raise ValueError("heads, kv heads, hidden and ffn must be divisible by D")
    pos = zigzag_positions(S, D)
    xz = zigzag_permute(x, D)  # [D, B, 2C, h]
    twoC = xz.shape[2]
    Az = np.zeros_like(xz)
    hps = heads // D  # heads per shard
    scale = 1.0 / math.sqrt(dh)
    for s in range(D):  # the owner of shard s broadcasts it
        Wq_s, Wk_s, Wv_s, Wo_s = attention_shard(w, s, D)
        Qs = [xz[r] @ Wq_s for r in range(D)]          # local projections
        Ks = [xz[r] @ Wk_s for r in range(D)]
        Vs = [xz[r] @ Wv_s for r in range(D)]
        Kfull = np.zeros((B, S, Wk_s.shape[1]))         # all-gather + zigzag reorder
        Vfull = np.zeros((B, S, Wv_s.shape[1]))
        for r in range(D):
            Kfull[:, pos[r]] = Ks[r]
            Vfull[:, pos[r]] = Vs[r]
        for r in range(D):
            Os = np.zeros((B, twoC, h // D))
            for b in range(B):
                for e in range(hps):
                    sl = slice(e * dh, (e + 1) * dh)
                    kv = kv_head_slice(e, hps, kv_heads // D, dh)  # within the shard
                    sc = (Qs[r][b, :, sl] @ Kfull[b, :, kv].T) * scale
                    sc = np.where(np.arange(S)[None, :] <= pos[r][:, None], sc, -np.inf)
                    p = np.exp(sc - sc.max(axis=1, keepdims=True))
                    p /= p.sum(axis=1, keepdims=True)
                    Os[b, :, sl] = p @ Vfull[b, :, kv]
            Az[r] += Os @ Wo_s                          # partial output stays on rank r
    Hz = xz + Az
    MLPz = np.zeros_like(xz)
    for r in range(D):
        for t in range(D):
            j = (r - t) % D
            Wg_j, Wu_j, Wd_j = mlp_shard(w, j, D)
            MLPz[r] += (silu(Hz[r] @ Wg_j) * (Hz[r] @ Wu_j)) @ Wd_j
    Yz = Hz + MLPz
    return {
        "A": zigzag_unpermute(Az, D),
        "H": zigzag_unpermute(Hz, D),
        "MLP": zigzag_unpermute(MLPz, D),
        "Y": zigzag_unpermute(Yz, D),
    }


# ---------------------------------------------------------------------------
# Decoding (one new token per sequence against a key/value cache)
# ---------------------------------------------------------------------------

def decode_step(x_new, w, heads: int, K_cache, V_cache, pos: int):
    """One decode step of the layer, fp64.

    The posts present TSP for inference as well as training ("for both
    training and inference workloads", ai-trends.today TSP article,
    introduction; the 7B model is "a reference for decoding", "Memory and
    Processing Results").  Plainest reading of a decode step: each of the B
    sequences holds ``pos`` cached tokens (positions 0..pos-1) and appends the
    token x_new at position ``pos``; that token attends to every cached key
    and to itself (all are at earlier or equal positions).

    x_new: [B, h]; K_cache, V_cache: [B, >= pos, hk] (row p = key/value of
    position p, hk = Hk*dh); only rows < pos are read.  Returns
    (Y [B, h], k_new [B, hk], v_new [B, hk]).
    """
    B, h = x_new.shape
    dh = h // heads
    kv_heads = w["Wk"].shape[1] // dh
    scale = 1.0 / math.sqrt(dh)
    q, k, v = x_new @ w["Wq"], x_new @ w["Wk"], x_new @ w["Wv"]
    Y = np.zeros((B, h))
    for b in range(B):
        O = np.zeros(h)
        for e in range(heads):
            sl = slice(e * dh, (e + 1) * dh)
            kv = kv_head_slice(e, heads, kv_heads, dh)
            # scores against the cached positions 0..pos-1 and the new token itself
            s = np.append(K_cache[b, :pos, kv] @ q[b, sl], k[b, kv] @ q[b, sl]) * scale
            p = np.exp(s - s.max())
            p /= p.sum()
            O[sl] = p[:pos] @ V_cache[b, :pos, kv] + p[pos] * v[b, kv]
        Hb = x_new[b] + O @ w["Wo"]
        Y[b] = Hb + gated_mlp(Hb[None, :], w)[0]
    return Y, k, v


def decode_attention_by_rank(q, K, V, heads: int, pos: int, D: int):
    """Attention of one new query (position pos) the TSP way: the cache of
    2D*C positions is sharded over D ranks by the zigzag rule (rank r holds
    chunks r and 2D-1-r); every rank computes, per head, the running max m_r,
    the sum l_r of exp(score - m_r) and the unnormalised output O_r over its
    own cached keys with position <= pos; the partial results are merged with
    the log-sum-exp rule m = max m_r, l = sum l_r e^(m_r - m),
    O = sum O_r e^(m_r - m) / l (the combination FlashAttention's online
    softmax uses; r007 chapter, "Параллелизм по контексту: Ring Attention
    против Ulysses").  q: [h]; K, V: [S, hk] with S = 2DC.  Returns O [h].
    """
    S, _ = K.shape
    h = q.shape[0]
    dh = h // heads
    kv_heads = K.shape[1] // dh
    pos_of = zigzag_positions(S, D)
    scale = 1.0 / math.sqrt(dh)
    out = np.zeros(h)
    for e in range(heads):
        sl = slice(e * dh, (e + 1) * dh)
        kv = kv_head_slice(e, heads, kv_heads, dh)
        parts = []
        for r in range(D):
            keys = pos_of[r][pos_of[r] <= pos]
            if len(keys) == 0:
                continue
            s = (K[keys, kv] @ q[sl]) * scale
            m = s.max()
            p = np.exp(s - m)
            parts.append((m, p.sum(), p @ V[keys, kv]))
        m = max(pm for pm, _, _ in parts)
        l = sum(pl * math.exp(pm - m) for pm, pl, _ in parts)
        out[sl] = sum(po * math.exp(pm - m) for pm, _, po in parts) / l
    return out


# ---------------------------------------------------------------------------
# Communication-volume model (forward, per rank, elements)
# ---------------------------------------------------------------------------

def forward_comm_elements(B: int, S: int, h: int, F: int, D: int, scheme: str, kv_hidden: int | None = None) -> float:
    """Elements each rank receives in one layer forward.

    tsp: attention weights of the D-1 remote shards ((2 h*h + 2 h*hk)/D each,
    hk = Hk*dh the K/V width, h for multi-head attention), the MLP ring's D-1
    hops (3 h * F/D each) and the K/V all-gather (2 * B*S*hk/D elements from
    each of the other D-1 ranks, head-sharded: 2 B S hk (D-1)/D^2 per shard
    step, summed over D shard steps).
    tp: two ring all-reduces of the full activation, 2 (D-1)/D * B*S*h each
    (bowenzhou.top "张量并行"; r007 chapter, "Тензорный параллелизм").
    """
    hk = h if kv_hidden is None else kv_hidden
    if scheme == "tsp":
        weights = (D - 1) * ((2 * h * h + 2 * h * hk) // D + 3 * h * F // D)
        kv = 2 * B * S * hk * (D - 1) / D
        return weights + kv
    if scheme == "tp":
        return 2 * 2 * (D - 1) / D * B * S * h
    raise ValueError(scheme)

"""CPU (fp64) stand-in for one rank's compute steps, for the multi-process
schedule tests -- test infrastructure built on the oracle's definitions.

``pack_attention_shard`` / ``pack_mlp_shard`` write a rank's weight shards in
the layout include/tsp.h documents for the tsp_rank_* calls, from the
oracle's own shard definitions (``attention_shard``, ``mlp_shard``);
:class:`OracleRankCompute` provides the same steps and buffers as the CUDA
``RankLayer`` (project, attend, mlp), computed in fp64 numpy, and records
every shard it was handed so a test can check what travelled.
"""
import numpy as np
import torch

from oracle import tsp_oracle as O


def pack_attention_shard(w, s, D):
    """[qkv_s (Q|K|V output columns as rows) [hs+2ks][h] | o_s [h][hs]] flattened, fp64."""
    Wq, Wk, Wv, Wo = O.attention_shard(w, s, D)  # [h][hs], [h][ks], [h][ks], [hs][h]
    qkv = np.concatenate([Wq, Wk, Wv], axis=1).T
    return np.concatenate([qkv.ravel(), Wo.T.ravel()])


def pack_mlp_shard(w, j, D):
    """[gu_j (128-column gate/up blocks as rows) [2fs][h] | down_j [h][fs]] flattened, fp64."""
    Wg, Wu, Wd = O.mlp_shard(w, j, D)  # [h][fs], [h][fs], [fs][h]
    fs = Wg.shape[1]
    blocks = []
    for q in range(fs // 128):
        blocks += [Wg[:, q * 128:(q + 1) * 128].T, Wu[:, q * 128:(q + 1) * 128].T]
    gu = np.concatenate(blocks, axis=0)
    return np.concatenate([gu.ravel(), Wd.T.ravel()])


class OracleRankCompute:
    """Rank ``rank``'s compute steps in fp64 (same interface as RankLayer)."""

    def __init__(self, rank, D, batch, seq, hidden, heads, kv_heads, ffn):
        self.rank, self.D, self.B, self.S, self.hid = rank, D, batch, seq, hidden
        self.heads, dh = heads, hidden // heads
        self.hs, self.ks, self.fs = hidden // D, kv_heads * dh // D, ffn // D
        self.C = seq // (2 * D)
        L = batch * 2 * self.C
        f = dict(dtype=torch.float64)
        self.q = torch.zeros(L, self.hs, **f)
        self.kv = torch.zeros(L, 2 * self.ks, **f)
        self.kv_all = torch.zeros(D, L, 2 * self.ks, **f)
        self.h = torch.zeros(L, hidden, **f)
        self.y = torch.zeros(L, hidden, **f)
        na = (self.hs + 2 * self.ks) * hidden + hidden * self.hs
        nm = 2 * self.fs * hidden + hidden * self.fs
        self.attn_recv = [torch.zeros(na, **f) for _ in range(2)]
        self.mlp_recv = [torch.zeros(nm, **f) for _ in range(2)]
        self.pos = O.zigzag_positions(seq, D)
        self.seen_attn, self.seen_kv_all, self.seen_mlp = [], [], []

    def _attn(self, shard):
        a = shard.numpy()
        n = (self.hs + 2 * self.ks) * self.hid
        qkv = a[:n].reshape(self.hs + 2 * self.ks, self.hid)
        o = a[n:].reshape(self.hid, self.hs)
        return (qkv[:self.hs].T, qkv[self.hs:self.hs + self.ks].T, qkv[self.hs + self.ks:].T, o.T)

    def project(self, x_local, shard):
        self.seen_attn.append(shard.clone())
        Wq, Wk, Wv, _ = self._attn(shard)
        x = x_local.numpy()
        self.q.copy_(torch.from_numpy(x @ Wq))
        self.kv.copy_(torch.from_numpy(x @ np.concatenate([Wk, Wv], axis=1)))
        return self.kv

    def attend(self, shard, resid):
        self.seen_kv_all.append(self.kv_all.clone())
        _, _, _, Wo = self._attn(shard)
        twoC, ks = 2 * self.C, self.ks
        kv_all = self.kv_all.numpy()
        O_local = np.zeros((self.B * twoC, self.hs))
        for b in range(self.B):
            K = np.zeros((self.S, ks))
            V = np.zeros((self.S, ks))
            for q in range(self.D):  # gathered rows of rank q -> their natural positions
                rows = kv_all[q, b * twoC:(b + 1) * twoC]
                K[self.pos[q]] = rows[:, :ks]
                V[self.pos[q]] = rows[:, ks:]
            Q = np.zeros((self.S, self.hs))
            Q[self.pos[self.rank]] = self.q.numpy()[b * twoC:(b + 1) * twoC]
            Ob, _ = O.causal_attention(Q, K, V, self.heads // self.D, rows=self.pos[self.rank])
            O_local[b * twoC:(b + 1) * twoC] = Ob
        self.h.copy_(torch.from_numpy(resid.numpy() + O_local @ Wo))

    def mlp(self, shard, resid):
        self.seen_mlp.append(shard.clone())
        a = shard.numpy()
        n = 2 * self.fs * self.hid
        gu = a[:n].reshape(2 * self.fs, self.hid)
        Wd = a[n:].reshape(self.hid, self.fs).T
        Wg = np.concatenate([gu[q * 256:q * 256 + 128] for q in range(self.fs // 128)], axis=0).T
        Wu = np.concatenate([gu[q * 256 + 128:(q + 1) * 256] for q in range(self.fs // 128)], axis=0).T
        Hm = self.h.numpy()
        self.y.copy_(torch.from_numpy(resid.numpy() + (O.silu(Hm @ Wg) * (Hm @ Wu)) @ Wd))

"""Named TSP layer workloads.

Each is one transformer layer (causal MHA + SwiGLU MLP, no norm/bias/positions)
computed the TSP way over D virtual ranks.  Shapes follow the 7B dense decoder
the TSP announcement measures (hidden 4096, 32 heads of 128, MHA) plus one
tiny fp32 and one mid-size case.
"""

from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerConfig:
    name: str
    D: int
    batch: int
    seq: int
    hidden: int
    heads: int
    head_dim: int
    ffn: int
    dtype: str  # "f32" or "bf16"
    backward: bool = False
    kv_heads: int = 0  # K/V heads for grouped-query attention; 0: as many as query heads
    decode: bool = False  # one decode step per sequence against a cache of `seq` positions (last position)

    @property
    def chunk(self) -> int:
        return self.seq // (2 * self.D)

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def kv_h(self) -> int:
        """Number of K/V heads."""
        return self.kv_heads or self.heads

    @property
    def kv_hidden(self) -> int:
        """Width of K and V (K/V heads x head_dim)."""
        return self.kv_h * self.head_dim

    def decode_flops(self) -> int:
        """Algorithmic flops of one decode step at the last cache position: projections of
        B tokens plus attention of each new query over all S positions."""
        B, h, F, hk = self.batch, self.hidden, self.ffn, self.kv_hidden
        return B * 2 * (h * (h + 2 * hk) + h * h + 3 * h * F) + 4 * B * self.heads * self.head_dim * self.seq

    def decode_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode step: every weight once, the K/V cache rows
        read, the new K/V rows written, the tokens in and out (bf16)."""
        B, h, F, hk, S = self.batch, self.hidden, self.ffn, self.kv_hidden, self.seq
        weights = h * (h + 2 * hk) + h * h + 3 * h * F
        return 2 * (weights + 2 * B * S * hk + 2 * B * hk + 2 * B * h)

    def fwd_flops(self) -> int:
        """Algorithmic forward flops: B*S*2*(h*(h + 2hk) + h^2 + 3hF) + 4*B*H*dh*S(S+1)/2
        (Q/K/V, output and MLP projections, causal triangle only; hk = h for multi-head
        attention, which gives the familiar B*S*(8h^2 + 6hF))."""
        B, S, h, F, hk = self.batch, self.seq, self.hidden, self.ffn, self.kv_hidden
        return (B * S * 2 * (h * (h + 2 * hk) + h * h + 3 * h * F)
                + 4 * B * self.heads * self.head_dim * S * (S + 1) // 2)

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


TINY_F32 = LayerConfig("tiny_f32_D2_s256_h128", D=2, batch=1, seq=256, hidden=128, heads=4,
                       head_dim=32, ffn=512, dtype="f32")
MID_BF16 = LayerConfig("bf16_D4_s4096_h2048", D=4, batch=1, seq=4096, hidden=2048, heads=16,
                       head_dim=128, ffn=5632, dtype="bf16")
LAYER_7B_S16K = LayerConfig("bf16_D8_b2_s16384_h4096", D=8, batch=2, seq=16384, hidden=4096,
                            heads=32, head_dim=128, ffn=14336, dtype="bf16")
LAYER_7B_S64K = LayerConfig("bf16_D8_b1_s65536_h4096", D=8, batch=1, seq=65536, hidden=4096,
                            heads=32, head_dim=128, ffn=14336, dtype="bf16")
TRAIN_7B_S8K = LayerConfig("bf16_fwdbwd_D8_b1_s8192_h4096", D=8, batch=1, seq=8192, hidden=4096,
                           heads=32, head_dim=128, ffn=14336, dtype="bf16", backward=True)

# Backward at the 16K-token shape (training step, no optimizer).
TRAIN_7B_S16K = LayerConfig("bf16_fwdbwd_D8_b2_s16384_h4096", D=8, batch=2, seq=16384, hidden=4096, heads=32,
                            head_dim=128, ffn=14336, dtype="bf16", backward=True)

# Grouped-query attention: 8 K/V heads for the 32 query heads (one K/V head per rank at D = 8).
LAYER_7B_GQA8_S16K = LayerConfig("bf16_gqa8_D8_b2_s16384_h4096", D=8, batch=2, seq=16384, hidden=4096, heads=32,
                                 head_dim=128, ffn=14336, dtype="bf16", kv_heads=8)
TRAIN_7B_GQA8_S8K = LayerConfig("bf16_fwdbwd_gqa8_D8_b1_s8192_h4096", D=8, batch=1, seq=8192, hidden=4096,
                                heads=32, head_dim=128, ffn=14336, dtype="bf16", backward=True, kv_heads=8)

# Decoding at the pages' 128K context: one new token per sequence attends to a full cache.
DECODE_7B_128K = LayerConfig("bf16_decode_D8_b1_ctx131072_h4096", D=8, batch=1, seq=131072, hidden=4096, heads=32,
                             head_dim=128, ffn=14336, dtype="bf16", decode=True)
DECODE_7B_GQA8_128K = LayerConfig("bf16_decode_gqa8_D8_b4_ctx131072_h4096", D=8, batch=4, seq=131072, hidden=4096,
                                  heads=32, head_dim=128, ffn=14336, dtype="bf16", kv_heads=8, decode=True)

ALL = [TINY_F32, MID_BF16, LAYER_7B_S16K, LAYER_7B_S64K, TRAIN_7B_S8K, TRAIN_7B_S16K, LAYER_7B_GQA8_S16K,
       TRAIN_7B_GQA8_S8K, DECODE_7B_128K, DECODE_7B_GQA8_128K]
BY_NAME = {c.name: c for c in ALL}

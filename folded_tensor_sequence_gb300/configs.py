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

    @property
    def chunk(self) -> int:
        return self.seq // (2 * self.D)

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def fwd_flops(self) -> int:
        """Algorithmic forward flops: B*S*(8h^2 + 6hF) + 4*B*H*dh*S(S+1)/2 (causal triangle only)."""
        B, S, h, F = self.batch, self.seq, self.hidden, self.ffn
        return B * S * (8 * h * h + 6 * h * F) + 4 * B * self.heads * self.head_dim * S * (S + 1) // 2

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

ALL = [TINY_F32, MID_BF16, LAYER_7B_S16K, LAYER_7B_S64K, TRAIN_7B_S8K, TRAIN_7B_S16K]
BY_NAME = {c.name: c for c in ALL}

"""Named restore workloads: model shapes, request mixes and block layouts.

These are the shapes the HCache page ("Fast State Restoration in LLM Serving
with HCache", cue 4) evaluates on -- Llama2-7B, Llama2-13B and OPT-30B, all
plain multi-head attention -- plus a tiny shape for exhaustive checks and a
ragged multi-request batch whose lengths follow the page's workload
statistics (cue 10: short chat rounds, long documents above 16K tokens;
the CacheFlow page, cue 4: traces past 20,000 tokens).

Nothing here computes any part of the restoration method; this module only
names sizes, seeds and request layouts.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    norm: str = "rms"          # "rms" (RMSNorm, gamma) or "ln" (LayerNorm, gamma+beta)
    norm_eps: float = 1e-5
    rope: bool = True          # rotate-half RoPE on K
    rope_theta: float = 1e4
    dtype: str = "bf16"        # storage dtype of weights, hidden states and cache
    kv_bias: bool = False      # K/V projection bias (OPT)

    @property
    def d_kv(self) -> int:
        return self.n_kv_heads * self.head_dim


@dataclass(frozen=True)
class Workload:
    """One restore call's worth of synthetic input.

    seq_lens[r] tokens of request r are restored at absolute positions
    start_pos[r] .. start_pos[r]+seq_lens[r]-1.  Positions below start_pos[r]
    belong to a prefix that is already resident and must not be touched.
    """
    name: str
    shape: ModelShape
    seq_lens: Tuple[int, ...]
    start_pos: Tuple[int, ...]
    block_size: int = 16
    block_order: str = "contiguous"   # "contiguous" | "shuffled"
    spare_blocks: int = 0             # extra physical blocks nobody owns
    seed: int = 0
    max_position: int = 0             # RoPE table size; 0 -> derived
    description: str = ""
    # Hidden-state distribution.  Default: every element ~ N(0,1).  With
    # hidden_means, each token row gets a mean drawn (seeded, uniformly) from
    # this set and added to its N(0,1) draw; outlier_channels are scaled by
    # outlier_scale before the mean is added.  Large row means and a few
    # large channels are what real LayerNorm inputs (OPT) carry.
    hidden_means: Tuple[float, ...] = ()
    outlier_channels: Tuple[int, ...] = ()
    outlier_scale: float = 1.0

    @property
    def n_req(self) -> int:
        return len(self.seq_lens)

    @property
    def n_tokens(self) -> int:
        return int(sum(self.seq_lens))

    @property
    def rope_positions(self) -> int:
        if self.max_position:
            return self.max_position
        need = max((s + n for s, n in zip(self.start_pos, self.seq_lens)), default=1)
        return max(need, 1)


# ---------------------------------------------------------------------------
# Model shapes (HCache page, cue 4 names the three evaluated models)
# ---------------------------------------------------------------------------
TINY = ModelShape("tiny", n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64)
LLAMA2_7B = ModelShape("llama2-7b", n_layers=32, d_model=4096, n_heads=32, n_kv_heads=32,
                       head_dim=128)
LLAMA2_13B = ModelShape("llama2-13b", n_layers=40, d_model=5120, n_heads=40, n_kv_heads=40,
                        head_dim=128)
OPT_30B = ModelShape("opt-30b", n_layers=48, d_model=7168, n_heads=56, n_kv_heads=56,
                     head_dim=128, norm="ln", rope=False, dtype="fp16", kv_bias=True)


def _ragged_lengths(seed: int, n_req: int, lo: int, hi: int, start_hi: int):
    """Seeded uniform request lengths in [lo, hi] and starts in [0, start_hi]."""
    import numpy as np
    rng = np.random.Generator(np.random.PCG64(seed + 0x5EED))
    lens = rng.integers(lo, hi + 1, size=n_req)
    starts = rng.integers(0, start_hi + 1, size=n_req)
    return tuple(int(x) for x in lens), tuple(int(x) for x in starts)


def ragged_7b(seed: int = 0) -> Workload:
    lens, starts = _ragged_lengths(seed, 64, 256, 20000, 4096)
    return Workload("ragged-7b", LLAMA2_7B, lens, starts, block_order="shuffled", seed=seed,
                    description="64 requests, len ~U[256,20000], start ~U[0,4096], "
                                "permuted block table, Llama2-7B shape, all 32 layers")


WORKLOADS = {
    "tiny": Workload("tiny", TINY, (128,), (0,), spare_blocks=2,
                     description="2 layers, d=256, 4x64 heads, 128 tokens at pos 0"),
    "llama2-7b": Workload("llama2-7b", LLAMA2_7B, (4096,), (0,),
                          description="Llama2-7B shape, 1 request of 4096 tokens at pos 0, "
                                      "contiguous blocks"),
    "llama2-13b": Workload("llama2-13b", LLAMA2_13B, (16384,), (0,), block_order="shuffled",
                           description="Llama2-13B shape, 1 request of 16384 tokens at pos 0, "
                                       "shuffled physical block ids"),
    "opt-30b": Workload("opt-30b", OPT_30B, (8192,), (0,),
                        description="OPT-30B shape, fp16, LayerNorm+bias, no RoPE, 8192 tokens"),
}


SHAPES = {s.name: s for s in (TINY, LLAMA2_7B, LLAMA2_13B, OPT_30B)}


def get(name: str, **overrides) -> Workload:
    """A named workload; "<shape>-T<n>" is one request of n tokens at position 0."""
    if name == "ragged-7b":
        w = ragged_7b()
    elif name in WORKLOADS:
        w = WORKLOADS[name]
    elif "-T" in name and name.rsplit("-T", 1)[0] in SHAPES:
        base, n = name.rsplit("-T", 1)
        w = short_n(SHAPES[base], int(n))
    else:
        raise KeyError(name)
    return replace(w, **overrides) if overrides else w


def with_layers(w: Workload, n_layers: int) -> Workload:
    """The same workload on a model cut to its first n_layers layers."""
    return replace(w, name=f"{w.name}-L{n_layers}", shape=replace(w.shape, n_layers=n_layers))


def short_n(shape: ModelShape, n_tokens: int, seed: int = 0) -> Workload:
    """Weight-bound regime: one short request (HCache page cue 20: 794 tokens)."""
    return Workload(f"{shape.name}-T{n_tokens}", shape, (n_tokens,), (0,), seed=seed,
                    description=f"{shape.name} shape, 1 request of {n_tokens} tokens")

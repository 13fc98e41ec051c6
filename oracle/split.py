"""Oracle for the layer-split restore.  TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this module; the CUDA library shares no code with it.

What it computes (HCache episode, "Fast State Restoration for Evicted LLM KV
Caches"):
  * cue 18: transfer and computation of a restore form a pipeline and the
    slower one sets the pace; the bubble-free scheduler therefore splits the
    layers into two groups -- most restored from hidden states, the rest by a
    complementary method (token recompute or KV offload) -- with the group
    sizes found by a min-max optimisation over costs profiled offline;
  * cue 20: the split is by layer, so every layer's GEMM keeps all tokens.

Readings (listed in the design notes too):
  * the complementary method is KV offload: a layer's saved K and V rows are
    copied back and placed in the paged cache (token recompute needs the
    whole model and is not part of this library);
  * per-layer costs are constants: a hidden-state layer costs `hidden_copy`
    of transfer and `restore` of GPU time, a K/V layer `kv_copy` and
    `kv_place`; the pipeline's time for k K/V layers is
    max(total transfer, total compute) -- the steady-state bound, with no
    fill or drain term;
  * the hidden-state group is the lower layers, the K/V group the upper ones
    (the page does not say which; only the counts matter to the cost);
  * ties go to fewer K/V layers, which take more host memory per layer.

The K/V store layout is this library's: kv[layer][0 = K, 1 = V][token][row],
tokens in cu_seqlens order, row = n_kv_heads * head_dim values.

Pins (tests/test_oracle_split.py): a hand-worked split, the closed-form
crossing of the two linear totals, the regimes where one method wins
outright, and placement round trips against the restore oracle's placement.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Tuple

import numpy as np

from oracle import restore as R


@dataclass
class LayerCosts:
    restore: float       # GPU time, one layer from hidden states
    hidden_copy: float   # transfer time, one layer's hidden states
    kv_copy: float       # transfer time, one layer's K and V
    kv_place: float      # GPU time, placing one layer's K and V


@dataclass
class Split:
    hidden_layers: int
    kv_layers: int
    transfer: float
    compute: float
    predicted: float


def pipeline_totals(c: LayerCosts, n_layers: int, kv_layers: int) -> Tuple[float, float]:
    """Total transfer and total GPU time when kv_layers of n_layers are loaded as K/V."""
    hidden = n_layers - kv_layers
    transfer = hidden * c.hidden_copy + kv_layers * c.kv_copy
    compute = hidden * c.restore + kv_layers * c.kv_place
    return transfer, compute


def plan_layer_split(c: LayerCosts, n_layers: int) -> Split:
    """The split minimising max(transfer, compute) over kv_layers = 0..n_layers."""
    best = None
    for k in range(n_layers + 1):
        transfer, compute = pipeline_totals(c, n_layers, k)
        t = max(transfer, compute)
        if best is None or t < best.predicted:
            best = Split(n_layers - k, k, transfer, compute, t)
    return best


# ----------------------------------------------------------------------------- K/V rows
def kv_rows_from_cache(k_cache, v_cache, cu_seqlens, start_pos, block_table, block_size):
    """Dense [L][2][T][row] rows of the requests' tokens, read from caches laid out
    [L][num_blocks * block_size][row] (any dtype, e.g. raw bits)."""
    pl = R.token_placement(cu_seqlens, start_pos, block_table, block_size, None)
    k = np.asarray(k_cache)
    v = np.asarray(v_cache)
    return np.stack([k[:, pl.slot], v[:, pl.slot]], axis=1)


def kv_rows_to_cache(kv, k_cache, v_cache, cu_seqlens, start_pos, block_table, block_size):
    """Writes dense [L][2][T][row] rows into the caches' slots; other slots keep
    their contents.  Returns the updated caches."""
    pl = R.token_placement(cu_seqlens, start_pos, block_table, block_size, None)
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    kv = np.asarray(kv)
    for t in range(len(pl.slot)):
        k[:, pl.slot[t]] = kv[:, 0, t]
        v[:, pl.slot[t]] = kv[:, 1, t]
    return k, v

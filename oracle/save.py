"""Oracle for the save side of hidden-state restoration.  TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this module; the CUDA library shares no code with it.

What it computes (HCache episode, "Fast State Restoration for Evicted LLM KV
Caches"):
  * cue 16: hidden states are produced layer-before-token during generation
    (every layer's input for the step's token), but a restore wants all
    tokens of one layer together (token-before-layer);
  * cue 22: they are stored in fixed 64-token chunks, which also avoids
    fragmentation from unpredictable output lengths.

Readings (listed in the design notes too):
  * a chunk holds positions [64k, 64k+64) of one request (logical chunk
    k = pos // 64), all layers: element (layer l, position p, i) lives at
    chunk[id][l][p % 64][i] -- token-before-layer inside the chunk;
  * physical chunk ids come from a per-request chunk table, as KV blocks
    come from a block table; chunk_tokens is a parameter (64 on the page);
  * the rows to save are given like a restore's: tokens of the requests
    concatenated, request r's token i at position start_pos[r] + i, one
    [T][d] array per layer.  A decode step is the case of one token per
    request.

Pins (tests/test_oracle_save.py): a hand-worked layout, a brute force that
walks chunks instead of tokens, save/load round trips, and the identity
"saving a sequence token by token over decode steps = saving it at once".
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np


@dataclass
class ChunkPlacement:
    request: np.ndarray   # int64 [T]
    pos: np.ndarray       # int64 [T]
    chunk: np.ndarray     # int64 [T]: physical chunk id
    offset: np.ndarray    # int64 [T]: pos % chunk_tokens


def chunk_placement(cu_seqlens, start_pos, chunk_table, chunk_tokens: int,
                    num_chunks: Optional[int] = None) -> ChunkPlacement:
    """Token t = cu_seqlens[r] + i of request r at position start_pos[r] + i
    goes to chunk chunk_table[r][pos // C] at offset pos % C."""
    cu = np.asarray(cu_seqlens, np.int64)
    st = np.asarray(start_pos, np.int64)
    tab = np.asarray(chunk_table, np.int64)
    T = int(cu[-1])
    out = ChunkPlacement(*(np.empty(T, np.int64) for _ in range(4)))
    for r in range(len(st)):
        a, b = int(cu[r]), int(cu[r + 1])
        if b < a:
            raise ValueError("cu_seqlens must be non-decreasing")
        p = st[r] + np.arange(b - a, dtype=np.int64)
        logical = p // chunk_tokens
        if b > a and int(logical.max()) >= tab.shape[1]:
            raise ValueError(f"request {r}: position beyond its chunk table")
        ids = tab[r, logical]
        if b > a and (int(ids.min()) < 0 or (num_chunks is not None and
                                              int(ids.max()) >= num_chunks)):
            raise ValueError(f"request {r}: invalid chunk id")
        out.request[a:b] = r
        out.pos[a:b] = p
        out.chunk[a:b] = ids
        out.offset[a:b] = p % chunk_tokens
    return out


def save_chunks(hidden: Sequence[np.ndarray], layer_begin: int, n_layers: int,
                cu_seqlens, start_pos, chunk_table, chunk_tokens: int, num_chunks: int,
                buf: Optional[np.ndarray] = None) -> np.ndarray:
    """Write the rows of layers [layer_begin, layer_begin + len(hidden)) into a
    chunk store [num_chunks][n_layers][chunk_tokens][d] (NaN = never written).
    hidden[i] is layer layer_begin + i, shape [T][d]."""
    d = np.asarray(hidden[0]).shape[-1] if len(hidden) else 0
    if buf is None:
        buf = np.full((num_chunks, n_layers, chunk_tokens, d), np.nan)
    pl = chunk_placement(cu_seqlens, start_pos, chunk_table, chunk_tokens, num_chunks)
    for i, h in enumerate(hidden):
        buf[pl.chunk, layer_begin + i, pl.offset] = np.asarray(h, np.float64)
    return buf


def load_chunks(buf: np.ndarray, layer_begin: int, layer_end: int, cu_seqlens, start_pos,
                chunk_table, chunk_tokens: int) -> np.ndarray:
    """The inverse gather: rows [layer_end-layer_begin][T][d] in restore order."""
    pl = chunk_placement(cu_seqlens, start_pos, chunk_table, chunk_tokens, buf.shape[0])
    return np.stack([buf[pl.chunk, l, pl.offset] for l in range(layer_begin, layer_end)])

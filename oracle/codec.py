"""Oracle for the hidden-state codec.  TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this module; the CUDA library shares no code with it.

What it computes.  The HCache episode ("Fast State Restoration for Evicted LLM
KV Caches", cues 30 and 32) says hidden states could be quantised the way
CacheGen quantises KV caches.  CacheGen's encoder (CacheGen review, section
核心方法, the core method) has three steps; the first two are built here:
  * change-based encoding: tokens are cut into groups of 10 consecutive
    tokens; the first token of a group is its anchor and is kept at higher
    precision; every other token is kept as its difference from the anchor,
    so a group's tokens decode in parallel (no chain of deltas);
  * layer-wise quantisation: the layers are split into a first, middle and
    last group, whose deltas are quantised with bins of 0.5, 1 and 1.5 (the
    deeper, the coarser); anchors use 8-bit quantisation.
The third step, arithmetic coding with distributions profiled offline per
channel and layer, is lossless and is not built: it needs activation
statistics of a trained model.

Readings (listed in the design notes too):
  * groups are formed per request: token i of a request belongs to the group
    whose anchor is token 10 * (i // 10) of the same request; a request's last
    group may be shorter;
  * anchor quantisation is symmetric per row: scale s = max|h| / 127,
    code q = round(h * (1 / s)) in [-127, 127], value q * s; a row whose s is
    below the smallest normal binary32 number (max|h| < 127 * 2^-126) is
    coded as all zero with s = 0, so 1 / s is always finite;
  * a delta is taken from the anchor as the decoder will see it (q * s), so
    its error is the delta quantisation's alone: code
    c = round((h - q s) * (1 / b)) clamped to [-127, 127], value q s + c b;
  * quantising multiplies by the reciprocal of the step (1 / s once per
    anchor row, 1 / b once per layer), each reciprocal one binary32 division:
    the page gives the step sizes, not the arithmetic;
  * a bin b is in the hidden states' own units; layer l of L uses bin
    bins[min(2, 3 l // L)];
  * all arithmetic is IEEE binary32 with round-half-to-even for round(), the
    decoded value rounded once (to nearest even) to the storage type;
  * the encoded form is codes int8 [layer][token][d] (anchor codes on anchor
    rows, delta codes elsewhere) plus one float32 scale per anchor row, in
    a [layer][token] array (other entries unused).

Pins (tests/test_oracle_codec.py): a hand-worked group with exact binary
values, error bounds on random rows, lossless inputs, saturation, zero rows,
group boundaries by brute force, the layer-group rule by hand, and planted
mistakes.
"""
from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np

GROUP_TOKENS = 10
DEFAULT_BINS = (0.5, 1.0, 1.5)
F32 = np.float32


def layer_bin(layer: int, n_layers: int, bins: Sequence[float] = DEFAULT_BINS) -> np.float32:
    """The delta bin of layer `layer` (0-based) in a model of n_layers layers."""
    return F32(bins[min(2, (3 * layer) // n_layers)])


def group_anchors(cu_seqlens, group_tokens: int = GROUP_TOKENS) -> np.ndarray:
    """Anchor token (index into the concatenated tokens) of every token."""
    cu = np.asarray(cu_seqlens, np.int64)
    out = np.empty(int(cu[-1]), np.int64)
    for r in range(len(cu) - 1):
        i = np.arange(int(cu[r + 1] - cu[r]), dtype=np.int64)
        out[cu[r]:cu[r + 1]] = cu[r] + (i // group_tokens) * group_tokens
    return out


def rint32(x: np.ndarray) -> np.ndarray:
    """Round half to even, in float32."""
    return np.rint(np.asarray(x, F32)).astype(F32)


SMALLEST_NORMAL = F32(np.finfo(F32).tiny)   # 2^-126


def quantise_anchor(h: np.ndarray) -> Tuple[np.ndarray, np.float32]:
    """8-bit symmetric quantisation of one float32 row: (codes int8, scale)."""
    h = np.asarray(h, F32)
    m = F32(np.max(np.abs(h))) if h.size else F32(0)
    s = F32(m / F32(127))
    if s < SMALLEST_NORMAL:
        return np.zeros(h.shape, np.int8), F32(0)
    inv = F32(F32(1) / s)
    q = np.clip(rint32((h * inv).astype(F32)), -127, 127)
    return q.astype(np.int8), s


def dequantise_anchor(q: np.ndarray, s: np.float32) -> np.ndarray:
    return (np.asarray(q, F32) * F32(s)).astype(F32)


def encode_layer(h: np.ndarray, anchors: np.ndarray, b: np.float32):
    """h: float32 [T][d] -> (codes int8 [T][d], scales float32 [T])."""
    h = np.asarray(h, F32)
    T, d = h.shape
    codes = np.zeros((T, d), np.int8)
    scales = np.zeros(T, F32)
    for t in range(T):
        if anchors[t] == t:
            codes[t], scales[t] = quantise_anchor(h[t])
    for t in range(T):
        a = anchors[t]
        if a == t:
            continue
        a_hat = dequantise_anchor(codes[a], scales[a])
        delta = (h[t] - a_hat).astype(F32)
        inv_b = F32(F32(1) / F32(b))
        codes[t] = np.clip(rint32((delta * inv_b).astype(F32)), -127, 127).astype(np.int8)
    return codes, scales


def decode_layer(codes: np.ndarray, scales: np.ndarray, anchors: np.ndarray,
                 b: np.float32) -> np.ndarray:
    """(codes, scales) -> float32 [T][d], before rounding to the storage type."""
    codes = np.asarray(codes, np.int8)
    T, d = codes.shape
    out = np.empty((T, d), F32)
    for t in range(T):
        a = anchors[t]
        a_hat = dequantise_anchor(codes[a], scales[a])
        if a == t:
            out[t] = a_hat
        else:
            step = (codes[t].astype(F32) * F32(b)).astype(F32)
            out[t] = (a_hat + step).astype(F32)
    return out


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> storage bits (uint16), rounding to nearest even.  Finite inputs."""
    x = np.ascontiguousarray(x, F32)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        lsb = (u >> np.uint64(16)) & np.uint64(1)
        return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    raise ValueError(dtype)


def encode(hidden: Sequence[np.ndarray], layer_begin: int, n_layers: int, cu_seqlens,
           bins: Sequence[float] = DEFAULT_BINS, group_tokens: int = GROUP_TOKENS):
    """hidden[i]: float32 [T][d] of layer layer_begin + i -> (codes [Lr][T][d], scales [Lr][T])."""
    anchors = group_anchors(cu_seqlens, group_tokens)
    out = [encode_layer(h, anchors, layer_bin(layer_begin + i, n_layers, bins))
           for i, h in enumerate(hidden)]
    return np.stack([c for c, _ in out]), np.stack([s for _, s in out])


def decode(codes, scales, layer_begin: int, n_layers: int, cu_seqlens,
           bins: Sequence[float] = DEFAULT_BINS, group_tokens: int = GROUP_TOKENS):
    """-> float32 [Lr][T][d]."""
    anchors = group_anchors(cu_seqlens, group_tokens)
    return np.stack([decode_layer(codes[i], scales[i], anchors,
                                  layer_bin(layer_begin + i, n_layers, bins))
                     for i in range(len(codes))])

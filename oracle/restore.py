"""Oracle for HCache-style KV-cache restoration.  TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this module.  The CUDA library never calls it, and it shares no code,
table or constant with the library.

What it computes (HCache episode, "Fast State Restoration for Evicted LLM KV
Caches", cue 14): instead of keeping K and V, keep each layer's input hidden
state H and rebuild the cache by running only the projections, K = W_k H and
V = W_v H, skipping attention and the FFN.  Cue 3 fixes H as the layer input
(layer 1's is the embedding output); cue 4 fixes one K and one V vector per
head per token (multi-head attention); cue 16 fixes that a restore reads all
tokens of one layer together.

Readings where the pages are silent (each also listed in the design notes):
  * the projection consumes the layer's input norm of H (pre-norm models):
    RMSNorm with gamma, or LayerNorm with gamma and beta for OPT;
  * PyTorch Linear convention, W is [out, in], so K = X W^T;
  * RoPE rotate-half pairs (i, i + dh/2), angle = pos * theta^(-2i/dh),
    applied to K only, at 0-based absolute positions start + i;
  * RMSNorm: x = h / sqrt(mean(h^2) + eps) * gamma;  LayerNorm: biased
    variance, eps inside the square root;
  * the cache is paged: slot = block_table[r][pos // B] * B + pos % B, cache
    layout [layer][block][offset][kv_head][head_dim].

Everything is float64, on inputs widened exactly from their stored bf16/fp16
bits.  Parity status: every function here is pinned by the CPU tests in
tests/test_oracle_pins.py (closed forms, invariants, brute force, a full
random-init transformer forward).  Parity with real checkpoints is unpinned:
no trained weights are available, so the rotate-half pairing (versus the
interleaved one) is a reading, not a measured fact.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# Storage formats
# ---------------------------------------------------------------------------
def widen_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of bf16 or IEEE binary16 bit patterns (uint16).

    bf16 is the upper half of an IEEE binary32 word; binary16 is numpy's
    float16.  Both widen to float64 exactly.  fp16_from_fields decodes
    binary16 from its fields and pins this conversion in the tests.
    """
    b = np.asarray(bits).astype(np.uint16)
    with np.errstate(invalid="ignore"):   # signalling-NaN patterns widen to NaN
        if dtype == "bf16":
            return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        if dtype == "fp16":
            return b.view(np.float16).astype(np.float64)
    raise ValueError(dtype)


def fp16_from_fields(bits: np.ndarray) -> np.ndarray:
    """binary16 from its definition: 1 sign bit, 5 exponent bits (bias 15), 10
    fraction bits; exponent 0 encodes subnormals 2^-14 * f/1024, exponent 31
    encodes inf (f = 0) and NaN."""
    b = np.asarray(bits).astype(np.uint16)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = ((b >> 10) & 0x1F).astype(np.int64)
    f = (b & 0x3FF).astype(np.float64)
    val = np.where(e == 0, np.ldexp(f / 1024.0, -14), np.ldexp(1.0 + f / 1024.0, e - 15))
    val = np.where(e == 31, np.where(f == 0, np.inf, np.nan), val)
    return sign * val


# ---------------------------------------------------------------------------
# Input norm of the layer (reading: pre-norm; the pages write K = W_k H)
# ---------------------------------------------------------------------------
def rms_norm(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """x_i = h_i / sqrt((1/d) sum_j h_j^2 + eps) * gamma_i, over the last axis."""
    h = np.asarray(h, dtype=np.float64)
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return h / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def layer_norm(h: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    """x_i = (h_i - mu) / sqrt(var + eps) * gamma_i + beta_i, biased variance."""
    h = np.asarray(h, dtype=np.float64)
    mu = np.mean(h, axis=-1, keepdims=True)
    var = np.mean((h - mu) ** 2, axis=-1, keepdims=True)
    return (h - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


# ---------------------------------------------------------------------------
# The projection (HCache episode, cue 14: K = W_k H, V = W_v H)
# ---------------------------------------------------------------------------
def project(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray] = None) -> np.ndarray:
    """y = x W^T (+ b): x [T, d_in], W [d_out, d_in] -> y [T, d_out]."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)
    return y


# ---------------------------------------------------------------------------
# Rotary position embedding on K (reading: rotate-half pairs)
# ---------------------------------------------------------------------------
def rope_angles(pos: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """alpha[t, i] = pos[t] * theta^(-2i/dh) for i < dh/2, in float64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    omega = np.power(float(theta), -2.0 * i / head_dim)
    return np.asarray(pos, np.float64)[:, None] * omega[None, :]


def rope_rotate_half(k: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate each pair (k[i], k[i+dh/2]) of every head by alpha[t, i].

    k: [T, H, dh].  (a, b) -> (a cos(alpha) - b sin(alpha), b cos(alpha) + a sin(alpha)).
    """
    k = np.asarray(k, np.float64)
    dh = k.shape[-1]
    half = dh // 2
    alpha = rope_angles(pos, dh, theta)[:, None, :]      # [T, 1, half]
    c, s = np.cos(alpha), np.sin(alpha)
    a, b = k[..., :half], k[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# ---------------------------------------------------------------------------
# Paged placement (reading: vLLM-style block table)
# ---------------------------------------------------------------------------
@dataclass
class Placement:
    request: np.ndarray   # int64 [T]: request of each concatenated token
    pos: np.ndarray       # int64 [T]: absolute position
    slot: np.ndarray      # int64 [T]: block_id * B + pos % B


def token_placement(cu_seqlens, start_pos, block_table, block_size: int,
                    num_blocks: Optional[int] = None) -> Placement:
    """Token t = cu_seqlens[r] + i of request r sits at position start_pos[r] + i,
    in physical block block_table[r][pos // B] at offset pos % B."""
    cu = np.asarray(cu_seqlens, np.int64)
    st = np.asarray(start_pos, np.int64)
    bt = np.asarray(block_table, np.int64)
    T = int(cu[-1])
    req = np.empty(T, np.int64)
    pos = np.empty(T, np.int64)
    slot = np.empty(T, np.int64)
    for r in range(len(st)):
        n = int(cu[r + 1] - cu[r])
        if n < 0:
            raise ValueError("cu_seqlens must be non-decreasing")
        p = st[r] + np.arange(n, dtype=np.int64)
        logical = p // block_size
        if n and int(logical.max()) >= bt.shape[1]:
            raise ValueError(f"request {r}: position beyond its block table")
        blk = bt[r, logical]
        if n and (int(blk.min()) < 0 or (num_blocks is not None and int(blk.max()) >= num_blocks)):
            raise ValueError(f"request {r}: invalid physical block id")
        req[cu[r]:cu[r + 1]] = r
        pos[cu[r]:cu[r + 1]] = p
        slot[cu[r]:cu[r + 1]] = blk * block_size + p % block_size
    return Placement(req, pos, slot)


# ---------------------------------------------------------------------------
# One layer and a whole restore
# ---------------------------------------------------------------------------
@dataclass
class ModelSpec:
    d_model: int
    n_kv_heads: int
    head_dim: int
    norm: str = "rms"
    norm_eps: float = 1e-5
    rope: bool = True
    rope_theta: float = 1e4


@dataclass
class LayerWeights:
    """float64 copies of one layer's parameters."""
    gamma: np.ndarray
    w_k: np.ndarray
    w_v: np.ndarray
    beta: Optional[np.ndarray] = None
    b_k: Optional[np.ndarray] = None
    b_v: Optional[np.ndarray] = None


def restore_layer(h: np.ndarray, lw: LayerWeights, pos: np.ndarray, spec: ModelSpec):
    """K, V [T, H_kv, dh] of one layer from its saved input h [T, d]."""
    if spec.norm == "rms":
        x = rms_norm(h, lw.gamma, spec.norm_eps)
    elif spec.norm == "ln":
        x = layer_norm(h, lw.gamma, lw.beta, spec.norm_eps)
    else:
        raise ValueError(spec.norm)
    T = x.shape[0]
    k = project(x, lw.w_k, lw.b_k).reshape(T, spec.n_kv_heads, spec.head_dim)
    v = project(x, lw.w_v, lw.b_v).reshape(T, spec.n_kv_heads, spec.head_dim)
    if spec.rope:
        k = rope_rotate_half(k, pos, spec.rope_theta)
    return k, v


@dataclass
class OracleCache:
    """Restored caches [L][num_blocks*B][H_kv][dh] in float64; NaN = untouched."""
    k: np.ndarray
    v: np.ndarray
    placement: Placement

    def written_slots(self) -> np.ndarray:
        return self.placement.slot


def restore(hidden: Sequence[np.ndarray], weights: Sequence[LayerWeights], spec: ModelSpec,
            cu_seqlens, start_pos, block_table, block_size: int,
            num_blocks: int) -> OracleCache:
    """Restore every layer in `hidden` (one [T, d] array per layer) into paged caches."""
    pl = token_placement(cu_seqlens, start_pos, block_table, block_size, num_blocks)
    L = len(hidden)
    shape = (L, num_blocks * block_size, spec.n_kv_heads, spec.head_dim)
    kc = np.full(shape, np.nan)
    vc = np.full(shape, np.nan)
    for l in range(L):
        k, v = restore_layer(hidden[l], weights[l], pl.pos, spec)
        kc[l, pl.slot] = k
        vc[l, pl.slot] = v
    return OracleCache(kc, vc, pl)


def kv_bytes(n_layers: int, n_kv_heads: int, head_dim: int, n_tokens: int,
             elem_bytes: int) -> int:
    """Bytes of K plus V for n_tokens (CacheFlow episode, cue 4: 2*L*H*d*N elements)."""
    return 2 * n_layers * n_kv_heads * head_dim * n_tokens * elem_bytes

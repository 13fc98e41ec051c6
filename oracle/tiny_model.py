"""A tiny random-init decoder, run in float64.  TEST INFRASTRUCTURE ONLY.

It pins the restore oracle to something other than itself: a full forward
pass records each layer's input hidden state H_l (HCache episode, "Fast State
Restoration for Evicted LLM KV Caches", cue 3: a layer's hidden state is the
previous layer's output, the first one the embedding) together with the K and
V its attention actually used (cue 4).  Restoring from H_l must give back
exactly that K/V (cue 14), and decoding one more token from the restored,
paged cache must give the same logits as the full forward pass.

The forward pass is written independently of oracle.restore: it projects Q,
K and V with one fused [3*d_kv, d] matrix, applies RoPE as a complex
multiplication, and uses its own norms.  Two families:

  * "llama": RMSNorm, RoPE on Q and K, SwiGLU MLP, no biases;
  * "opt":   LayerNorm with gamma/beta, learned position embeddings added to
             the token embedding (so no RoPE), biases on every projection,
             ReLU MLP.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np


@dataclass
class TinyConfig:
    family: str = "llama"
    vocab: int = 97
    d_model: int = 64
    n_heads: int = 4
    n_kv_heads: int = 4
    head_dim: int = 16
    n_layers: int = 3
    d_ff: int = 96
    norm_eps: float = 1e-5
    rope_theta: float = 1e4
    max_pos: int = 256


@dataclass
class TinyLayer:
    norm1_g: np.ndarray
    norm1_b: Optional[np.ndarray]
    w_qkv: np.ndarray               # [(H + 2 H_kv) * dh, d]: rows Q, then K, then V
    b_qkv: Optional[np.ndarray]
    w_o: np.ndarray
    b_o: Optional[np.ndarray]
    norm2_g: np.ndarray
    norm2_b: Optional[np.ndarray]
    w_up: np.ndarray                # llama: [2*d_ff, d] (gate rows first); opt: [d_ff, d]
    b_up: Optional[np.ndarray]
    w_down: np.ndarray
    b_down: Optional[np.ndarray]

    # views used by the restore oracle
    def w_k(self, cfg: TinyConfig) -> np.ndarray:
        q = cfg.n_heads * cfg.head_dim
        return self.w_qkv[q:q + cfg.n_kv_heads * cfg.head_dim]

    def w_v(self, cfg: TinyConfig) -> np.ndarray:
        q = cfg.n_heads * cfg.head_dim
        kv = cfg.n_kv_heads * cfg.head_dim
        return self.w_qkv[q + kv:q + 2 * kv]

    def b_k(self, cfg: TinyConfig) -> Optional[np.ndarray]:
        if self.b_qkv is None:
            return None
        q = cfg.n_heads * cfg.head_dim
        return self.b_qkv[q:q + cfg.n_kv_heads * cfg.head_dim]

    def b_v(self, cfg: TinyConfig) -> Optional[np.ndarray]:
        if self.b_qkv is None:
            return None
        q = cfg.n_heads * cfg.head_dim
        kv = cfg.n_kv_heads * cfg.head_dim
        return self.b_qkv[q + kv:q + 2 * kv]


@dataclass
class TinyModel:
    cfg: TinyConfig
    embed: np.ndarray               # [vocab, d]
    pos_embed: Optional[np.ndarray] # [max_pos, d] (opt only)
    layers: List[TinyLayer]
    final_g: np.ndarray
    final_b: Optional[np.ndarray]
    lm_head: np.ndarray             # [vocab, d]


def random_model(cfg: TinyConfig, seed: int = 0) -> TinyModel:
    rng = np.random.Generator(np.random.PCG64(seed))
    d, dh = cfg.d_model, cfg.head_dim
    opt = cfg.family == "opt"

    def n(*shape, std=0.02, mean=0.0):
        return rng.normal(mean, std, size=shape)

    qkv_rows = (cfg.n_heads + 2 * cfg.n_kv_heads) * dh
    layers = []
    for _ in range(cfg.n_layers):
        layers.append(TinyLayer(
            norm1_g=n(d, std=0.1, mean=1.0), norm1_b=n(d) if opt else None,
            w_qkv=n(qkv_rows, d, std=0.2), b_qkv=n(qkv_rows) if opt else None,
            w_o=n(d, cfg.n_heads * dh, std=0.1), b_o=n(d) if opt else None,
            norm2_g=n(d, std=0.1, mean=1.0), norm2_b=n(d) if opt else None,
            w_up=n((cfg.d_ff if opt else 2 * cfg.d_ff), d, std=0.1),
            b_up=n(cfg.d_ff) if opt else None,
            w_down=n(d, cfg.d_ff, std=0.1), b_down=n(d) if opt else None,
        ))
    return TinyModel(cfg, embed=n(cfg.vocab, d, std=1.0),
                     pos_embed=n(cfg.max_pos, d, std=0.5) if opt else None,
                     layers=layers, final_g=n(d, std=0.1, mean=1.0),
                     final_b=n(d) if opt else None, lm_head=n(cfg.vocab, d, std=0.1))


# ---------------------------------------------------------------------------
# Building blocks, written for this forward pass only
# ---------------------------------------------------------------------------
def _norm(cfg: TinyConfig, x: np.ndarray, g: np.ndarray, b: Optional[np.ndarray]) -> np.ndarray:
    if cfg.family == "opt":
        c = x - x.mean(axis=-1, keepdims=True)
        return c / np.sqrt((c * c).mean(axis=-1, keepdims=True) + cfg.norm_eps) * g + b
    return x * (1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + cfg.norm_eps)) * g


def _rope_complex(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """x [T, H, dh]: pair (x[i], x[i+dh/2]) as the complex number x[i] + 1j*x[i+dh/2],
    multiplied by exp(1j * pos * theta^(-2i/dh))."""
    dh = x.shape[-1]
    half = dh // 2
    z = x[..., :half] + 1j * x[..., half:]
    freqs = theta ** (-(2.0 * np.arange(half)) / dh)
    z = z * np.exp(1j * np.outer(pos, freqs))[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1)


def _attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
            k_pos: np.ndarray, group: int) -> np.ndarray:
    """Causal softmax attention. q [Tq, H, dh]; k, v [Tk, H_kv, dh]."""
    dh = q.shape[-1]
    out = np.empty_like(q)
    for hq in range(q.shape[1]):
        hk = hq // group
        s = q[:, hq, :] @ k[:, hk, :].T / np.sqrt(dh)          # [Tq, Tk]
        s = np.where(k_pos[None, :] <= q_pos[:, None], s, -np.inf)
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=-1, keepdims=True)
        out[:, hq, :] = p @ v[:, hk, :]
    return out


def _mlp(cfg: TinyConfig, lay: TinyLayer, x: np.ndarray) -> np.ndarray:
    if cfg.family == "opt":
        u = np.maximum(x @ lay.w_up.T + lay.b_up, 0.0)
        return u @ lay.w_down.T + lay.b_down
    gu = x @ lay.w_up.T
    g, u = gu[:, :cfg.d_ff], gu[:, cfg.d_ff:]
    return (g / (1.0 + np.exp(-g)) * u) @ lay.w_down.T


def _qkv(cfg: TinyConfig, lay: TinyLayer, x: np.ndarray, pos: np.ndarray):
    T, dh = x.shape[0], cfg.head_dim
    y = x @ lay.w_qkv.T
    if lay.b_qkv is not None:
        y = y + lay.b_qkv
    nq, nkv = cfg.n_heads * dh, cfg.n_kv_heads * dh
    q = y[:, :nq].reshape(T, cfg.n_heads, dh)
    k = y[:, nq:nq + nkv].reshape(T, cfg.n_kv_heads, dh)
    v = y[:, nq + nkv:].reshape(T, cfg.n_kv_heads, dh)
    if cfg.family == "llama":
        q = _rope_complex(q, pos, cfg.rope_theta)
        k = _rope_complex(k, pos, cfg.rope_theta)
    return q, k, v


def _embed(m: TinyModel, tokens: np.ndarray, pos: np.ndarray) -> np.ndarray:
    h = m.embed[tokens]
    if m.pos_embed is not None:
        h = h + m.pos_embed[pos]
    return h


@dataclass
class ForwardRecord:
    logits: np.ndarray               # [T, vocab]
    hidden: List[np.ndarray]         # per layer: its input H_l [T, d]
    k: List[np.ndarray]              # per layer: K after RoPE [T, H_kv, dh]
    v: List[np.ndarray]              # per layer: V [T, H_kv, dh]


def forward(m: TinyModel, tokens: np.ndarray, start: int = 0) -> ForwardRecord:
    """Full causal forward over tokens at positions start .. start+T-1."""
    cfg = m.cfg
    T = len(tokens)
    pos = np.arange(start, start + T)
    h = _embed(m, np.asarray(tokens), pos)
    rec = ForwardRecord(None, [], [], [])
    group = cfg.n_heads // cfg.n_kv_heads
    for lay in m.layers:
        rec.hidden.append(h.copy())
        x = _norm(cfg, h, lay.norm1_g, lay.norm1_b)
        q, k, v = _qkv(cfg, lay, x, pos)
        rec.k.append(k)
        rec.v.append(v)
        a = _attend(q, k, v, pos, pos, group).reshape(T, -1)
        o = a @ lay.w_o.T
        if lay.b_o is not None:
            o = o + lay.b_o
        h = h + o
        h = h + _mlp(cfg, lay, _norm(cfg, h, lay.norm2_g, lay.norm2_b))
    rec.logits = _norm(cfg, h, m.final_g, m.final_b) @ m.lm_head.T
    return rec


def decode_from_paged_cache(m: TinyModel, token: int, pos: int, k_cache: np.ndarray,
                            v_cache: np.ndarray, block_table_row: np.ndarray,
                            block_size: int) -> np.ndarray:
    """Logits of one new token at `pos`, attending to positions 0..pos-1 read
    from paged caches k_cache/v_cache [L][num_blocks*B][H_kv][dh] through the
    request's block table, plus the new token's own K/V."""
    cfg = m.cfg
    past = np.arange(pos)
    slots = np.asarray(block_table_row)[past // block_size] * block_size + past % block_size
    p1 = np.array([pos])
    h = _embed(m, np.array([token]), p1)
    group = cfg.n_heads // cfg.n_kv_heads
    for l, lay in enumerate(m.layers):
        x = _norm(cfg, h, lay.norm1_g, lay.norm1_b)
        q, k_new, v_new = _qkv(cfg, lay, x, p1)
        k_all = np.concatenate([k_cache[l, slots], k_new], axis=0)
        v_all = np.concatenate([v_cache[l, slots], v_new], axis=0)
        kp = np.concatenate([past, p1])
        a = _attend(q, k_all, v_all, p1, kp, group).reshape(1, -1)
        o = a @ lay.w_o.T
        if lay.b_o is not None:
            o = o + lay.b_o
        h = h + o
        h = h + _mlp(cfg, lay, _norm(cfg, h, lay.norm2_g, lay.norm2_b))
    return (_norm(cfg, h, m.final_g, m.final_b) @ m.lm_head.T)[0]

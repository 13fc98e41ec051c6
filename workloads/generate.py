"""Seeded synthetic inputs for restore workloads.

Every tensor is drawn from its own torch generator whose seed is a fixed mix
of (workload seed, tensor tag, layer, chunk), so any one layer's parameters or
hidden states can be regenerated alone.  Values are drawn in fp32 and rounded
once (round-to-nearest-even) to the storage dtype; the CUDA library and the
oracle both consume those same stored bytes.

Distributions: hidden ~ N(0,1); W_k, W_v ~ N(0, 0.02) (0.02 is the standard
deviation); gamma ~ 1 + N(0, 0.1); beta, b_k, b_v ~ N(0, 0.02).

A generator is tied to a device type: torch's CPU and CUDA generators give
different streams for one seed.  A workload drawn on CUDA is therefore copied
to the host (where the oracle needs it), never redrawn there.

This module computes no part of the restoration method.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from .configs import ModelShape, Workload

TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16}

_TAGS = {"hidden": 1, "gamma": 2, "beta": 3, "w_k": 4, "w_v": 5, "b_k": 6, "b_v": 7,
         "blocks": 8, "row_mean": 9}

_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & _MASK64
    return x ^ (x >> 31)


def stream_seed(seed: int, tag: str, layer: int = 0, chunk: int = 0) -> int:
    """63-bit seed for one (tensor, layer, chunk) stream."""
    x = _splitmix64(seed & _MASK64)
    for part in (_TAGS[tag], layer, chunk):
        x = _splitmix64(x ^ (part & _MASK64))
    return x & ((1 << 63) - 1)


def normal(shape, mean: float, std: float, seed: int, device, dtype: torch.dtype,
           chunk_rows: int = 0, post=None) -> torch.Tensor:
    """N(mean, std^2) drawn in fp32 then rounded once to `dtype`.

    With chunk_rows > 0 the leading dimension is drawn in chunks of that many
    rows, each from its own stream, to bound the fp32 temporary.  `post`, if
    given, is called as post(x, r0, r1) on each fp32 chunk (rows r0..r1-1)
    before the rounding and may change it in place.
    """
    device = torch.device(device)
    out = torch.empty(shape, dtype=dtype, device=device)
    rows = shape[0] if len(shape) else 1
    step = chunk_rows if chunk_rows > 0 else max(rows, 1)
    for c, r0 in enumerate(range(0, rows, step)):
        r1 = min(rows, r0 + step)
        g = torch.Generator(device=device)
        g.manual_seed(_splitmix64(seed ^ c) & ((1 << 63) - 1) if chunk_rows > 0 else seed)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if mean != 0.0:
            x.add_(mean)
        if post is not None:
            post(x, r0, r1)
        out[r0:r1] = x.to(dtype)
    return out


@dataclass
class LayerParams:
    gamma: torch.Tensor             # [d]
    beta: Optional[torch.Tensor]    # [d] (LayerNorm only)
    w_k: torch.Tensor               # [d_kv, d]
    w_v: torch.Tensor               # [d_kv, d]
    b_k: Optional[torch.Tensor]     # [d_kv]
    b_v: Optional[torch.Tensor]     # [d_kv]


def layer_params(shape: ModelShape, layer: int, seed: int, device="cpu") -> LayerParams:
    dt = TORCH_DTYPE[shape.dtype]
    d, dkv = shape.d_model, shape.d_kv
    gamma = normal((d,), 1.0, 0.1, stream_seed(seed, "gamma", layer), device, dt)
    beta = (normal((d,), 0.0, 0.02, stream_seed(seed, "beta", layer), device, dt)
            if shape.norm == "ln" else None)
    w_k = normal((dkv, d), 0.0, 0.02, stream_seed(seed, "w_k", layer), device, dt)
    w_v = normal((dkv, d), 0.0, 0.02, stream_seed(seed, "w_v", layer), device, dt)
    b_k = (normal((dkv,), 0.0, 0.02, stream_seed(seed, "b_k", layer), device, dt)
           if shape.kv_bias else None)
    b_v = (normal((dkv,), 0.0, 0.02, stream_seed(seed, "b_v", layer), device, dt)
           if shape.kv_bias else None)
    return LayerParams(gamma, beta, w_k, w_v, b_k, b_v)


def hidden_row_means(w: Workload, layer: int) -> Optional[np.ndarray]:
    """The mean added to each token row of layer `layer`'s hidden states (a
    seeded uniform choice from w.hidden_means), or None for zero-mean rows."""
    if not w.hidden_means:
        return None
    rng = np.random.Generator(np.random.PCG64(stream_seed(w.seed, "row_mean", layer)))
    pick = rng.integers(0, len(w.hidden_means), size=w.n_tokens)
    return np.asarray(w.hidden_means, np.float32)[pick]


def hidden_states(w: Workload, layer: int, device="cpu", out: Optional[torch.Tensor] = None,
                  chunk_rows: int = 65536) -> torch.Tensor:
    """Saved layer input H_l [T, d] for the workload's concatenated tokens."""
    dt = TORCH_DTYPE[w.shape.dtype]
    post = None
    if w.hidden_means or w.outlier_channels:
        means = hidden_row_means(w, layer)
        row_mean = None if means is None else torch.as_tensor(means, device=device)
        cols = torch.as_tensor(list(w.outlier_channels), dtype=torch.long, device=device)

        def post(x, r0, r1):
            if len(w.outlier_channels):
                x[:, cols] *= w.outlier_scale
            if row_mean is not None:
                x.add_(row_mean[r0:r1, None])
    h = normal((w.n_tokens, w.shape.d_model), 0.0, 1.0,
               stream_seed(w.seed, "hidden", layer), device, dt, chunk_rows=chunk_rows,
               post=post)
    if out is not None:
        out.copy_(h)
        return out
    return h


@dataclass
class RequestLayout:
    cu_seqlens: np.ndarray      # int32 [R+1]
    start_pos: np.ndarray       # int32 [R]
    block_table: np.ndarray     # int32 [R, max_blocks]; -1 past a request's last block
    num_blocks: int             # physical blocks in the cache
    max_blocks: int             # columns of block_table
    block_size: int


def request_layout(w: Workload) -> RequestLayout:
    """Per-request token ranges and a block table covering [0, start+len).

    Logical block i of request r holds positions [i*B, (i+1)*B).  Physical
    ids are handed out in request order ("contiguous") or from a seeded
    permutation of all ids ("shuffled").  spare_blocks extra physical blocks
    belong to no request.
    """
    B = w.block_size
    lens = np.asarray(w.seq_lens, dtype=np.int64)
    starts = np.asarray(w.start_pos, dtype=np.int64)
    cu = np.zeros(len(lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    need = [(int(s) + int(n) + B - 1) // B for s, n in zip(starts, lens)]
    total = int(sum(need))
    num_blocks = total + w.spare_blocks
    ids = np.arange(num_blocks, dtype=np.int64)
    if w.block_order == "shuffled":
        rng = np.random.Generator(np.random.PCG64(stream_seed(w.seed, "blocks")))
        ids = rng.permutation(num_blocks)
    elif w.block_order != "contiguous":
        raise ValueError(w.block_order)
    max_blocks = max(need) if need else 1
    max_blocks = max(max_blocks, 1)
    table = np.full((len(lens), max_blocks), -1, dtype=np.int64)
    k = 0
    for r, nb in enumerate(need):
        table[r, :nb] = ids[k:k + nb]
        k += nb
    return RequestLayout(cu.astype(np.int32), starts.astype(np.int32),
                         table.astype(np.int32), num_blocks, max_blocks, B)


SENTINEL_BITS = 0x7FA5   # a NaN payload: the restore computation never produces it


def sentinel_cache(n_layers: int, num_blocks: int, block_size: int, n_kv_heads: int,
                   head_dim: int, dtype: str, device) -> torch.Tensor:
    """Paged cache [L][num_blocks][B][H_kv][dh] with every element = SENTINEL_BITS."""
    t = torch.empty((n_layers, num_blocks, block_size, n_kv_heads, head_dim),
                    dtype=torch.int16, device=device)
    t.fill_(SENTINEL_BITS)
    return t.view(TORCH_DTYPE[dtype])


@dataclass
class DeviceInputs:
    """Everything one restore call reads or writes, resident on a device."""
    params: list                 # LayerParams per model layer
    layout: RequestLayout
    hidden: torch.Tensor         # [Lr][T][d] for layers [layer_begin, layer_end)
    k_cache: torch.Tensor        # [Lr][num_blocks][B][H_kv][dh], sentinel-filled
    v_cache: torch.Tensor
    cu: torch.Tensor             # int32 [R+1]
    start: torch.Tensor          # int32 [R]
    table: torch.Tensor          # int32 [R][max_blocks]


def device_inputs(w: Workload, device, layer_begin: int = 0, layer_end: Optional[int] = None,
                  params: Optional[list] = None, gen_device=None) -> DeviceInputs:
    """Seeded inputs for layers [layer_begin, layer_end) of workload w on `device`.

    Random tensors are drawn on gen_device (default: the CPU for small
    workloads, `device` for large ones) and copied; hidden layer i is drawn
    from the stream of absolute layer layer_begin + i, so splitting a layer
    range gives the same inputs.
    """
    s = w.shape
    layer_end = s.n_layers if layer_end is None else layer_end
    if gen_device is None:
        big = w.n_tokens * s.d_model * (layer_end - layer_begin) > (1 << 26)
        gen_device = device if big else "cpu"
    if params is None:
        params = []
        for l in range(s.n_layers):
            p = layer_params(s, l, w.seed, gen_device)
            params.append(LayerParams(*[None if t is None else t.to(device) for t in
                                        (p.gamma, p.beta, p.w_k, p.w_v, p.b_k, p.b_v)]))
    lay = request_layout(w)
    Lr = layer_end - layer_begin
    hidden = torch.empty((Lr, w.n_tokens, s.d_model), dtype=TORCH_DTYPE[s.dtype], device=device)
    for i in range(Lr):
        hidden[i].copy_(hidden_states(w, layer_begin + i, gen_device))
    kc = sentinel_cache(Lr, lay.num_blocks, w.block_size, s.n_kv_heads, s.head_dim, s.dtype,
                        device)
    vc = sentinel_cache(Lr, lay.num_blocks, w.block_size, s.n_kv_heads, s.head_dim, s.dtype,
                        device)

    def to(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return DeviceInputs(params, lay, hidden, kc, vc, to(lay.cu_seqlens), to(lay.start_pos),
                        to(lay.block_table))

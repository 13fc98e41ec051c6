"""Shared test plumbing: build a workload's inputs, run the CUDA restore through
the C ABI, and compare the paged caches with the oracle.

Tolerance (the floating-point bar for bf16/fp16 storage with fp32
accumulation: 2e-2 absolute and 1e-2 relative, read elementwise): a restored value
g passes against the oracle's float64 value o when
    |g - o| <= max(2e-2, 1e-2 * |o|),
i.e. 2e-2 absolute for |o| <= 2 and 1% relative above.  bf16 storage alone
rounds by up to 2^-9 |o| (half an ulp), which this bound covers with room
for fp32 accumulation and the once-rounded gamma-folded weights.
Placement is bit-exact: every restored row must sit in the oracle's slot and
every other cache element must still hold the sentinel bit pattern.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import List, Optional, Sequence

import numpy as np
import torch

from oracle import restore as R
from workloads import generate as G
from workloads.configs import ModelShape, Workload

ATOL = 2e-2
RTOL = 1e-2


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def widen(t: torch.Tensor, dtype: str) -> np.ndarray:
    return R.widen_bits(bits_of(t), dtype)


def dims_for(w: Workload):
    from kv_cache_restoration_gb300 import make_dims
    s = w.shape
    return make_dims(s.n_layers, s.d_model, s.n_heads, s.n_kv_heads, s.head_dim, s.norm,
                     s.norm_eps, s.rope, s.rope_theta, w.rope_positions, s.dtype, s.kv_bias)


def spec_for(s: ModelShape) -> R.ModelSpec:
    return R.ModelSpec(d_model=s.d_model, n_kv_heads=s.n_kv_heads, head_dim=s.head_dim,
                       norm=s.norm, norm_eps=s.norm_eps, rope=s.rope, rope_theta=s.rope_theta)


def oracle_weights(p: G.LayerParams, dtype: str) -> R.LayerWeights:
    f = lambda t: None if t is None else widen(t, dtype)  # noqa: E731
    return R.LayerWeights(gamma=f(p.gamma), w_k=f(p.w_k), w_v=f(p.w_v), beta=f(p.beta),
                          b_k=f(p.b_k), b_v=f(p.b_v))


@dataclass
class Case:
    w: Workload
    layer_begin: int
    layer_end: int
    params: List[G.LayerParams]
    layout: G.RequestLayout
    hidden: torch.Tensor          # [Lr][T][d]
    k_cache: torch.Tensor         # [Lr][num_blocks][B][H][dh]
    v_cache: torch.Tensor
    cu: torch.Tensor
    start: torch.Tensor
    table: torch.Tensor
    restorer: object = None
    status: int = 0
    flags: int = 0


def make_case(w: Workload, device, layer_begin: int = 0, layer_end: Optional[int] = None,
              params: Optional[List[G.LayerParams]] = None, restorer=None,
              gen_device=None) -> Case:
    """Seeded inputs on `device` plus a Restorer (a new one unless given)."""
    s = w.shape
    layer_end = s.n_layers if layer_end is None else layer_end
    d = G.device_inputs(w, device, layer_begin, layer_end, params=params, gen_device=gen_device)
    case = Case(w, layer_begin, layer_end, d.params, d.layout, d.hidden, d.k_cache, d.v_cache,
                d.cu, d.start, d.table)
    if restorer is None:
        from kv_cache_restoration_gb300 import Restorer
        restorer = Restorer(dims_for(w), d.params)
    case.restorer = restorer
    return case


def run(case: Case, stream=None, check: bool = True) -> Case:
    lay = case.layout
    case.restorer.restore(case.hidden, case.layer_begin, case.layer_end, case.cu, case.start,
                          case.table, case.k_cache, case.v_cache, lay.num_blocks,
                          lay.block_size, stream=stream, check=check)
    case.status, case.flags = case.restorer.check(stream)
    return case


def _assert_close(g: np.ndarray, o: np.ndarray, what: str):
    assert g.shape == o.shape, (what, g.shape, o.shape)
    err = np.abs(g - o)
    tol = np.maximum(ATOL, RTOL * np.abs(o))
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
            f"first {idx.tolist()}: got {g[bad][:5]}, want {o[bad][:5]}")


@dataclass
class Report:
    rows_checked: int = 0
    max_abs_small: float = 0.0   # max |g-o| over |o| < 1
    max_rel_large: float = 0.0   # max |g-o|/|o| over |o| >= 1


def compare(case: Case, rows: Optional[np.ndarray] = None,
            layers: Optional[Sequence[int]] = None, check_sentinel: bool = True) -> Report:
    """Oracle check of restored rows (all, or the given token indices) in the
    given absolute layers (default all in range), plus the sentinel check."""
    w, s = case.w, case.w.shape
    lay = case.layout
    pl = R.token_placement(lay.cu_seqlens, lay.start_pos, lay.block_table, lay.block_size,
                           lay.num_blocks)
    T = w.n_tokens
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    layers = range(case.layer_begin, case.layer_end) if layers is None else layers
    spec = spec_for(s)
    rep = Report()
    H, dh = s.n_kv_heads, s.head_dim
    for l in layers:
        li = l - case.layer_begin
        lw = oracle_weights(case.params[l], s.dtype)
        h = widen(case.hidden[li][torch.as_tensor(rows, device=case.hidden.device)], s.dtype)
        ok, ov = R.restore_layer(h, lw, pl.pos[rows], spec)
        slots = torch.as_tensor(pl.slot[rows], device=case.k_cache.device)
        gk = widen(case.k_cache[li].reshape(-1, H, dh)[slots], s.dtype)
        gv = widen(case.v_cache[li].reshape(-1, H, dh)[slots], s.dtype)
        _assert_close(gk, ok, f"K layer {l}")
        _assert_close(gv, ov, f"V layer {l}")
        for g, o in ((gk, ok), (gv, ov)):
            small = np.abs(o) < 1
            if small.any():
                rep.max_abs_small = max(rep.max_abs_small, float(np.abs(g - o)[small].max()))
            if (~small).any():
                rep.max_rel_large = max(rep.max_rel_large,
                                        float((np.abs(g - o) / np.abs(o))[~small].max()))
        rep.rows_checked += len(rows)
    if check_sentinel:
        check_sentinels(case, pl.slot)
    return rep


def check_sentinels(case: Case, written_slots: np.ndarray):
    """Every slot no restored token maps to keeps the sentinel, bit for bit, in
    every layer of both caches, and every restored slot was written (checked
    on the device one layer at a time, counted on the host)."""
    nslots = case.layout.num_blocks * case.layout.block_size
    mask = torch.ones(nslots, dtype=torch.bool, device=case.k_cache.device)
    if len(written_slots):
        mask[torch.as_tensor(written_slots, device=mask.device)] = False
    for c, name in ((case.k_cache, "K"), (case.v_cache, "V")):
        for li in range(c.shape[0]):
            bits = c[li].view(torch.int16).reshape(nslots, -1)
            n_bad = int((bits[mask] != G.SENTINEL_BITS).sum().item())
            assert n_bad == 0, f"{name} cache layer {li}: {n_bad} elements of unwritten slots changed"
            n_sent = int((bits[~mask] == G.SENTINEL_BITS).sum().item())
            assert n_sent == 0, f"{name} cache layer {li}: {n_sent} restored elements not written"


def sample_rows(w: Workload, fraction: float, seed: int = 1) -> np.ndarray:
    """A seeded sample of token rows plus every request's first and last row."""
    T = w.n_tokens
    rng = np.random.Generator(np.random.PCG64(seed))
    n = max(64, int(T * fraction))
    rows = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    cu = np.concatenate([[0], np.cumsum(w.seq_lens)])
    for r in range(w.n_req):
        if cu[r + 1] > cu[r]:
            rows.update((int(cu[r]), int(cu[r + 1] - 1)))
    return np.array(sorted(rows), dtype=np.int64)

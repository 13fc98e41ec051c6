"""Each plausible mistake planted in the oracle (on the CPU) trips a pin.

The mistakes are planted by monkeypatching oracle.restore; composite
functions look their helpers up at call time, so the planted helper is used
throughout the restore.
"""
import json
import os

import numpy as np
import pytest

from oracle import restore as R
from tests import pins

ORIG = {name: getattr(R, name) for name in
        ("rms_norm", "layer_norm", "project", "rope_rotate_half", "rope_angles",
         "token_placement", "restore_layer")}


def _rope_sign_flipped(k, pos, theta):
    return ORIG["rope_rotate_half"](k, -np.asarray(pos), theta)


def _rope_interleaved(k, pos, theta):
    k = np.asarray(k, np.float64)
    dh = k.shape[-1]
    alpha = ORIG["rope_angles"](pos, dh, theta)[:, None, :]
    a, b = k[..., 0::2], k[..., 1::2]
    out = np.empty_like(k)
    out[..., 0::2] = a * np.cos(alpha) - b * np.sin(alpha)
    out[..., 1::2] = b * np.cos(alpha) + a * np.sin(alpha)
    return out


def _angles_wrong_exponent(pos, head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.asarray(pos, np.float64)[:, None] * np.power(theta, -i / head_dim)[None, :]


def _rms_eps_outside(h, gamma, eps):
    h = np.asarray(h, np.float64)
    return h / (np.sqrt(np.mean(h * h, axis=-1, keepdims=True)) + eps) * gamma


def _rms_no_gamma(h, gamma, eps):
    return ORIG["rms_norm"](h, np.ones_like(np.asarray(gamma, np.float64)), eps)


def _ln_unbiased(h, gamma, beta, eps):
    h = np.asarray(h, np.float64)
    mu = h.mean(axis=-1, keepdims=True)
    var = ((h - mu) ** 2).sum(axis=-1, keepdims=True) / (h.shape[-1] - 1)
    return (h - mu) / np.sqrt(var + eps) * gamma + beta


def _ln_no_beta(h, gamma, beta, eps):
    return ORIG["layer_norm"](h, gamma, np.zeros_like(np.asarray(beta, np.float64)), eps)


def _project_transposed(x, w, b=None):
    w = np.asarray(w, np.float64)
    if w.shape[0] == w.shape[1]:
        y = np.asarray(x, np.float64) @ w
    else:   # keep shapes valid: transpose within the leading square block
        n = min(w.shape)
        w2 = w.copy()
        w2[:n, :n] = w[:n, :n].T
        y = np.asarray(x, np.float64) @ w2.T
    return y if b is None else y + b


def _project_no_bias(x, w, b=None):
    return ORIG["project"](x, w, None)


def _restore_layer_swapped(h, lw, pos, spec):
    lw2 = R.LayerWeights(gamma=lw.gamma, beta=lw.beta, w_k=lw.w_v, w_v=lw.w_k, b_k=lw.b_v,
                         b_v=lw.b_k)
    return ORIG["restore_layer"](h, lw2, pos, spec)


def _restore_layer_pos_off_by_one(h, lw, pos, spec):
    return ORIG["restore_layer"](h, lw, np.asarray(pos) + 1, spec)


def _restore_layer_rope_on_v(h, lw, pos, spec):
    k, v = ORIG["restore_layer"](h, lw, pos, spec)
    if spec.rope:
        v = ORIG["rope_rotate_half"](v, pos, spec.rope_theta)
    return k, v


def _placement_offset_from_start(cu_seqlens, start_pos, block_table, block_size, num_blocks=None):
    # mistake: offset within the block taken from the token index, not the position
    pl = ORIG["token_placement"](cu_seqlens, start_pos, block_table, block_size, num_blocks)
    cu = np.asarray(cu_seqlens)
    idx = pl.pos - np.asarray(start_pos)[pl.request]
    pl.slot = (pl.slot // block_size) * block_size + idx % block_size
    return pl


def _placement_block_from_index(cu_seqlens, start_pos, block_table, block_size, num_blocks=None):
    # mistake: logical block from the token index within the request, ignoring start
    pl = ORIG["token_placement"](cu_seqlens, start_pos, block_table, block_size, num_blocks)
    bt = np.asarray(block_table)
    idx = pl.pos - np.asarray(start_pos)[pl.request]
    pl.slot = bt[pl.request, idx // block_size] * block_size + pl.pos % block_size
    return pl


def _facts():
    with open(os.path.join(os.path.dirname(__file__), "golden", "kv_capacity_a100.json")) as f:
        return json.load(f)


def _all_pins():
    yield pins.pin_rms_constant, (R,)
    yield pins.pin_rms_values, (R,)
    yield pins.pin_layer_norm, (R,)
    yield pins.pin_project_bruteforce, (R,)
    yield pins.pin_rope_closed_form, (R,)
    yield pins.pin_rope_invariants, (R,)
    yield pins.pin_placement, (R,)
    yield pins.pin_identity_weights, (R,)
    yield pins.pin_tiny_forward, (R, "llama")
    yield pins.pin_tiny_forward, (R, "opt")


MUTANTS = [
    ("rope_rotate_half", _rope_sign_flipped),
    ("rope_rotate_half", _rope_interleaved),
    ("rope_angles", _angles_wrong_exponent),
    ("rms_norm", _rms_eps_outside),
    ("rms_norm", _rms_no_gamma),
    ("layer_norm", _ln_unbiased),
    ("layer_norm", _ln_no_beta),
    ("project", _project_transposed),
    ("project", _project_no_bias),
    ("restore_layer", _restore_layer_swapped),
    ("restore_layer", _restore_layer_pos_off_by_one),
    ("restore_layer", _restore_layer_rope_on_v),
    ("token_placement", _placement_offset_from_start),
    ("token_placement", _placement_block_from_index),
]


@pytest.mark.parametrize("attr,mutant", MUTANTS, ids=[m.__name__.strip("_") for _, m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, attr, mutant):
    monkeypatch.setattr(R, attr, mutant)
    failed = []
    for pin, args in _all_pins():
        try:
            pin(*args)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant.__name__}"


def test_unmutated_oracle_passes_every_pin():
    for pin, args in _all_pins():
        pin(*args)
    pins.pin_kv_bytes(R, _facts())


# ----------------------------------------------------------------------------- save side
from oracle import save as S  # noqa: E402
from tests import test_oracle_save as TS  # noqa: E402

SAVE_ORIG = S.chunk_placement


def _offset_from_index(cu_seqlens, start_pos, chunk_table, chunk_tokens, num_chunks=None):
    pl = SAVE_ORIG(cu_seqlens, start_pos, chunk_table, chunk_tokens, num_chunks)
    idx = pl.pos - np.asarray(start_pos)[pl.request]
    pl.offset = idx % chunk_tokens
    return pl


def _chunk_from_index(cu_seqlens, start_pos, chunk_table, chunk_tokens, num_chunks=None):
    pl = SAVE_ORIG(cu_seqlens, start_pos, chunk_table, chunk_tokens, num_chunks)
    idx = pl.pos - np.asarray(start_pos)[pl.request]
    pl.chunk = np.asarray(chunk_table)[pl.request, idx // chunk_tokens]
    return pl


def _save_layer_inner(hidden, layer_begin, n_layers, cu_seqlens, start_pos, chunk_table,
                      chunk_tokens, num_chunks, buf=None):
    # mistake: token-major inside the chunk ([C][L][d]) written into the [L][C][d] store
    d = np.asarray(hidden[0]).shape[-1]
    if buf is None:
        buf = np.full((num_chunks, n_layers, chunk_tokens, d), np.nan)
    pl = SAVE_ORIG(cu_seqlens, start_pos, chunk_table, chunk_tokens, num_chunks)
    flat = buf.reshape(num_chunks, -1, d)
    for i, h in enumerate(hidden):
        flat[pl.chunk, pl.offset * n_layers + layer_begin + i] = h
    return buf


SAVE_PINS = [TS.test_hand_worked_layout, lambda: TS.test_against_chunk_walk(4),
             TS.test_round_trip_and_layer_ranges, TS.test_decode_steps_equal_one_save]


@pytest.mark.parametrize("attr,mutant", [("chunk_placement", _offset_from_index),
                                         ("chunk_placement", _chunk_from_index),
                                         ("save_chunks", _save_layer_inner)],
                         ids=["offset_from_index", "chunk_from_index", "token_major_chunk"])
def test_planted_save_mistake_is_caught(monkeypatch, attr, mutant):
    monkeypatch.setattr(S, attr, mutant)
    failed = 0
    for pin in SAVE_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed, f"no pin caught {mutant.__name__}"


# ----------------------------------------------------------------------------- layer split
from oracle import split as SP  # noqa: E402
from tests import test_oracle_split as TSP  # noqa: E402

SPLIT_ORIG = {"pipeline_totals": SP.pipeline_totals, "plan_layer_split": SP.plan_layer_split,
              "kv_rows_from_cache": SP.kv_rows_from_cache}


def _totals_copies_swapped(c, n_layers, kv_layers):
    return SPLIT_ORIG["pipeline_totals"](
        SP.LayerCosts(c.restore, c.kv_copy, c.hidden_copy, c.kv_place), n_layers, kv_layers)


def _totals_place_as_restore(c, n_layers, kv_layers):
    return SPLIT_ORIG["pipeline_totals"](
        SP.LayerCosts(c.restore, c.hidden_copy, c.kv_copy, c.restore), n_layers, kv_layers)


def _plan_min_of_totals(c, n_layers):
    best = None
    for k in range(n_layers + 1):
        tr, co = SP.pipeline_totals(c, n_layers, k)
        t = min(tr, co)
        if best is None or t < best.predicted:
            best = SP.Split(n_layers - k, k, tr, co, t)
    return best


def _plan_never_all_kv(c, n_layers):
    best = None
    for k in range(max(n_layers, 1)):
        tr, co = SP.pipeline_totals(c, n_layers, k)
        t = max(tr, co)
        if best is None or t < best.predicted:
            best = SP.Split(n_layers - k, k, tr, co, t)
    return best


def _rows_k_v_swapped(k_cache, v_cache, *a):
    return SPLIT_ORIG["kv_rows_from_cache"](v_cache, k_cache, *a)


SPLIT_PINS = [TSP.test_hand_worked_split, lambda: TSP.test_crossing_point_closed_form(3),
              TSP.test_transfer_bound_keeps_every_layer_on_hidden_states,
              TSP.test_cheaper_kv_everywhere_loads_every_layer,
              TSP.test_ties_keep_fewer_kv_layers_and_empty_model,
              TSP.test_kv_rows_round_trip_and_untouched_slots]


@pytest.mark.parametrize("attr,mutant", [("pipeline_totals", _totals_copies_swapped),
                                         ("pipeline_totals", _totals_place_as_restore),
                                         ("plan_layer_split", _plan_min_of_totals),
                                         ("plan_layer_split", _plan_never_all_kv),
                                         ("kv_rows_from_cache", _rows_k_v_swapped)],
                         ids=["copies_swapped", "place_as_restore", "min_of_totals",
                              "never_all_kv", "rows_k_v_swapped"])
def test_planted_split_mistake_is_caught(monkeypatch, attr, mutant):
    monkeypatch.setattr(SP, attr, mutant)
    failed = 0
    for pin in SPLIT_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed, f"no pin caught {mutant.__name__}"


# ----------------------------------------------------------------------------- codec
from oracle import codec as CK  # noqa: E402
from tests import test_oracle_codec as TCK  # noqa: E402

CODEC_ORIG = {n: getattr(CK, n) for n in ("encode_layer", "group_anchors", "layer_bin",
                                          "quantise_anchor", "rint32", "decode_layer")}


def _encode_open_loop(h, anchors, b):
    # mistake: delta from the original anchor row, not the decoded one
    codes, scales = CODEC_ORIG["encode_layer"](h, anchors, b)
    h = np.asarray(h, np.float32)
    for t in range(len(h)):
        if anchors[t] != t:
            d = (h[t] - h[anchors[t]]).astype(np.float32)
            codes[t] = np.clip(np.rint(d / np.float32(b)), -127, 127).astype(np.int8)
    return codes, scales


def _encode_chained(h, anchors, b):
    # mistake: each delta from the previous token's decoded row
    codes, scales = CODEC_ORIG["encode_layer"](h, anchors, b)
    h = np.asarray(h, np.float32)
    prev = None
    for t in range(len(h)):
        if anchors[t] == t:
            prev = CK.dequantise_anchor(codes[t], scales[t])
            continue
        d = (h[t] - prev).astype(np.float32)
        codes[t] = np.clip(np.rint(d / np.float32(b)), -127, 127).astype(np.int8)
        prev = (prev + codes[t].astype(np.float32) * np.float32(b)).astype(np.float32)
    return codes, scales


def _anchors_ignore_requests(cu_seqlens, group_tokens=10):
    T = int(np.asarray(cu_seqlens)[-1])
    return (np.arange(T) // group_tokens) * group_tokens


def _bins_reversed(layer, n_layers, bins=CK.DEFAULT_BINS):
    return np.float32(bins[2 - min(2, (3 * layer) // n_layers)])


def _bins_by_thirds_rounded(layer, n_layers, bins=CK.DEFAULT_BINS):
    return np.float32(bins[min(2, round(3 * layer / n_layers))])


def _anchor_255(h):
    h = np.asarray(h, np.float32)
    m = np.float32(np.max(np.abs(h)))
    s = np.float32(m / np.float32(255))
    if s == 0:
        return np.zeros(h.shape, np.int8), np.float32(0)
    return np.clip(np.rint(h / s), -127, 127).astype(np.int8), s


def _round_half_away(x):
    x = np.asarray(x, np.float32)
    return (np.sign(x) * np.floor(np.abs(x) + np.float32(0.5))).astype(np.float32)


def _decode_plain_code(codes, scales, anchors, b):
    # mistake: a delta row decodes to c * b without the anchor
    out = CODEC_ORIG["decode_layer"](codes, scales, anchors, b)
    for t in range(len(out)):
        if anchors[t] != t:
            out[t] = codes[t].astype(np.float32) * np.float32(b)
    return out


CODEC_PINS = [TCK.test_hand_worked_group, TCK.test_group_boundaries_by_request,
              lambda: TCK.test_group_anchors_brute_force(1), TCK.test_layer_group_rule_by_hand,
              lambda: TCK.test_error_bounds(0.5), TCK.test_lossless_when_values_sit_on_the_grids,
              TCK.test_saturation_and_zero_rows, TCK.test_groups_decode_independently,
              TCK.test_multi_layer_encode_uses_each_layers_bin]


@pytest.mark.parametrize("attr,mutant", [("encode_layer", _encode_open_loop),
                                         ("encode_layer", _encode_chained),
                                         ("group_anchors", _anchors_ignore_requests),
                                         ("layer_bin", _bins_reversed),
                                         ("layer_bin", _bins_by_thirds_rounded),
                                         ("quantise_anchor", _anchor_255),
                                         ("rint32", _round_half_away),
                                         ("decode_layer", _decode_plain_code)],
                         ids=["open_loop", "chained", "groups_cross_requests", "bins_reversed",
                              "bins_rounded", "anchor_255", "round_half_away",
                              "decode_without_anchor"])
def test_planted_codec_mistake_is_caught(monkeypatch, attr, mutant):
    monkeypatch.setattr(CK, attr, mutant)
    failed = 0
    for pin in CODEC_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed, f"no pin caught {mutant.__name__}"

"""Pins for the layer-split oracle (oracle/split.py) and the C planner against it.

The planner's cost model is two linear totals in k, the number of layers
loaded as K/V:
    transfer(k) = (L - k) * h + k * kc,   compute(k) = (L - k) * r + k * p.
When the hidden-state restore is compute-bound (r > h), K/V transfer is
dearer than hidden-state transfer (kc > h) and K/V placement cheaper than a
restore (p < r), transfer rises and compute falls with k, so max() is
smallest where they cross:
    k* = L (r - h) / ((kc - h) + (r - p)),
and the integer optimum is floor(k*) or ceil(k*).
"""
import math
import random

import numpy as np
import pytest

from oracle import restore as R
from oracle import split as SP


def test_hand_worked_split():
    # r = 1.1, h = 0.8, kc = 1.6, p = 0.1 (ms), L = 40.  By hand:
    #   k = 6: transfer 34*0.8 + 6*1.6 = 36.8, compute 34*1.1 + 6*0.1 = 38.0 -> 38.0
    #   k = 7: transfer 33*0.8 + 7*1.6 = 37.6, compute 33*1.1 + 7*0.1 = 37.0 -> 37.6
    #   k = 8: transfer 32*0.8 + 8*1.6 = 38.4, compute 32*1.1 + 8*0.1 = 36.0 -> 38.4
    s = SP.plan_layer_split(SP.LayerCosts(1.1, 0.8, 1.6, 0.1), 40)
    assert (s.hidden_layers, s.kv_layers) == (33, 7)
    assert s.transfer == pytest.approx(37.6) and s.compute == pytest.approx(37.0)
    assert s.predicted == pytest.approx(37.6)


def _random_compute_bound(rng):
    h = rng.uniform(0.1, 1.0)
    r = h * rng.uniform(1.05, 3.0)
    kc = h * rng.uniform(1.05, 4.0)
    p = r * rng.uniform(0.0, 0.5)
    return SP.LayerCosts(r, h, kc, p)


@pytest.mark.parametrize("seed", range(40))
def test_crossing_point_closed_form(seed):
    rng = random.Random(seed)
    c = _random_compute_bound(rng)
    L = rng.randint(1, 96)
    s = SP.plan_layer_split(c, L)
    k_star = L * (c.restore - c.hidden_copy) / ((c.kv_copy - c.hidden_copy) + (c.restore - c.kv_place))
    candidates = {min(L, max(0, math.floor(k_star))), min(L, max(0, math.ceil(k_star)))}
    assert s.kv_layers in candidates
    best = min(max(*SP.pipeline_totals(c, L, k)) for k in candidates)
    assert s.predicted == pytest.approx(best)
    # at the crossing both totals equal the continuous optimum; the integer
    # optimum cannot beat it
    t_star = (L - k_star) * c.hidden_copy + k_star * c.kv_copy
    assert s.predicted >= t_star - 1e-12
    assert s.hidden_layers + s.kv_layers == L


def test_transfer_bound_keeps_every_layer_on_hidden_states():
    # hidden-state transfer already dominates and K/V transfer is dearer:
    # loading K/V only lengthens the critical resource.
    s = SP.plan_layer_split(SP.LayerCosts(0.5, 0.8, 1.6, 0.05), 32)
    assert (s.hidden_layers, s.kv_layers) == (32, 0)
    assert s.predicted == pytest.approx(32 * 0.8)


def test_cheaper_kv_everywhere_loads_every_layer():
    # a model whose K/V are smaller than its hidden states (few KV heads) and
    # whose placement is cheaper than a restore: K/V wins on both resources.
    s = SP.plan_layer_split(SP.LayerCosts(1.0, 0.8, 0.4, 0.1), 24)
    assert (s.hidden_layers, s.kv_layers) == (0, 24)
    assert s.predicted == pytest.approx(24 * 0.4)


def test_ties_keep_fewer_kv_layers_and_empty_model():
    s = SP.plan_layer_split(SP.LayerCosts(1.0, 1.0, 1.0, 1.0), 10)
    assert s.kv_layers == 0
    s0 = SP.plan_layer_split(SP.LayerCosts(1.0, 0.5, 2.0, 0.1), 0)
    assert (s0.hidden_layers, s0.kv_layers, s0.predicted) == (0, 0, 0.0)


def test_every_split_is_no_better_than_the_plan():
    rng = random.Random(7)
    for _ in range(50):
        c = SP.LayerCosts(*(rng.uniform(0.0, 2.0) for _ in range(4)))
        L = rng.randint(0, 60)
        s = SP.plan_layer_split(c, L)
        for k in range(L + 1):
            assert max(*SP.pipeline_totals(c, L, k)) >= s.predicted


def _layout():
    cu = np.array([0, 3, 3, 10])
    start = np.array([5, 0, 5])
    table = np.array([[4, 1, 0], [2, 0, 0], [6, 3, 5]])
    return cu, start, table


def test_kv_rows_round_trip_and_untouched_slots():
    cu, start, table = _layout()
    B, L, row = 4, 2, 3
    rng = np.random.default_rng(0)
    kc = rng.integers(0, 1 << 15, (L, 7 * B, row))
    vc = rng.integers(0, 1 << 15, (L, 7 * B, row))
    dense = SP.kv_rows_from_cache(kc, vc, cu, start, table, B)
    assert dense.shape == (L, 2, 10, row)
    # by hand: request 0's token 1 sits at position 6 -> block table[0][1] = 1, offset 2;
    # request 2's token 3 (t = 6) at position 8 -> block table[2][2] = 5, offset 0
    assert np.array_equal(dense[:, 0, 1], kc[:, 1 * B + 2])
    assert np.array_equal(dense[:, 1, 6], vc[:, 5 * B + 0])
    blank_k = np.full_like(kc, -1)
    blank_v = np.full_like(vc, -1)
    k2, v2 = SP.kv_rows_to_cache(dense, blank_k, blank_v, cu, start, table, B)
    slots = R.token_placement(cu, start, table, B).slot
    assert np.array_equal(k2[:, slots], kc[:, slots])
    assert np.array_equal(v2[:, slots], vc[:, slots])
    others = np.setdiff1d(np.arange(7 * B), slots)
    assert (k2[:, others] == -1).all() and (v2[:, others] == -1).all()


# ----------------------------------------------------------------------------- C planner
def _c_plan(c, L):
    from kv_cache_restoration_gb300 import binding as B
    return B.hcr_plan_layer_split(B.hcr_layer_costs(c.restore, c.hidden_copy, c.kv_copy,
                                                    c.kv_place), L)


def test_c_planner_matches_oracle():
    """hcr_plan_layer_split is host-only: it runs here without a GPU."""
    rng = random.Random(11)
    cases = [(SP.LayerCosts(1.1, 0.8, 1.6, 0.1), 40), (SP.LayerCosts(1.0, 1.0, 1.0, 1.0), 10)]
    cases += [(SP.LayerCosts(*(rng.uniform(0.0, 2.0) for _ in range(4))), rng.randint(0, 80))
              for _ in range(200)]
    cases += [(_random_compute_bound(rng), rng.randint(1, 96)) for _ in range(100)]
    for c, L in cases:
        want = SP.plan_layer_split(c, L)
        got = _c_plan(c, L)
        assert (got.hidden_layers, got.kv_layers) == (want.hidden_layers, want.kv_layers)
        assert got.predicted_s == pytest.approx(want.predicted, rel=1e-12, abs=0)
        assert got.transfer_s == pytest.approx(want.transfer, rel=1e-12, abs=0)
        assert got.compute_s == pytest.approx(want.compute, rel=1e-12, abs=0)


@pytest.mark.parametrize("bad", [(-1.0, 1, 1, 1), (1, float("nan"), 1, 1), (1, 1, float("inf"), 1)])
def test_c_planner_rejects_bad_costs(bad):
    from kv_cache_restoration_gb300 import binding as B
    with pytest.raises(B.HcrError) as e:
        B.hcr_plan_layer_split(B.hcr_layer_costs(*bad), 8)
    assert e.value.status == B.HCR_ERR_INVALID_ARG
    with pytest.raises(B.HcrError):
        B.hcr_plan_layer_split(B.hcr_layer_costs(1, 1, 1, 1), -1)


@pytest.mark.parametrize("seed", range(20))
def test_meet_in_the_middle_closed_form(seed):
    """CacheFlow episode, cue 12: with one method costing only compute (r per
    layer) and the other only transfer (kc per layer), splitting so both
    finish together takes L * r * kc / (r + kc) -- the product over the sum
    of the two per-layer costs.  The planner reduces to that case when the
    hidden-state transfer and the K/V placement cost nothing; the integer
    split is within one layer's cost of it and never below it."""
    rng = random.Random(100 + seed)
    r, kc = rng.uniform(0.1, 3.0), rng.uniform(0.1, 3.0)
    L = rng.randint(1, 120)
    s = SP.plan_layer_split(SP.LayerCosts(r, 0.0, kc, 0.0), L)
    t_star = L * r * kc / (r + kc)
    assert t_star - 1e-12 <= s.predicted <= t_star + max(r, kc)
    # and the split itself sits where the two totals cross
    assert abs(s.kv_layers - L * r / (r + kc)) <= 1

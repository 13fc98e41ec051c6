"""Seeded synthetic inputs (CPU): the hidden-state distribution options, and
the oracle's LayerNorm on rows with large means."""
from dataclasses import replace

import numpy as np
import torch

from oracle import restore as R
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

SHAPE = ModelShape("gen", 1, 512, 4, 4, 128, norm="ln", dtype="fp16")


def _f64(t):
    return t.float().double().numpy()


def test_default_rows_are_standard_normal_draws():
    """Without the options, hidden states are the plain N(0,1) stream of the
    workload seed (the options leave existing workloads unchanged)."""
    w = Workload("g", SHAPE, (300,), (0,))
    h = G.hidden_states(w, 0, "cpu")
    again = G.normal((300, 512), 0.0, 1.0, G.stream_seed(0, "hidden", 0), "cpu",
                     torch.float16, chunk_rows=65536)
    assert torch.equal(h.view(torch.int16), again.view(torch.int16))
    assert G.hidden_row_means(w, 0) is None


def test_row_means_and_outlier_channels():
    means = (-50.0, 10.0, 100.0)
    w = Workload("g", SHAPE, (3000,), (0,), hidden_means=means, outlier_channels=(0, 7),
                 outlier_scale=50.0)
    base = _f64(G.hidden_states(replace(w, hidden_means=(), outlier_channels=()), 0, "cpu"))
    h = _f64(G.hidden_states(w, 0, "cpu"))
    mu = G.hidden_row_means(w, 0)
    assert set(np.unique(mu).tolist()) == set(means)
    # every value occurs in roughly a third of the rows
    for m in means:
        assert 0.25 < np.mean(mu == m) < 0.42
    # the same N(0,1) draw underneath: ordinary channels are base + mean,
    # outlier channels 50 * base + mean (each rounded once to fp16)
    ordinary = np.setdiff1d(np.arange(512), [0, 7])
    want = (base[:, ordinary] + mu[:, None]).astype(np.float16).astype(np.float64)
    assert np.max(np.abs(h[:, ordinary] - want)) <= 0.0625   # one fp16 ulp at |x| < 128
    spread = h[:, [0, 7]] - mu[:, None]
    assert 35 < spread.std() < 65
    # row means differ per layer
    assert not np.array_equal(G.hidden_row_means(w, 1), mu)


def test_oracle_layer_norm_ignores_a_constant_shift():
    """LayerNorm is invariant under adding a constant to every element of a
    row, up to rounding of the shifted input: LN(h + c) = LN(h)."""
    rng = np.random.default_rng(5)
    h = rng.standard_normal((16, 512))
    gamma = 1 + 0.1 * rng.standard_normal(512)
    beta = 0.02 * rng.standard_normal(512)
    ref = R.layer_norm(h, gamma, beta, 1e-5)
    for c in (-50.0, 10.0, 100.0, 1e4):
        got = R.layer_norm(h + c, gamma, beta, 1e-5)
        assert np.max(np.abs(got - ref)) < 1e-9 * max(1.0, abs(c))


def test_large_mean_workloads_keep_their_placement():
    """The distribution options change values only: the request layout is
    the same."""
    w = C.get("tiny")
    a = G.request_layout(w)
    b = G.request_layout(replace(w, hidden_means=(100.0,), outlier_channels=(0,),
                                 outlier_scale=50.0))
    assert np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.cu_seqlens, b.cu_seqlens)

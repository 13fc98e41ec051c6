"""The restore's host-side choices without a GPU (hcr_debug_plan): the tile
variant of every measured shape on a GB300's unit counts (152 SMs, 76
co-resident CTA pairs), and when the norm statistics move into the
projection."""
import pytest

SMS, PAIRS = 152, 76
BIG = 1 << 40          # a workspace with room for the statistics flags
SINGLE, PAIR, ROWS = 1, 2, 3


@pytest.fixture(scope="module")
def plan():
    from kv_cache_restoration_gb300 import binding as B, make_dims
    from workloads.configs import LLAMA2_7B, LLAMA2_13B, OPT_30B

    def dims(shape):
        return make_dims(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                         shape.head_dim, shape.norm, shape.norm_eps, shape.rope,
                         shape.rope_theta, 32768, shape.dtype, shape.kv_bias)

    shapes = {"7b": dims(LLAMA2_7B), "13b": dims(LLAMA2_13B), "opt": dims(OPT_30B)}

    def f(model, tokens, layers, ws=BIG, sms=SMS, pairs=PAIRS, swap=PAIRS):
        return B.hcr_debug_plan(shapes[model], tokens, layers, sms, pairs, swap, ws)
    return f


@pytest.mark.parametrize("tokens,layers,want", [
    (16, 32, SINGLE), (64, 32, SINGLE), (128, 32, SINGLE),   # one 128-row tile
    (129, 32, PAIR), (256, 32, PAIR),
    (257, 32, ROWS), (300, 32, ROWS), (320, 32, ROWS),       # weight rows as M
    (321, 32, PAIR), (794, 32, PAIR), (1100, 32, PAIR), (4096, 32, PAIR),
    (16384, 32, SINGLE),                                     # 35 TFLOP: above 32
    (629259, 8, SINGLE),                                     # the ragged batch's windows
])
def test_llama2_7b_variants(plan, tokens, layers, want):
    assert plan("7b", tokens, layers)[0] == want


@pytest.mark.parametrize("model,tokens,layers,want", [
    ("13b", 256, 40, PAIR), ("13b", 400, 40, PAIR), ("13b", 512, 40, PAIR),
    ("13b", 1024, 40, PAIR), ("13b", 1536, 40, PAIR),        # <= 6.5 TFLOP, no half tail
    ("13b", 300, 40, ROWS),
    ("13b", 384, 40, SINGLE), ("13b", 513, 40, SINGLE),      # a half tail tile
    ("13b", 2048, 40, SINGLE), ("13b", 16384, 40, SINGLE),   # 8.6 / 68.7 TFLOP
    ("opt", 256, 48, PAIR), ("opt", 512, 48, PAIR),
    ("opt", 300, 48, ROWS),
    ("opt", 384, 48, SINGLE), ("opt", 640, 48, SINGLE), ("opt", 794, 48, SINGLE),
    ("opt", 768, 48, SINGLE), ("opt", 8192, 48, SINGLE),     # 7.6 / 80.8 TFLOP
])
def test_wide_model_variants(plan, model, tokens, layers, want):
    assert plan(model, tokens, layers)[0] == want


def test_without_pairs_or_weight_rows(plan):
    # no co-resident pairs: single CTAs everywhere, the weight rows need pairs too
    for t in (256, 300, 4096):
        assert plan("7b", t, 32, pairs=0, swap=0)[0] == SINGLE
    # pairs but no weight-row kernel: 300 tokens fall back to the token-row rules
    assert plan("7b", 300, 32, swap=0)[0] in (SINGLE, PAIR)


@pytest.mark.parametrize("model,tokens,layers,layer0", [
    ("7b", 1100, 32, 2),     # pairs: 5 m-tiles x 32 n-tiles; three rounds of 76 reach 2 layers
    ("7b", 794, 32, 2),
    ("7b", 2048, 32, 1),
    ("7b", 64, 32, 15),      # single CTAs: one m-tile; three rounds of 152 reach 15 layers
    ("13b", 256, 40, 6),     # pairs: 1 m-tile x 40 n-tiles; three rounds of 76 reach 6 layers
])
def test_fused_statistics_layers(plan, model, tokens, layers, layer0):
    assert plan(model, tokens, layers)[1] == layer0
    # without room for the flags the prepare kernel computes every layer
    assert plan(model, tokens, layers, ws=0)[1] == 0


@pytest.mark.parametrize("model,tokens,layers", [
    ("7b", 4096, 32),        # 16 m-tiles: the projection runs at its ingress limit
    ("7b", 300, 32),         # weight-row tiles keep the prepare pass
    ("7b", 1100, 2),         # the prepare kernel's first layers cover the call
    ("7b", 1100, 1),
    ("13b", 16384, 40),
])
def test_statistics_stay_in_prepare(plan, model, tokens, layers):
    assert plan(model, tokens, layers)[1] == 0


def test_rejects_null_arguments():
    from kv_cache_restoration_gb300 import binding as B
    assert B.lib.hcr_debug_plan(None, 300, 32, SMS, PAIRS, PAIRS, BIG, None) == 1

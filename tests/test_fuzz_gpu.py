"""Seeded random configurations against the oracle, every element and every
slot (GPU).

Each case draws a model shape (width, head size, grouped-query ratio, norm,
RoPE, storage type, biases), a batch of requests (count, lengths including
empty ones, start positions, block size, block order, spare blocks) and a
tile variant, then checks the restore in full: every restored value within
the tolerance and every other cache element still the sentinel.
"""
import random

import pytest

from tests import harness as Hn
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

VARIANTS = (0, 1, 2, 3)   # automatic, single CTAs, CTA pairs, weight-row CTA pairs


def _case(seed: int):
    rng = random.Random(9000 + seed)
    head_dim = rng.choice((64, 128, 256))
    n_kv = rng.choice((1, 2, 3, 4))
    group = rng.choice((1, 1, 2, 4))
    d_model = 8 * rng.randint(8, 96)                 # 64 .. 768, any multiple of 8
    norm = rng.choice(("rms", "ln"))
    shape = ModelShape(f"fz{seed}", rng.randint(1, 3), d_model, n_kv * group, n_kv, head_dim,
                       norm=norm, rope=rng.random() < 0.7, rope_theta=rng.choice((1e4, 5e5)),
                       dtype=rng.choice(("bf16", "fp16")), kv_bias=rng.random() < 0.4)
    n_req = rng.randint(1, 10)
    lens = tuple(rng.choice((0, 1, rng.randint(2, 40), rng.randint(41, 400)))
                 for _ in range(n_req))
    if sum(lens) == 0:
        lens = (rng.randint(1, 50),) + lens[1:]
    starts = tuple(rng.randint(0, 1500) for _ in range(n_req))
    w = Workload(f"fuzz{seed}", shape, lens, starts, block_size=rng.choice((1, 8, 16, 32, 64)),
                 block_order=rng.choice(("contiguous", "shuffled")),
                 spare_blocks=rng.randint(0, 4), seed=seed)
    variant = VARIANTS[seed % 4]
    if variant >= 3 and head_dim != 128:     # weight-row tiles need 128-wide heads
        variant = 0
    return w, variant


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration_matches_oracle(cuda_device, seed):
    from kv_cache_restoration_gb300 import binding as B
    w, variant = _case(seed)
    case = Hn.make_case(w, cuda_device)
    assert B.hcr_debug_set_variant(case.restorer.handle, variant) == 0
    Hn.run(case)
    assert case.status == 0, (case.status, case.flags, w)
    Hn.compare(case)

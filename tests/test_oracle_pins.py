"""The oracle against what the pages and the mathematics fix (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import restore as R
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_widen_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = R.widen_bits(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_widen_fp16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = R.widen_bits(bits, "fp16")
    want = R.fp16_from_fields(bits)          # decoded from the binary16 fields
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    # and the field decoding agrees with torch's half conversion
    want = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_rms_constant_vector():
    pins.pin_rms_constant(R)


def test_rms_values():
    pins.pin_rms_values(R)


def test_layer_norm():
    pins.pin_layer_norm(R)


def test_project_bruteforce():
    pins.pin_project_bruteforce(R)


def test_rope_closed_form():
    pins.pin_rope_closed_form(R)


def test_rope_invariants():
    pins.pin_rope_invariants(R)


def test_placement():
    pins.pin_placement(R)


def test_placement_rejects_bad_tables():
    with pytest.raises(ValueError):
        R.token_placement([0, 3], [0], [[5]], 2, num_blocks=4)      # block id 5 >= 4
    with pytest.raises(ValueError):
        R.token_placement([0, 3], [0], [[0]], 2, num_blocks=4)      # position 2 has no block
    with pytest.raises(ValueError):
        R.token_placement([0, 3], [0], [[-1, 1]], 2, num_blocks=4)  # negative id


def test_identity_weights():
    pins.pin_identity_weights(R)


@pytest.mark.parametrize("family", ["llama", "opt"])
def test_tiny_forward_roundtrip(family):
    pins.pin_tiny_forward(R, family)


def test_tiny_forward_roundtrip_gqa():
    pins.pin_tiny_forward(R, "llama", n_kv_heads=2)


def test_kv_bytes_capacity_facts():
    with open(os.path.join(GOLDEN, "kv_capacity_a100.json")) as f:
        facts = json.load(f)
    pins.pin_kv_bytes(R, facts)

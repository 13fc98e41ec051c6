"""Pins for the hidden-state codec oracle (oracle/codec.py)."""
import numpy as np
import pytest

from oracle import codec as K

F32 = np.float32


def test_hand_worked_group():
    # Anchor max 127/64 gives scale exactly 1/64, so the anchor codes are
    # h * 64 exactly: [127, -64, 32, 2].  Second row = anchor + [0.5, -1.0,
    # 0.25, 0.75] with bin 0.5: codes round(delta / 0.5) = [1, -2, round(0.5),
    # round(1.5)] = [1, -2, 0, 2] (half to even), decoded deltas [0.5, -1.0,
    # 0.0, 1.0].
    anchor = np.array([127 / 64, -1.0, 0.5, 0.03125], F32)
    row2 = anchor + np.array([0.5, -1.0, 0.25, 0.75], F32)
    h = np.stack([anchor, row2])
    anchors = K.group_anchors([0, 2])
    codes, scales = K.encode_layer(h, anchors, F32(0.5))
    assert scales[0] == F32(1 / 64)
    assert codes[0].tolist() == [127, -64, 32, 2]
    assert codes[1].tolist() == [1, -2, 0, 2]
    dec = K.decode_layer(codes, scales, anchors, F32(0.5))
    assert np.array_equal(dec[0], anchor)
    assert np.array_equal(dec[1], anchor + np.array([0.5, -1.0, 0.0, 1.0], F32))


def test_group_boundaries_by_request():
    # lengths 13, 0, 3, 25 -> anchors at request starts and every 10th token
    cu = [0, 13, 13, 16, 41]
    a = K.group_anchors(cu)
    want = [0] * 10 + [10] * 3 + [13] * 3 + [16] * 10 + [26] * 10 + [36] * 5
    assert a.tolist() == want


@pytest.mark.parametrize("seed", range(5))
def test_group_anchors_brute_force(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 40, 12)
    cu = np.concatenate([[0], np.cumsum(lens)])
    g = int(rng.integers(1, 12))
    a = K.group_anchors(cu, g)
    # walk each request token by token, starting a new group every g tokens
    t = 0
    for n in lens:
        anchor = None
        for i in range(n):
            if i % g == 0:
                anchor = t
            assert a[t] == anchor
            t += 1


def test_layer_group_rule_by_hand():
    bins = [K.layer_bin(l, 32) for l in range(32)]
    assert bins[:11] == [F32(0.5)] * 11 and bins[11:22] == [F32(1.0)] * 11
    assert bins[22:] == [F32(1.5)] * 10
    b40 = [K.layer_bin(l, 40) for l in range(40)]
    assert b40.index(F32(1.0)) == 14 and b40.index(F32(1.5)) == 27
    assert K.layer_bin(0, 1) == F32(0.5) and K.layer_bin(2, 3) == F32(1.5)


def _random_rows(rng, T, d, spread=1.0):
    return (rng.standard_normal((T, d)) * spread).astype(F32)


@pytest.mark.parametrize("b", [0.5, 1.0, 1.5, 0.03])
def test_error_bounds(b):
    rng = np.random.default_rng(7)
    cu = [0, 23, 30, 57]
    h = _random_rows(rng, 57, 64)
    anchors = K.group_anchors(cu)
    codes, scales = K.encode_layer(h, anchors, F32(b))
    dec = K.decode_layer(codes, scales, anchors, F32(b))
    for t in range(57):
        err = np.abs(dec[t].astype(np.float64) - h[t])
        if anchors[t] == t:
            # 8-bit anchor: half a step of max|h| / 127 (float32 rounding aside)
            assert err.max() <= scales[t] * 0.5 * (1 + 1e-5) + 1e-7
            assert np.abs(codes[t]).max() == 127
        else:
            delta = h[t].astype(np.float64) - K.dequantise_anchor(codes[anchors[t]],
                                                                  scales[anchors[t]])
            inside = np.abs(delta) <= 126.5 * b
            assert (err[inside] <= b * 0.5 * (1 + 1e-5) + 1e-6).all()


def test_lossless_when_values_sit_on_the_grids():
    rng = np.random.default_rng(3)
    b = F32(0.5)
    s = F32(1 / 32)
    q = rng.integers(-127, 128, (1, 48)).astype(F32)
    q[0, 0] = 127                                    # max|anchor| = 127 s -> scale s
    anchor = q * s
    deltas = rng.integers(-100, 101, (9, 48)).astype(F32) * b
    h = np.concatenate([anchor, anchor + deltas]).astype(F32)
    anchors = K.group_anchors([0, 10])
    codes, scales = K.encode_layer(h, anchors, b)
    assert scales[0] == s
    assert np.array_equal(K.decode_layer(codes, scales, anchors, b), h)


def test_saturation_and_zero_rows():
    h = np.zeros((3, 8), F32)
    h[1, 0] = 1000.0       # delta far beyond 127 bins
    h[1, 1] = -1000.0
    anchors = K.group_anchors([0, 3])
    codes, scales = K.encode_layer(h, anchors, F32(1.0))
    assert scales[0] == 0 and (codes[0] == 0).all()
    assert codes[1, 0] == 127 and codes[1, 1] == -127
    dec = K.decode_layer(codes, scales, anchors, F32(1.0))
    assert dec[1, 0] == 127.0 and dec[1, 1] == -127.0 and (dec[2] == 0).all()


def test_groups_decode_independently():
    """A group decodes from its own anchor only: changing another group's
    rows changes nothing in this one (no chain of deltas across groups)."""
    rng = np.random.default_rng(5)
    cu = [0, 30]
    h = _random_rows(rng, 30, 16)
    anchors = K.group_anchors(cu)
    c1, s1 = K.encode_layer(h, anchors, F32(1.0))
    h2 = h.copy()
    h2[10:20] += 3.0
    c2, s2 = K.encode_layer(h2, anchors, F32(1.0))
    assert np.array_equal(c1[:10], c2[:10]) and np.array_equal(c1[20:], c2[20:])
    assert np.array_equal(s1[:10], s2[:10]) and np.array_equal(s1[20:], s2[20:])


def test_round_to_storage():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], F32)
    # bf16 keeps 8 significant bits: 1 + 2^-8 is a tie -> even (1.0);
    # 1 + 3 * 2^-8 is a tie -> even (1 + 2^-6)
    bits = K.round_to_storage(x, "bf16")
    assert bits[0] == 0x3F80 and bits[1] == 0x3F80 and bits[2] == 0x3F82
    assert bits[3] == 0xC020
    assert np.array_equal(K.round_to_storage(x, "fp16"), x.astype(np.float16).view(np.uint16))


def test_multi_layer_encode_uses_each_layers_bin():
    rng = np.random.default_rng(9)
    cu = [0, 12]
    hs = [_random_rows(rng, 12, 8, 4.0) for _ in range(3)]
    codes, scales = K.encode(hs, 0, 3, cu)
    for i, b in enumerate((0.5, 1.0, 1.5)):
        c, s = K.encode_layer(hs[i], K.group_anchors(cu), F32(b))
        assert np.array_equal(codes[i], c) and np.array_equal(scales[i], s)
    dec = K.decode(codes, scales, 0, 3, cu)
    assert dec.shape == (3, 12, 8)


def test_tiny_rows_code_as_zero():
    """max|h| below 127 * 2^-126: scale 0 and all codes 0, so 1 / s stays finite."""
    h = np.zeros((2, 4), F32)
    h[0] = [1e-37, -2e-37, 0.0, 5e-38]
    h[1] = [1.0, 0.0, 0.0, 0.0]
    anchors = K.group_anchors([0, 2])
    codes, scales = K.encode_layer(h, anchors, F32(0.5))
    assert scales[0] == 0 and (codes[0] == 0).all()
    assert codes[1].tolist() == [2, 0, 0, 0]
    q, s = K.quantise_anchor(np.array([127 * 2.0 ** -126, 0.0], F32))
    assert s == F32(2.0 ** -126) and q.tolist() == [127, 0]


def test_reciprocal_step_differs_from_division_only_by_rounding():
    """The codes use x * (1/b); against x / b they differ by at most one step,
    and only where x / b sits within a rounding of a half-integer."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(200000) * 50).astype(F32)
    for b in (0.5, 1.0, 1.5, 0.3):
        inv = F32(F32(1) / F32(b))
        a = K.rint32((x * inv).astype(F32))
        d = K.rint32((x / F32(b)).astype(F32))
        assert np.abs(a - d).max() <= 1
        if b in (0.5, 1.0):           # power-of-two steps: identical
            assert np.array_equal(a, d)


def test_defaults_are_the_pages_parameters():
    """The oracle's and the library binding's codec defaults, and the save
    side's chunk size used throughout, are the values the pages print
    (tests/golden/page_parameters.json, each with its citation)."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "page_parameters.json")) as f:
        g = json.load(f)
    assert K.GROUP_TOKENS == g["codec"]["group_tokens"]
    assert tuple(K.DEFAULT_BINS) == tuple(g["codec"]["bins_first_middle_last"])
    # 8-bit symmetric anchors: codes span [-(2^7 - 1), 2^7 - 1]
    q, _ = K.quantise_anchor(np.array([1.0, -1.0, 0.5], F32))
    assert q.max() == 2 ** (g["codec"]["anchor_bits"] - 1) - 1
    assert q.min() == -(2 ** (g["codec"]["anchor_bits"] - 1) - 1)
    from kv_cache_restoration_gb300 import binding as B
    p = B.codec_params()
    assert list(p.bins) == g["codec"]["bins_first_middle_last"]
    assert p.group_tokens == g["codec"]["group_tokens"]
    assert g["save_chunk_tokens"]["value"] == 64

"""The weight-row tiles' host plan without a GPU: for every token count the
chunks cover the tokens with less than 16 tokens of padding per chunk, and the
TMEM accumulator slots fit the 512 allocated columns on 32-column boundaries,
with every MMA's N a multiple of 16 between 16 and 256 (the cta_group::2,
M = 256 shapes)."""
import pytest

TMEM_COLS = 512


@pytest.fixture(scope="module")
def B():
    from kv_cache_restoration_gb300 import binding   # built at session start
    return binding


def mma_widths(n, slot_cols):
    """N of the MMAs of a unit of n tokens: the first n - slot_cols columns in
    the small slot when the unit is wider than a big slot, the rest in it."""
    return [n] if n <= slot_cols else [n - slot_cols, slot_cols]


def split_halves(n):
    """A split tail tile's two units (the first rounded up to 16 tokens)."""
    n1 = (n // 2 + 15) & ~15
    return [n1, n - n1]


def test_every_token_count_has_a_valid_plan(B):
    for t in range(1, 4097):
        p = B.hcr_debug_swap_plan(t)
        assert p["ok"] == 1, (t, p)
        chunk, n_chunks, last_n = p["chunk"], p["n_chunks"], p["last_n"]
        assert chunk % 16 == 0 and last_n % 16 == 0 and 16 <= last_n <= chunk, (t, p)
        covered = (n_chunks - 1) * chunk + last_n
        assert t <= covered < t + 16 * n_chunks, (t, p)
        assert (n_chunks - 1) * chunk < t, (t, p)   # the last chunk holds tokens


@pytest.mark.parametrize("t", [1, 16, 64, 255, 256, 257, 271, 272, 288, 300, 304, 319, 320,
                               321, 512, 794, 4096])
def test_slots_fit_tensor_memory(B, t):
    p = B.hcr_debug_swap_plan(t)
    sc, ns, chunk = p["slot_cols"], p["n_slots"], p["chunk"]
    if 256 < t <= 320:
        # one chunk on two big slots and a small one after them
        assert (ns, p["n_chunks"]) == (3, 1), p
        assert sc % 32 == 0 and sc <= 256, p
        small = chunk - sc
        assert 16 <= small and small % 16 == 0, p
        assert 2 * sc + small <= TMEM_COLS, p
        # the largest such big slot: one more 32 columns would not fit
        assert sc + 32 + chunk > TMEM_COLS, p
    else:
        assert (ns, sc) == (2, 256) and chunk <= 256, p
    units = [chunk, p["last_n"]]
    if chunk >= 32 and p["last_n"] >= 32:
        units += split_halves(chunk) + split_halves(p["last_n"])
    for n in units:
        widths = mma_widths(n, sc)
        assert sum(widths) == n
        for w in widths:
            assert 16 <= w <= 256 and w % 16 == 0, (t, n, widths)
        if len(widths) == 2:
            assert ns == 3 and widths[0] <= chunk - sc, (t, n, widths)


def test_three_slot_splits(B):
    # big + small columns of each chunk of the three-slot layout
    want = {257: (272, 224), 288: (288, 224), 300: (304, 192), 320: (320, 192)}
    for t, (chunk, big) in want.items():
        p = B.hcr_debug_swap_plan(t)
        assert (p["chunk"], p["slot_cols"]) == (chunk, big), p


def test_rejects_null_output(B):
    assert B.lib.hcr_debug_swap_plan(300, None) == 1

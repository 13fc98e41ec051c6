"""The save-side oracle against hand-worked values, brute force and identities (CPU)."""
import numpy as np
import pytest

from oracle import save as S


def test_hand_worked_layout():
    # chunk size 4, two layers, d = 1, value = 100*layer + token index.
    # r0: start 0, 6 tokens, chunks [3, 1]: positions 0..3 -> chunk 3 offsets 0..3,
    #     positions 4, 5 -> chunk 1 offsets 0, 1.
    # r1: start 2, 3 tokens, chunks [0, 2]: positions 2, 3 -> chunk 0 offsets 2, 3,
    #     position 4 -> chunk 2 offset 0.
    cu, st, tab = [0, 6, 9], [0, 2], [[3, 1], [0, 2]]
    h = [np.array([[100.0 * l + t] for t in range(9)]) for l in range(2)]
    buf = S.save_chunks(h, 0, 2, cu, st, tab, 4, num_chunks=5)
    for l in range(2):
        assert buf[3, l, :, 0].tolist() == [100 * l + t for t in (0, 1, 2, 3)]
        assert buf[1, l, :2, 0].tolist() == [100 * l + 4, 100 * l + 5]
        assert np.isnan(buf[1, l, 2:, 0]).all()
        assert np.isnan(buf[0, l, :2, 0]).all()
        assert buf[0, l, 2:, 0].tolist() == [100 * l + 6, 100 * l + 7]
        assert buf[2, l, 0, 0] == 100 * l + 8 and np.isnan(buf[2, l, 1:, 0]).all()
        assert np.isnan(buf[4]).all()


def _random_layout(rng, n_req, C, spare=3):
    lens = rng.integers(0, 50, n_req)
    st = rng.integers(0, 40, n_req)
    need = [(s + n + C - 1) // C for s, n in zip(st, lens)]
    ids = rng.permutation(sum(need) + spare)
    tab = np.full((n_req, max(max(need), 1)), -1)
    k = 0
    for r, nc in enumerate(need):
        tab[r, :nc] = ids[k:k + nc]
        k += nc
    cu = np.concatenate([[0], np.cumsum(lens)])
    return cu, st, tab, len(ids)


@pytest.mark.parametrize("C", [1, 4, 64])
def test_against_chunk_walk(C):
    """Brute force from the other side: every (request, logical chunk, offset)
    slot gets the token at that position, if the request saved one."""
    rng = np.random.default_rng(C)
    cu, st, tab, n = _random_layout(rng, 6, C)
    L, d = 3, 5
    T = int(cu[-1])
    h = [rng.normal(size=(T, d)) for _ in range(L)]
    buf = S.save_chunks(h, 0, L, cu, st, tab, C, n)
    want = np.full_like(buf, np.nan)
    for r in range(len(st)):
        for k, cid in enumerate(tab[r]):
            if cid < 0:
                continue
            for off in range(C):
                p = k * C + off
                if st[r] <= p < st[r] + (cu[r + 1] - cu[r]):
                    t = cu[r] + p - st[r]
                    for l in range(L):
                        want[cid, l, off] = h[l][t]
    assert np.array_equal(np.isnan(buf), np.isnan(want))
    assert np.array_equal(np.nan_to_num(buf), np.nan_to_num(want))


def test_round_trip_and_layer_ranges():
    rng = np.random.default_rng(7)
    cu, st, tab, n = _random_layout(rng, 5, 64)
    L, d = 4, 8
    T = int(cu[-1])
    h = [rng.normal(size=(T, d)) for _ in range(L)]
    buf = S.save_chunks(h[:2], 0, L, cu, st, tab, 64, n)
    buf = S.save_chunks(h[2:], 2, L, cu, st, tab, 64, n, buf=buf)
    got = S.load_chunks(buf, 0, L, cu, st, tab, 64)
    assert np.array_equal(got, np.stack(h))
    assert np.array_equal(S.load_chunks(buf, 1, 3, cu, st, tab, 64), np.stack(h[1:3]))


def test_decode_steps_equal_one_save():
    """Saving each request's tokens one decode step at a time (one token per
    request per step, layer-before-token as generation produces them) fills the
    chunks exactly like saving all tokens at once."""
    rng = np.random.default_rng(9)
    n_req, steps, L, d, C = 3, 70, 2, 4, 64
    start = np.array([0, 5, 63])
    need = [(s + steps + C - 1) // C for s in start]
    ids = rng.permutation(sum(need))
    tab = np.full((n_req, max(need)), -1)
    k = 0
    for r, nc in enumerate(need):
        tab[r, :nc] = ids[k:k + nc]
        k += nc
    hid = rng.normal(size=(L, n_req, steps, d))          # [layer][request][step][d]
    once = S.save_chunks([hid[l].reshape(n_req * steps, d) for l in range(L)], 0, L,
                         np.arange(n_req + 1) * steps, start, tab, C, len(ids))
    buf = None
    for s in range(steps):
        buf = S.save_chunks([hid[l][:, s] for l in range(L)], 0, L, np.arange(n_req + 1),
                            start + s, tab, C, len(ids), buf=buf)
    assert np.array_equal(np.isnan(buf), np.isnan(once))
    assert np.array_equal(np.nan_to_num(buf), np.nan_to_num(once))


def test_rejects_bad_tables():
    with pytest.raises(ValueError):
        S.chunk_placement([0, 3], [62], [[0]], 64, num_chunks=2)     # position 64 has no chunk
    with pytest.raises(ValueError):
        S.chunk_placement([0, 3], [0], [[2]], 64, num_chunks=2)      # id 2 >= 2

"""Pin checks for the oracle: each returns None or raises AssertionError.

They are functions of an oracle module (oracle.restore) so the mutation tests
can hand them a copy with a planted mistake and see them fail.  The expected
values here are closed forms, invariants, brute force on tiny inputs and an
independent transformer forward pass -- never the oracle re-typed.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import tiny_model as tm


def _close(a, b, tol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"max abs error {err} > {tol}"


# ---------------------------------------------------------------------------
# Norms
# ---------------------------------------------------------------------------
def pin_rms_constant(R):
    """RMSNorm of c*1 is gamma*c/sqrt(c^2+eps): y/gamma = sign(c) up to 5e-6 for |c|>=1, 0 at c=0."""
    rng = np.random.default_rng(1)
    gamma = rng.normal(1.0, 0.1, 64)
    for c in (1.0, -1.0, 3.5, -7.25, 100.0):
        y = R.rms_norm(np.full((2, 64), c), gamma, 1e-5)
        _close(y / gamma, np.full((2, 64), math.copysign(1.0, c)), 5e-6)
        _close(y, np.broadcast_to(gamma * c / math.sqrt(c * c + 1e-5), (2, 64)), 1e-14)
    _close(R.rms_norm(np.zeros((1, 64)), gamma, 1e-5), np.zeros((1, 64)), 0.0)


def pin_rms_values(R):
    # (3, 4): mean of squares = 12.5; eps = 0 -> divide by sqrt(12.5)
    y = R.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    _close(y, [[3.0 / math.sqrt(12.5), 8.0 / math.sqrt(12.5)]], 1e-15)
    # eps sits inside the square root: h = (0, 0, 0, 2): ms = 1, eps = 3 -> /2
    y = R.rms_norm(np.array([[0.0, 0.0, 0.0, 2.0]]), np.ones(4), 3.0)
    _close(y, [[0.0, 0.0, 0.0, 1.0]], 1e-15)
    # with gamma = 1 and eps = 0 the output has unit root-mean-square
    h = np.random.default_rng(2).normal(0, 3, (5, 96))
    y = R.rms_norm(h, np.ones(96), 0.0)
    _close(np.sqrt((y * y).mean(axis=-1)), np.ones(5), 1e-12)


def pin_layer_norm(R):
    rng = np.random.default_rng(3)
    g, b = rng.normal(1, 0.1, 32), rng.normal(0, 0.02, 32)
    # LN of a constant vector is beta
    _close(R.layer_norm(np.full((3, 32), 4.2), g, b, 1e-5), np.broadcast_to(b, (3, 32)), 1e-12)
    # (1, 2, 3, 4): mean 2.5, biased variance 1.25
    y = R.layer_norm(np.array([[1.0, 2.0, 3.0, 4.0]]), np.ones(4), np.zeros(4), 0.0)
    s = math.sqrt(1.25)
    _close(y, [[-1.5 / s, -0.5 / s, 0.5 / s, 1.5 / s]], 1e-15)
    # eps inside the square root: (1, -1): var 1, eps 3 -> /2
    y = R.layer_norm(np.array([[1.0, -1.0]]), np.ones(2), np.zeros(2), 3.0)
    _close(y, [[0.5, -0.5]], 1e-15)
    # gamma=1, beta=0, eps=0: zero mean, unit biased variance, shift-invariant
    h = rng.normal(5, 2, (4, 32))
    y = R.layer_norm(h, np.ones(32), np.zeros(32), 0.0)
    _close(y.mean(axis=-1), np.zeros(4), 1e-12)
    _close((y * y).mean(axis=-1), np.ones(4), 1e-12)
    _close(R.layer_norm(h + 3.0, g, b, 1e-5), R.layer_norm(h, g, b, 1e-5), 1e-10)


# ---------------------------------------------------------------------------
# Projection
# ---------------------------------------------------------------------------
def pin_project_bruteforce(R):
    """y[t][j] = sum_i x[t][i] * W[j][i] (+ b[j]) by explicit loops."""
    rng = np.random.default_rng(4)
    x, w, b = rng.normal(size=(3, 5)), rng.normal(size=(4, 5)), rng.normal(size=4)
    want = [[sum(x[t][i] * w[j][i] for i in range(5)) + b[j] for j in range(4)]
            for t in range(3)]
    _close(R.project(x, w, b), want, 1e-13)
    # W is [out, in]: a one-hot input picks column i of W
    e = np.zeros((1, 5))
    e[0, 2] = 1.0
    _close(R.project(e, w), w[:, 2][None, :], 0.0)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------
def pin_rope_closed_form(R):
    """Unit vectors at positions chosen so the angle is exactly 1 radian.

    With dh = 8 and theta = 1e4 the frequencies are 1, 0.1, 0.01, 0.001, so
    pair i at position 10^i turns by 1 rad: (a, b) -> (a cos1 - b sin1, b cos1 + a sin1),
    with b the coordinate dh/2 further along (rotate-half pairing).
    """
    c1, s1 = math.cos(1.0), math.sin(1.0)
    cases = [  # (input index list, position, expected dense vector)
        ([0], 1, {0: c1, 4: s1}),
        ([1], 10, {1: c1, 5: s1}),
        ([6], 100, {2: -s1, 6: c1}),
        ([3, 7], 1000, {3: c1 - s1, 7: c1 + s1}),
    ]
    for idx, p, out in cases:
        x = np.zeros((1, 1, 8))
        x[0, 0, idx] = 1.0
        want = np.zeros((1, 1, 8))
        for k, v in out.items():
            want[0, 0, k] = v
        _close(R.rope_rotate_half(x, np.array([p]), 1e4), want, 1e-12)


def pin_rope_invariants(R):
    rng = np.random.default_rng(5)
    k = rng.normal(size=(6, 3, 64))
    pos = np.array([0, 1, 7, 300, 4095, 24000])
    # position 0 is the identity, exactly
    assert np.array_equal(R.rope_rotate_half(k[:1], np.array([0]), 1e4), k[:1])
    # each rotated pair keeps its norm
    y = R.rope_rotate_half(k, pos, 1e4)
    n_in = k[..., :32] ** 2 + k[..., 32:] ** 2
    n_out = y[..., :32] ** 2 + y[..., 32:] ** 2
    _close(n_out, n_in, 1e-11)
    # composition: rope(rope(x, p), q) == rope(x, p + q)
    p, q = np.array([3, 50, 1000]), np.array([4, 77, 2048])
    _close(R.rope_rotate_half(R.rope_rotate_half(k[:3], p, 1e4), q, 1e4),
           R.rope_rotate_half(k[:3], p + q, 1e4), 1e-9)
    # <rope(a, m), rope(b, n)> depends only on m - n
    a, b = rng.normal(size=(1, 1, 64)), rng.normal(size=(1, 1, 64))

    def dot(m, n):
        return float(np.sum(R.rope_rotate_half(a, np.array([m]), 1e4)
                            * R.rope_rotate_half(b, np.array([n]), 1e4)))
    base = dot(10, 3)
    for m, n in ((17, 10), (1007, 1000), (20007, 20000)):
        assert abs(dot(m, n) - base) < 1e-9, (m, n)


# ---------------------------------------------------------------------------
# Placement
# ---------------------------------------------------------------------------
def _placement_by_blocks(cu, st, bt, B):
    """Brute force from the other side: walk every (request, logical block,
    offset) and record which concatenated token lands at that physical slot."""
    slots = {}
    for r in range(len(st)):
        n = cu[r + 1] - cu[r]
        for lb, phys in enumerate(bt[r]):
            if phys < 0:
                continue
            for off in range(B):
                p = lb * B + off
                if st[r] <= p < st[r] + n:
                    slots[cu[r] + (p - st[r])] = phys * B + off
    return np.array([slots[t] for t in range(cu[-1])], dtype=np.int64)


def pin_placement(R):
    # hand-worked: B = 4.  r0: start 0, 5 tokens, blocks [7, 2]: positions 0..3 ->
    # block 7 (slots 28..31), position 4 -> block 2 offset 0 (slot 8).
    # r1: start 6, 3 tokens, blocks [0, 5, 9]: positions 6, 7 -> block 5 offsets 2, 3
    # (slots 22, 23), position 8 -> block 9 offset 0 (slot 36).  r2: empty.
    cu, st = [0, 5, 8, 8], [0, 6, 3]
    bt = [[7, 2, -1], [0, 5, 9], [4, -1, -1]]
    pl = R.token_placement(cu, st, bt, 4, num_blocks=10)
    assert pl.slot.tolist() == [28, 29, 30, 31, 8, 22, 23, 36]
    assert pl.pos.tolist() == [0, 1, 2, 3, 4, 6, 7, 8]
    assert pl.request.tolist() == [0, 0, 0, 0, 0, 1, 1, 1]
    # random ragged layouts against the block-walking brute force
    rng = np.random.default_rng(6)
    for B in (1, 4, 16):
        R_ = 5
        lens = rng.integers(0, 40, R_)
        st = rng.integers(0, 30, R_)
        need = [(s + n + B - 1) // B for s, n in zip(st, lens)]
        ids = rng.permutation(sum(need) + 3)
        bt = np.full((R_, max(need)), -1)
        k = 0
        for r, nb in enumerate(need):
            bt[r, :nb] = ids[k:k + nb]
            k += nb
        cu = np.concatenate([[0], np.cumsum(lens)])
        pl = R.token_placement(cu, st, bt, B, num_blocks=len(ids))
        assert np.array_equal(pl.slot, _placement_by_blocks(cu, st, bt, B))
        assert len(set(pl.slot.tolist())) == len(pl.slot)   # injective


# ---------------------------------------------------------------------------
# Whole restore
# ---------------------------------------------------------------------------
def pin_identity_weights(R):
    """W_k = W_v = I, gamma = 1, position 0: K = V = RMSNorm(h) (library-free closed form)."""
    rng = np.random.default_rng(7)
    d = 32
    h = rng.normal(size=(3, d))
    lw = R.LayerWeights(gamma=np.ones(d), w_k=np.eye(d), w_v=np.eye(d))
    spec = R.ModelSpec(d_model=d, n_kv_heads=2, head_dim=16)
    k, v = R.restore_layer(h, lw, np.zeros(3, np.int64), spec)
    want = (h / np.sqrt((h ** 2).mean(axis=1, keepdims=True) + 1e-5)).reshape(3, 2, 16)
    _close(k, want, 1e-14)
    _close(v, want, 1e-14)


def _oracle_from_tiny(R, m: tm.TinyModel):
    cfg = m.cfg
    spec = R.ModelSpec(d_model=cfg.d_model, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                       norm="ln" if cfg.family == "opt" else "rms", norm_eps=cfg.norm_eps,
                       rope=cfg.family == "llama", rope_theta=cfg.rope_theta)
    weights = [R.LayerWeights(gamma=l.norm1_g, beta=l.norm1_b, w_k=l.w_k(cfg), w_v=l.w_v(cfg),
                              b_k=l.b_k(cfg), b_v=l.b_v(cfg)) for l in m.layers]
    return spec, weights


def pin_tiny_forward(R, family: str, n_kv_heads: int = 4):
    """Restoring from each layer's recorded input gives back the K/V that the
    forward pass's attention used; then decoding one more token from the
    restored paged cache reproduces the full forward pass's logits.

    The request restores positions [S, S+N) into a shuffled block table; the
    resident prefix [0, S) is written from the forward pass itself.
    """
    cfg = tm.TinyConfig(family=family, n_kv_heads=n_kv_heads)
    m = tm.random_model(cfg, seed=11)
    rng = np.random.default_rng(12)
    S, N, B = 9, 30, 4
    toks = rng.integers(0, cfg.vocab, S + N + 1)
    full = tm.forward(m, toks)                   # S+N+1 tokens from position 0
    ctx = tm.forward(m, toks[:S + N])            # the evicted context
    spec, weights = _oracle_from_tiny(R, m)
    pos = np.arange(S, S + N)
    for l in range(cfg.n_layers):
        k, v = R.restore_layer(ctx.hidden[l][S:], weights[l], pos, spec)
        _close(k, ctx.k[l][S:], 1e-11)
        _close(v, ctx.v[l][S:], 1e-11)
    nb = (S + N + 1 + B - 1) // B
    table = rng.permutation(nb + 2)[:nb]
    cache = R.restore([ctx.hidden[l][S:] for l in range(cfg.n_layers)], weights, spec,
                      [0, N], [S], table[None, :], B, num_blocks=nb + 2)
    kc, vc = cache.k.copy(), cache.v.copy()
    pre = np.arange(S)
    pslots = table[pre // B] * B + pre % B
    for l in range(cfg.n_layers):
        assert np.all(np.isnan(kc[l, pslots]))   # restore leaves the prefix alone
        kc[l, pslots] = ctx.k[l][:S]
        vc[l, pslots] = ctx.v[l][:S]
    logits = tm.decode_from_paged_cache(m, int(toks[S + N]), S + N, kc, vc, table, B)
    _close(logits, full.logits[-1], 1e-9)
    # and the context's own logits match the longer pass (causality sanity)
    _close(ctx.logits, full.logits[:S + N], 1e-9)


def pin_kv_bytes(R, facts):
    """Byte accounting against the pages' KV size rule and capacity facts."""
    # one token, one layer, one head of width 1, 2-byte elements: one K and one V element
    assert R.kv_bytes(1, 1, 1, 1, 2) == 4
    assert R.kv_bytes(3, 5, 7, 11, 2) == 2 * 3 * 5 * 7 * 11 * 2
    for f in facts["a100_40gb_capacity"]:
        per_tok = R.kv_bytes(f["n_layers"], f["n_heads"], f["head_dim"], 1, 2)
        kv_gb = f["tokens"] * per_tok / 1e9
        weights_gb = f["params_billion"] * 2.0
        total = kv_gb + weights_gb
        assert f["fits_within_gb"][0] <= total <= f["fits_within_gb"][1], (f, total)

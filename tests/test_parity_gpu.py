"""CUDA restore vs the oracle, through the C ABI (GPU)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from tests import harness as Hn
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu


def W(name, shape, lens, starts, **kw):
    return Workload(name, shape, tuple(lens), tuple(starts), **kw)


# Small cases the oracle checks in full: several M-tiles with a ragged tail,
# several N-tiles, every head width, both norms and dtypes, biases, GQA,
# a partial K block, a ragged last N tile, empty requests, prefixes.
SMALL_CASES = [
    C.get("tiny"),
    W("ragged-small", ModelShape("s128", 3, 512, 4, 4, 128), [1, 200, 0, 77, 300],
      [0, 5, 9, 1000, 31], block_order="shuffled", spare_blocks=3),
    W("dh64", ModelShape("s64", 2, 384, 6, 6, 64), [130, 129], [3, 0], block_order="shuffled"),
    W("dh256", ModelShape("s256", 2, 256, 2, 2, 256), [70, 100], [0, 17]),
    W("ln-fp16-bias", ModelShape("ln", 2, 512, 4, 4, 128, norm="ln", rope=False, dtype="fp16",
                                 kv_bias=True), [250, 10], [0, 40], block_order="shuffled"),
    W("rms-bias", ModelShape("rmsb", 1, 256, 2, 2, 128, kv_bias=True), [129], [2]),
    W("gqa", ModelShape("gqa", 2, 512, 8, 2, 128), [300], [100], block_order="shuffled"),
    W("ragged-n", ModelShape("h5", 2, 256, 5, 5, 64), [140], [0]),
    W("odd-d", ModelShape("d200", 2, 200, 2, 2, 64), [131], [7]),
    W("block1", ModelShape("b1", 1, 256, 2, 2, 64), [40, 9], [3, 0], block_size=1,
      block_order="shuffled"),
    W("theta5e5", ModelShape("t5", 1, 256, 2, 2, 128, rope_theta=5e5), [64], [20000]),
    W("fp16-rope", ModelShape("f16r", 2, 384, 3, 3, 128, dtype="fp16"), [200, 57], [11, 300],
      block_order="shuffled"),
    W("many-requests", ModelShape("mr", 1, 256, 2, 2, 64),
      [int(x) for x in np.random.default_rng(3).integers(0, 21, 150)],
      [int(x) for x in np.random.default_rng(4).integers(0, 200, 150)], block_size=32,
      block_order="shuffled"),
    W("single-token", ModelShape("one", 2, 256, 2, 2, 128), [1], [77]),
    W("ln-dh256", ModelShape("ln256", 1, 512, 2, 2, 256, norm="ln", kv_bias=True), [260], [3]),
    W("d8192", ModelShape("d8k", 1, 8192, 2, 2, 128), [300], [0]),
    W("block64", ModelShape("b64", 1, 256, 4, 4, 64), [333, 2], [65, 0], block_size=64,
      block_order="shuffled"),
    # the CTA pairs' last tile: 128 rows (384 tokens) is a half tile, 129 rows
    # (385) a full one
    W("tail128", ModelShape("t128", 2, 256, 2, 2, 128), [100, 284], [0, 9]),
    W("tail129", ModelShape("t129", 2, 256, 2, 2, 128), [100, 285], [0, 9]),
]


VARIANTS = {"auto": 0, "single": 1, "pair": 2, "swap": 3}


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("w", SMALL_CASES, ids=[w.name for w in SMALL_CASES])
def test_small_full(cuda_device, w, variant):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(w, cuda_device)
    st = B.hcr_debug_set_variant(case.restorer.handle, VARIANTS[variant])
    if variant.startswith("swap") and w.shape.head_dim != 128:
        assert st == B.HCR_ERR_UNSUPPORTED      # weight-row tiles need 128-wide heads
        return
    assert st == 0
    Hn.run(case)
    assert case.status == 0, (case.status, case.flags)
    Hn.compare(case)


AGREE_CASES = [SMALL_CASES[1], SMALL_CASES[4], SMALL_CASES[6], SMALL_CASES[11]]


@pytest.mark.parametrize("w", AGREE_CASES, ids=[w.name for w in AGREE_CASES])
def test_variants_agree(cuda_device, w):
    """Single-CTA, CTA-pair and weight-row tiles restore the same values
    (compared bit for bit; a difference would show as a count of differing
    elements): RMSNorm and LayerNorm with bias, bf16 and fp16, GQA, RoPE."""
    from kv_cache_restoration_gb300 import binding as B
    a = Hn.make_case(w, cuda_device)
    B.hcr_debug_set_variant(a.restorer.handle, 1)
    Hn.run(a)
    for v in (2, 3):
        b = Hn.make_case(w, cuda_device, params=a.params, restorer=a.restorer)
        assert B.hcr_debug_set_variant(b.restorer.handle, v) == 0
        Hn.run(b)
        assert b.status == 0
        for c in ("k_cache", "v_cache"):
            diff = int((getattr(a, c).view(torch.int16) != getattr(b, c).view(torch.int16)).sum())
            assert diff == 0, f"variant {v}, {c}: {diff} elements differ from single CTAs"


def test_empty_restore_is_a_noop(cuda_device):
    w = C.get("tiny")
    case = Hn.make_case(w, cuda_device)
    before = case.k_cache.clone()
    lay = case.layout
    empty = case.hidden[:, :0]
    case.restorer.restore(empty, 0, 2, case.cu[:1], case.start[:0], case.table, case.k_cache,
                          case.v_cache, lay.num_blocks, lay.block_size)
    case.restorer.restore(case.hidden[:0], 1, 1, case.cu, case.start, case.table, case.k_cache,
                          case.v_cache, lay.num_blocks, lay.block_size)
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), case.k_cache.view(torch.int16))


def test_split_stages_match_restore_bitwise(cuda_device):
    w = SMALL_CASES[1]
    a = Hn.run(Hn.make_case(w, cuda_device))
    b = Hn.make_case(w, cuda_device, params=a.params, restorer=a.restorer)
    lay = b.layout
    for stage in ("prepare", "project"):
        b.restorer.restore(b.hidden, 0, w.shape.n_layers, b.cu, b.start, b.table, b.k_cache,
                           b.v_cache, lay.num_blocks, lay.block_size, stage=stage)
    torch.cuda.synchronize()
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))


def test_deterministic(cuda_device):
    w = SMALL_CASES[1]
    a = Hn.run(Hn.make_case(w, cuda_device))
    b = Hn.run(Hn.make_case(w, cuda_device, params=a.params, restorer=a.restorer))
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))


def test_layer_split_bitwise(cuda_device):
    """Restoring [0, L) at once equals restoring [0, k) then [k, L)."""
    w = W("split", ModelShape("sp", 4, 256, 2, 2, 128), [150, 60], [0, 9])
    full = Hn.run(Hn.make_case(w, cuda_device))
    lo = Hn.run(Hn.make_case(w, cuda_device, 0, 1, params=full.params, restorer=full.restorer))
    hi = Hn.run(Hn.make_case(w, cuda_device, 1, 4, params=full.params, restorer=full.restorer))
    for c in ("k_cache", "v_cache"):
        whole = getattr(full, c).view(torch.int16)
        parts = torch.cat([getattr(lo, c), getattr(hi, c)]).view(torch.int16)
        assert torch.equal(whole, parts)


def test_layer_stride_and_offset_base(cuda_device):
    """Caches with padding between layers, restored from a base in the middle."""
    w = W("stride", ModelShape("st", 3, 256, 2, 2, 64), [90], [0])
    ref = Hn.run(Hn.make_case(w, cuda_device))
    case = Hn.make_case(w, cuda_device, 1, 3, params=ref.params, restorer=ref.restorer)
    lay = case.layout
    per_layer = lay.num_blocks * lay.block_size * 2 * 64
    stride = per_layer + 24
    big_k = torch.full((3 * stride,), G.SENTINEL_BITS, dtype=torch.int16, device=cuda_device)
    big_v = big_k.clone()
    case.restorer.restore(case.hidden, 1, 3, case.cu, case.start, case.table,
                          big_k[stride:].view(torch.bfloat16), big_v[stride:].view(torch.bfloat16),
                          lay.num_blocks, lay.block_size, layer_stride_elems=stride)
    torch.cuda.synchronize()
    for li, l in enumerate((1, 2)):
        got = big_k[stride * (1 + li): stride * (1 + li) + per_layer]
        assert torch.equal(got, ref.k_cache[l].reshape(-1).view(torch.int16))
        pad = big_k[stride * (1 + li) + per_layer: stride * (2 + li)]
        assert bool((pad == G.SENTINEL_BITS).all())
    assert bool((big_k[:stride] == G.SENTINEL_BITS).all())


def test_request_permutation_invariance(cuda_device):
    """Reordering requests (rows of hidden and of the block table) changes no
    cache bit: placement depends only on each request's own table."""
    w = SMALL_CASES[1]
    a = Hn.run(Hn.make_case(w, cuda_device))
    perm = [3, 0, 4, 2, 1]
    lay = a.layout
    cu = lay.cu_seqlens
    segs = [np.arange(cu[r], cu[r + 1]) for r in range(len(perm))]
    rows = np.concatenate([segs[r] for r in perm]).astype(np.int64)
    lens = np.array([cu[r + 1] - cu[r] for r in perm])
    cu2 = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    b = Hn.make_case(w, cuda_device, params=a.params, restorer=a.restorer)
    b.hidden = b.hidden[:, torch.as_tensor(rows, device=cuda_device)].contiguous()
    b.cu = torch.as_tensor(cu2, device=cuda_device)
    b.start = b.start[torch.as_tensor(perm, device=cuda_device)].contiguous()
    b.table = b.table[torch.as_tensor(perm, device=cuda_device)].contiguous()
    b.restorer.restore(b.hidden, 0, w.shape.n_layers, b.cu, b.start, b.table, b.k_cache,
                       b.v_cache, lay.num_blocks, lay.block_size)
    torch.cuda.synchronize()
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))


def test_v_independent_of_start(cuda_device):
    w1 = W("s0", ModelShape("vs", 1, 256, 2, 2, 64), [64], [0])
    w2 = replace(w1, start_pos=(48,))
    a = Hn.run(Hn.make_case(w1, cuda_device))
    b = Hn.run(Hn.make_case(w2, cuda_device, params=a.params))
    la, lb = a.layout, b.layout
    pa = np.arange(64)
    pb = 48 + np.arange(64)
    sa = la.block_table[0][pa // 16] * 16 + pa % 16
    sb = lb.block_table[0][pb // 16] * 16 + pb % 16
    va = a.v_cache[0].reshape(-1, 2, 64)[torch.as_tensor(sa, device=cuda_device)]
    vb = b.v_cache[0].reshape(-1, 2, 64)[torch.as_tensor(sb, device=cuda_device)]
    assert torch.equal(va.view(torch.int16), vb.view(torch.int16))
    ka = a.k_cache[0].reshape(-1, 2, 64)[torch.as_tensor(sa, device=cuda_device)]
    kb = b.k_cache[0].reshape(-1, 2, 64)[torch.as_tensor(sb, device=cuda_device)]
    assert not torch.equal(ka.view(torch.int16), kb.view(torch.int16))


def test_rope_position_zero_is_exact(cuda_device):
    """At position 0 the rotation is the identity (cos 1, sin 0 in the table),
    so K columns equal an unrotated restore of the same row, bit for bit."""
    shape = ModelShape("p0", 1, 256, 2, 2, 64)
    a = Hn.run(Hn.make_case(W("r", shape, [16], [0]), cuda_device))
    b = Hn.run(Hn.make_case(W("n", replace(shape, rope=False), [16], [0]), cuda_device,
                            params=a.params))
    assert torch.equal(a.k_cache[0, 0, 0].view(torch.int16), b.k_cache[0, 0, 0].view(torch.int16))
    assert not torch.equal(a.k_cache[0, 0, 1].view(torch.int16),
                           b.k_cache[0, 0, 1].view(torch.int16))


# ----------------------------------------------------------------------------- device bounds
def test_bad_block_id_is_skipped_and_flagged(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    w = W("bad", ModelShape("bb", 1, 256, 2, 2, 64), [40, 30], [0, 0], spare_blocks=2)
    case = Hn.make_case(w, cuda_device)
    lay = case.layout
    case.table[1, 1] = lay.num_blocks + 7        # positions 16..29 of request 1
    Hn.run(case)
    assert case.status == B.HCR_ERR_DEVICE_BOUNDS
    assert case.flags & B.HCR_DEVERR_BLOCK_ID
    keep = np.r_[np.arange(0, 40), np.arange(40, 56)]       # every other row is restored
    Hn.compare(case, rows=keep, check_sentinel=False)
    from oracle import restore as R
    pl = R.token_placement(lay.cu_seqlens, lay.start_pos, lay.block_table, 16, lay.num_blocks)
    Hn.check_sentinels(case, pl.slot[keep])
    assert case.restorer.check()[0] == 0          # the error word was cleared


def test_position_beyond_rope_table_is_flagged(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    w = W("pos", ModelShape("pp", 1, 256, 2, 2, 64), [20], [10], max_position=25)
    case = Hn.run(Hn.make_case(w, cuda_device))
    assert case.status == B.HCR_ERR_DEVICE_BOUNDS and case.flags & B.HCR_DEVERR_POSITION
    Hn.compare(case, rows=np.arange(15), check_sentinel=False)


def test_seqlens_mismatch_is_flagged(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    w = W("cu", ModelShape("cu", 1, 256, 2, 2, 64), [20, 12], [0, 0])
    case = Hn.make_case(w, cuda_device)
    case.cu[2] = 30                                   # host says 32 tokens
    Hn.run(case)
    assert case.status == B.HCR_ERR_DEVICE_BOUNDS and case.flags & B.HCR_DEVERR_SEQLENS


def test_host_validation(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    w = C.get("tiny")
    case = Hn.make_case(w, cuda_device)
    lay = case.layout
    r = case.restorer
    ws = r.workspace(w.n_tokens, 2, cuda_device)
    layout = B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0)
    good = dict(handle=r.handle, hidden=case.hidden, layer_begin=0, layer_end=2, n_req=1,
                n_tokens=w.n_tokens, cu_seqlens=case.cu, start_pos=case.start,
                block_table=case.table, max_blocks_per_req=lay.max_blocks, k_cache=case.k_cache,
                v_cache=case.v_cache, layout=layout, workspace=ws, workspace_bytes=ws.numel())

    def call(**kw):
        args = dict(good, **kw)
        return B.hcr_restore(*args.values(), check=False)

    assert call(layer_end=3) == B.HCR_ERR_INVALID_ARG
    assert call(layer_begin=-1) == B.HCR_ERR_INVALID_ARG
    assert call(n_tokens=-1) == B.HCR_ERR_INVALID_ARG
    assert call(hidden=None) == B.HCR_ERR_INVALID_ARG
    assert call(hidden=case.hidden.data_ptr() + 2) == B.HCR_ERR_INVALID_ARG
    assert call(block_table=None) == B.HCR_ERR_INVALID_ARG
    assert call(max_blocks_per_req=0) == B.HCR_ERR_INVALID_ARG
    assert call(k_cache=None) == B.HCR_ERR_INVALID_ARG
    assert call(layout=None) == B.HCR_ERR_INVALID_ARG
    assert call(layout=B.hcr_cache_layout(lay.num_blocks, lay.block_size, 8)) == \
        B.HCR_ERR_INVALID_ARG
    assert call(workspace=None) == B.HCR_ERR_WORKSPACE
    assert call(workspace_bytes=16) == B.HCR_ERR_WORKSPACE
    assert call(workspace=ws.data_ptr() + 16) == B.HCR_ERR_WORKSPACE
    assert call(handle=None) == B.HCR_ERR_INVALID_ARG
    torch.cuda.synchronize()
    # nothing was launched: the caches still hold only sentinels
    assert bool((case.k_cache.view(torch.int16) == G.SENTINEL_BITS).all())
    assert call() == B.HCR_OK


def test_variant_policy_decisions(cuda_device):
    """The automatic tile variant on the cases it was measured on."""
    from kv_cache_restoration_gb300 import Restorer, binding as B, make_dims
    from workloads import generate as G
    from workloads.configs import LLAMA2_7B, LLAMA2_13B

    def handle(shape):
        # a 1-layer handle of the shape: the policy reads dims, not weights
        params = [G.layer_params(shape, 0, 0, cuda_device)]
        return Restorer(make_dims(1, shape.d_model, shape.n_heads, shape.n_kv_heads,
                                  shape.head_dim, shape.norm, shape.norm_eps, shape.rope,
                                  shape.rope_theta, 16384, shape.dtype, shape.kv_bias), params)
    r7 = handle(LLAMA2_7B)
    h = r7.handle
    # weight rows as M (3) for 257..320 tokens, where token-row tiles pad most
    want = {(64, 32): 1, (128, 32): 1, (256, 32): 2, (257, 32): 3, (300, 32): 3, (320, 32): 3,
            (321, 32): 2, (500, 32): 2, (794, 32): 2, (4096, 32): 2, (4096, 4): 2,
            (16384, 32): 1, (629259, 8): 1}
    assert {k: B.hcr_project_variant(h, *k) for k in want} == want
    assert B.hcr_project_variant(h, 0, 32) == 0
    assert B.hcr_debug_set_variant(h, 2) == 0
    assert B.hcr_project_variant(h, 16384, 32) == 2
    assert B.hcr_debug_set_variant(h, 1) == 0
    assert B.hcr_project_variant(h, 4096, 32) == 1
    r13 = handle(LLAMA2_13B)
    assert B.hcr_project_variant(r13.handle, 4096, 40) == 1     # d_model 5120
    assert B.hcr_project_variant(r13.handle, 300, 40) == 3
    # shorter calls of the wider models: pairs up to 6.5 TFLOP, unless the
    # pairs would end in a half tail tile
    assert B.hcr_project_variant(r13.handle, 256, 40) == 2
    assert B.hcr_project_variant(r13.handle, 512, 40) == 2
    assert B.hcr_project_variant(r13.handle, 400, 40) == 2
    assert B.hcr_project_variant(r13.handle, 1536, 40) == 2      # 6.4 TFLOP
    assert B.hcr_project_variant(r13.handle, 384, 40) == 1       # half tail
    assert B.hcr_project_variant(r13.handle, 513, 40) == 1       # half tail
    assert B.hcr_project_variant(r13.handle, 2048, 40) == 1      # 8.6 TFLOP
    assert B.hcr_debug_set_variant(h, 3) == 0
    assert B.hcr_project_variant(h, 4096, 32) == 3


# More weight-row tiles than CTA pairs: 2 layers x 40 head pairs = 80 tiles of
# 300 tokens on 76 pairs, so the last 4 tiles run as two half-chunk units each
# (160 + 144 tokens).  With two layers of 512 inputs the oracle checks every
# element.
SPLIT_TAIL = Workload("split-tail", ModelShape("st", 2, 512, 40, 40, 128), (300,), (11,))


def test_weight_rows_with_split_tail_units(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    a = Hn.make_case(SPLIT_TAIL, cuda_device)
    assert B.hcr_project_variant(a.restorer.handle, 300, 2) == 3
    Hn.run(a)
    assert a.status == 0, (a.status, a.flags)
    Hn.compare(a)
    b = Hn.make_case(SPLIT_TAIL, cuda_device, params=a.params, restorer=a.restorer)
    assert B.hcr_debug_set_variant(b.restorer.handle, 2) == 0
    Hn.run(b)
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c


# The three-slot TMEM layout for chunks of 257..320 tokens: two big slots taken
# in turn and a small slot for each tile's first columns.  Each token count
# gives a different split of its chunk (big + small columns): 257 -> 272 =
# 224 + 48, 288 = 224 + 64, 300 -> 304 = 192 + 112, 320 = 192 + 128.  Four
# layers of 40 head pairs are 160 tiles on 76 pairs, so every pair runs two or
# three units in turn (both big slots, the small slot reused) and the last 8
# tiles split in halves.
RING3_TOKENS = [257, 288, 300, 320]


@pytest.mark.parametrize("n_tokens", RING3_TOKENS)
def test_weight_rows_three_slot_layout(cuda_device, n_tokens):
    from kv_cache_restoration_gb300 import binding as B
    w = Workload(f"ring3-{n_tokens}", ModelShape("r3", 4, 512, 40, 40, 128), (n_tokens,), (5,),
                 block_order="shuffled")
    a = Hn.make_case(w, cuda_device)
    assert B.hcr_project_variant(a.restorer.handle, n_tokens, 4) == 3
    Hn.run(a)
    assert a.status == 0, (a.status, a.flags)
    Hn.compare(a)
    b = Hn.make_case(w, cuda_device, params=a.params, restorer=a.restorer)
    assert B.hcr_debug_set_variant(b.restorer.handle, 2) == 0
    Hn.run(b)
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c


# CTA pairs over several rounds of the persistent grid, with a half tail tile
# per layer: 4 layers x 32 n-tiles x 4 m-tiles (794 tokens) = 512 tiles, and x
# 2 m-tiles (384 tokens) = 256 tiles, on 76 pairs, so every pair runs several
# tiles and the last round is partial.  Each pair's place in a round rotates,
# so its tiles mix full and half tail m-tiles.
@pytest.mark.parametrize("n_tokens", [794, 384])
def test_pair_rounds_with_half_tails(cuda_device, n_tokens):
    from kv_cache_restoration_gb300 import binding as B
    w = Workload(f"rounds-{n_tokens}", ModelShape("rd", 4, 512, 32, 32, 128), (n_tokens,), (3,),
                 block_order="shuffled")
    a = Hn.make_case(w, cuda_device)
    assert B.hcr_debug_set_variant(a.restorer.handle, 2) == 0
    Hn.run(a)
    assert a.status == 0, (a.status, a.flags)
    Hn.compare(a)
    b = Hn.make_case(w, cuda_device, params=a.params, restorer=a.restorer)
    assert B.hcr_debug_set_variant(b.restorer.handle, 1) == 0
    Hn.run(b)
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c


# Norm statistics fused into the token-row projection: the same bits as the
# prepare kernel's.  Each case runs twice on the same inputs: with the
# workspace hcr_workspace_bytes asks for (the projection's statistics warps
# compute layers L0.. and each epilogue waits for its rows' flags) and with one
# byte less (the prepare kernel computes every layer).  Cases: CTA pairs with
# a half tail tile, pairs with a 232-row last tile, single CTAs with
# LayerNorm, fp16 and K/V bias, and a ragged GQA batch.
FUSED_CASES = [
    (W("fused-pairs-ht", ModelShape("fh", 6, 512, 32, 32, 128), [794], [0]), 2),
    (W("fused-pairs", ModelShape("fp", 6, 512, 32, 32, 128), [1000], [7],
       block_order="shuffled"), 2),
    (W("fused-single-ln", ModelShape("fs", 10, 512, 32, 32, 128, norm="ln", dtype="fp16",
                                     kv_bias=True), [130, 70], [0, 33]), 1),
    (W("fused-gqa", ModelShape("fg", 8, 1024, 64, 16, 128), [300, 5, 411, 64], [3, 0, 40, 9],
       block_order="shuffled"), 2),
    # LayerNorm rows with large means and outlier channels (the two-pass
    # statistics where one pass would cancel)
    (replace(W("fused-ln-means", ModelShape("fm", 10, 512, 32, 32, 128, norm="ln", dtype="fp16",
                                            kv_bias=True), [150, 50], [0, 7]),
             hidden_means=(-50.0, 10.0, 100.0), outlier_channels=(0, 17, 170, 511),
             outlier_scale=50.0), 1),
]


@pytest.mark.parametrize("w,variant", FUSED_CASES, ids=[c[0].name for c in FUSED_CASES])
def test_fused_statistics_match_prepare(cuda_device, w, variant):
    from kv_cache_restoration_gb300 import binding as B
    s = w.shape
    T = w.n_tokens
    a = Hn.make_case(w, cuda_device)
    assert B.hcr_debug_set_variant(a.restorer.handle, variant) == 0
    ws = a.restorer.workspace(T, s.n_layers, cuda_device)
    layer0 = B.hcr_debug_fused_stats(a.restorer.handle, T, s.n_layers, ws.numel())
    assert 1 <= layer0 < s.n_layers, layer0
    assert B.hcr_debug_fused_stats(a.restorer.handle, T, s.n_layers, ws.numel() - 1) == 0
    lay = a.layout
    a.restorer.restore(a.hidden, 0, s.n_layers, a.cu, a.start, a.table, a.k_cache, a.v_cache,
                       lay.num_blocks, lay.block_size, workspace=ws)
    a.status, a.flags = a.restorer.check()
    assert a.status == 0, (a.status, a.flags)
    Hn.compare(a)
    b = Hn.make_case(w, cuda_device, params=a.params, restorer=a.restorer)
    b.restorer.restore(b.hidden, 0, s.n_layers, b.cu, b.start, b.table, b.k_cache, b.v_cache,
                       lay.num_blocks, lay.block_size, workspace=ws[:ws.numel() - 1])
    b.status, b.flags = b.restorer.check()
    assert b.status == 0, (b.status, b.flags)
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c

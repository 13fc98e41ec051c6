"""hcr_restore_encoded (GPU): the restore that decodes the codec's int8 form
inside its kernels, against hcr_decode_hidden followed by hcr_restore, bit for
bit, and against the oracle restoring the decoded rows.

The codec is the HCache episode's proposal ("Fast State Restoration for
Evicted LLM KV Caches", cues 30 and 32) of compressing hidden states the way
the CacheGen review describes for KV (section 核心方法: groups of 10 tokens,
an 8-bit anchor, deltas quantised with layer-third bins).  The projection's
converter warps decode a run of 8 rows per lane and fetch a group anchor that
lies before the CTA's rows from global memory, so the cases put group and
request boundaries at every offset from a tile edge: ragged requests, group
sizes 1, 3, 10 and 25, half-tail and full-tail last tiles, a ragged last
k-block, and a layer subrange whose bins follow the model layer.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from tests import harness as Hn
from workloads import configs as C
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

CASES = [
    # ragged requests (an empty one, single tokens), shuffled blocks, 6 layers over 3 thirds
    Workload("enc-ragged", ModelShape("er", 6, 512, 4, 4, 128), (1, 200, 0, 77, 300, 13),
             (0, 5, 9, 1000, 31, 2), block_order="shuffled"),
    # LayerNorm, fp16, biases, no RoPE; 384 = 6 k-blocks; 260 tokens: half-tail last tile
    Workload("enc-ln-fp16", ModelShape("el", 3, 384, 3, 3, 128, norm="ln", rope=False,
                                       dtype="fp16", kv_bias=True), (250, 10), (0, 40)),
    # GQA, 400 tokens: full-size last tile (144 rows)
    Workload("enc-gqa", ModelShape("eg", 2, 1024, 8, 2, 128), (400,), (17,)),
    # 64-wide heads; d_model 336 = 5.25 k-blocks (ragged last k-block)
    Workload("enc-dh64-ragged-k", ModelShape("ed", 2, 336, 4, 4, 64), (129, 131), (3, 0)),
    # 256-wide heads (no half tail), 300 tokens
    Workload("enc-dh256", ModelShape("e2", 2, 512, 2, 2, 256), (300,), (7,)),
]


def _encode_decode(case, params):
    r = case.restorer
    n_req = int(case.start.numel())
    codes, scales = r.encode(case.hidden, case.layer_begin, case.layer_end, case.cu, n_req,
                             bins=params[0], group_tokens=params[1])
    dec = r.decode(codes, scales, case.layer_begin, case.layer_end, case.cu, n_req,
                   bins=params[0], group_tokens=params[1])
    torch.cuda.synchronize()
    assert r.check()[0] == 0
    return codes, scales, dec


def _restore_encoded(case, codes, scales, params):
    lay = case.layout
    case.restorer.restore_encoded(codes, scales, case.layer_begin, case.layer_end, case.cu,
                                  case.start, case.table, case.k_cache, case.v_cache,
                                  lay.num_blocks, lay.block_size, bins=params[0],
                                  group_tokens=params[1])
    case.status, case.flags = case.restorer.check()
    assert case.status == 0, (case.status, case.flags)


def _check(w, device, params=((0.5, 1.0, 1.5), 10), layer_begin=0, layer_end=None, oracle=True):
    """Fused restore == decode + restore (every cache bit, sentinels included),
    and the oracle on the decoded rows."""
    ref = Hn.make_case(w, device, layer_begin, layer_end)
    codes, scales, dec = _encode_decode(ref, params)
    fused = Hn.make_case(w, device, layer_begin, layer_end, params=ref.params,
                         restorer=ref.restorer)
    ref.hidden = dec
    Hn.run(ref)
    assert ref.status == 0
    _restore_encoded(fused, codes, scales, params)
    for c in ("k_cache", "v_cache"):
        got, want = getattr(fused, c).view(torch.int16), getattr(ref, c).view(torch.int16)
        assert torch.equal(got, want), c
    if oracle:
        fused.hidden = dec
        Hn.compare(fused)


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_encoded_restore_matches_decode_then_restore(cuda_device, w):
    _check(w, cuda_device)


@pytest.mark.parametrize("group", [1, 3, 25])
def test_encoded_restore_group_sizes(cuda_device, group):
    # 25: runs start up to 24 rows after their anchor, often before the CTA's rows
    _check(CASES[0], cuda_device, ((0.5, 1.0, 1.5), group), oracle=group == 25)


def test_encoded_restore_general_bins_and_layer_subrange(cuda_device):
    # bins with full binary32 significands; layers 1..4 of 6 use the model layer's third
    _check(CASES[0], cuda_device, ((0.3, 0.7, 1.9), 10), 1, 5)


def test_encoded_restore_large_row_means(cuda_device):
    # LayerNorm rows mean_row + N(0,1) with outlier channels: anchors carry the mean
    w = replace(CASES[1], hidden_means=(-50.0, 10.0, 100.0), outlier_channels=(0, 17, 200),
                outlier_scale=50.0)
    _check(w, cuda_device, ((0.5, 1.0, 1.5), 10))


def test_encoded_restore_full_size_7b(cuda_device):
    """The bench's workload (Llama2-7B shape, 4096 tokens, all 32 layers): every
    cache bit against decode + restore."""
    w = C.get("llama2-7b")
    params = ((0.5, 1.0, 1.5), 10)
    ref = Hn.make_case(w, cuda_device, gen_device=cuda_device)
    codes, scales, dec = _encode_decode(ref, params)
    ref.hidden = dec
    Hn.run(ref)
    assert ref.status == 0
    k_ref, v_ref = ref.k_cache, ref.v_cache
    fused = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer,
                         gen_device=cuda_device)
    del ref
    fused.hidden = None
    _restore_encoded(fused, codes, scales, params)
    assert torch.equal(fused.k_cache.view(torch.int16), k_ref.view(torch.int16))
    assert torch.equal(fused.v_cache.view(torch.int16), v_ref.view(torch.int16))
    # and a row sample of the last layer against the oracle
    fused.hidden = dec
    Hn.compare(fused, rows=Hn.sample_rows(w, 1 / 64), layers=[31], check_sentinel=False)


def test_encoded_restore_rejects_bad_arguments(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    w = CASES[0]
    case = Hn.make_case(w, cuda_device)
    lay = case.layout
    L, T, d = case.hidden.shape
    codes = torch.zeros((L, T, d), dtype=torch.int8, device=cuda_device)
    scales = torch.zeros((L, T), dtype=torch.float32, device=cuda_device)
    h = case.restorer.handle
    need = B.hcr_encoded_workspace_bytes(h, T, L)
    assert need > B.hcr_workspace_bytes(h, T, L)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    layout = B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0)

    def call(params=B.codec_params(), codes=codes, scales=scales, ws_bytes=need):
        return B.hcr_restore_encoded(h, params, codes, scales, 0, L, int(case.start.numel()), T,
                                     case.cu, case.start, case.table, lay.max_blocks,
                                     case.k_cache, case.v_cache, layout, ws, ws_bytes,
                                     torch.cuda.current_stream(), check=False)

    assert call(params=B.codec_params(group_tokens=0)) == B.HCR_ERR_INVALID_ARG
    assert call(params=B.codec_params((0.5, -1.0, 1.5))) == B.HCR_ERR_INVALID_ARG
    assert call(scales=None) == B.HCR_ERR_INVALID_ARG
    assert call(codes=codes.cpu().pin_memory()) == B.HCR_ERR_INVALID_ARG
    assert call(ws_bytes=B.hcr_workspace_bytes(h, T, L)) == B.HCR_ERR_WORKSPACE
    torch.cuda.synchronize()
    Hn.check_sentinels(case, np.zeros(0, dtype=np.int64))   # nothing was enqueued
    # d_model not a multiple of 16: the codes' rows cannot be TMA boxes
    w16 = Workload("enc-d8", ModelShape("e8", 1, 520, 4, 4, 128), (20,), (0,))
    c8 = Hn.make_case(w16, cuda_device)
    L8, T8, d8 = c8.hidden.shape
    st = B.hcr_restore_encoded(
        c8.restorer.handle, B.codec_params(), torch.zeros((L8, T8, d8), dtype=torch.int8,
                                                          device=cuda_device),
        torch.zeros((L8, T8), dtype=torch.float32, device=cuda_device), 0, L8, 1, T8, c8.cu,
        c8.start, c8.table, c8.layout.max_blocks, c8.k_cache, c8.v_cache,
        B.hcr_cache_layout(c8.layout.num_blocks, c8.layout.block_size, 0),
        torch.empty(1 << 20, dtype=torch.uint8, device=cuda_device), 1 << 20,
        torch.cuda.current_stream(), check=False)
    assert st == B.HCR_ERR_UNSUPPORTED


def test_stalled_encoded_pipeline_times_out_and_context_survives(cuda_device):
    """The stall hook withholds each CTA's first code load: the converters'
    wait (or the MMA's, or the code producer's for a stage that is never
    released) gives up after its time limit, the call reports HCR_ERR_TIMEOUT,
    and the next restore on the same handle is exact again."""
    import time

    from kv_cache_restoration_gb300 import binding as B
    w = Workload("enc-stall", ModelShape("es", 1, 256, 2, 2, 128), (300,), (2,))
    params = ((0.5, 1.0, 1.5), 10)
    ref = Hn.make_case(w, cuda_device)
    codes, scales, dec = _encode_decode(ref, params)
    h = ref.restorer.handle
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer)
    lay = case.layout
    assert B.hcr_debug_set_stall(h, True) == B.HCR_OK
    t0 = time.monotonic()
    case.restorer.restore_encoded(codes, scales, 0, 1, case.cu, case.start, case.table,
                                  case.k_cache, case.v_cache, lay.num_blocks, lay.block_size,
                                  check=False)
    status, flags = case.restorer.check()
    elapsed = time.monotonic() - t0
    assert status == B.HCR_ERR_TIMEOUT
    assert flags & B.HCR_DEVERR_TIMEOUT
    assert 1.5 < elapsed < 60.0
    st, rec = B.hcr_debug_timeout_record(h)
    assert st == B.HCR_OK
    # converters waiting for codes (9), the MMA for a stage (4), the code
    # producer for a stage release (8) or the epilogue for an accumulator (7)
    assert rec[0] in (4, 7, 8, 9), rec
    assert B.hcr_debug_set_stall(h, False) == B.HCR_OK
    ref.hidden = dec
    Hn.run(ref)
    again = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer)
    _restore_encoded(again, codes, scales, params)
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(again, c).view(torch.int16), getattr(ref, c).view(torch.int16))


# One layer of each benchmark workload at full size, one per layer third (bins
# 0.5 / 1.0 / 1.5): the 13B shape with shuffled blocks, OPT-30B (fp16,
# LayerNorm, biases, d = 7168), and the ragged batch of 64 requests, whose
# anchor groups restart at every request boundary.
FULL = [("llama2-13b", 20), ("opt-30b", 47), ("ragged-7b", 0)]


@pytest.mark.parametrize("name,layer", FULL, ids=[n for n, _ in FULL])
def test_encoded_restore_full_size_layer(cuda_device, name, layer):
    w = C.get(name)
    params = ((0.5, 1.0, 1.5), 10)
    ref = Hn.make_case(w, cuda_device, layer, layer + 1, gen_device=cuda_device)
    codes, scales, dec = _encode_decode(ref, params)
    ref.hidden = dec
    Hn.run(ref)
    assert ref.status == 0
    k_ref, v_ref = ref.k_cache, ref.v_cache
    fused = Hn.make_case(w, cuda_device, layer, layer + 1, params=ref.params,
                         restorer=ref.restorer, gen_device=cuda_device)
    del ref
    fused.hidden = None
    torch.cuda.empty_cache()
    _restore_encoded(fused, codes, scales, params)
    assert torch.equal(fused.k_cache.view(torch.int16), k_ref.view(torch.int16))
    assert torch.equal(fused.v_cache.view(torch.int16), v_ref.view(torch.int16))
    del k_ref, v_ref
    fused.hidden = dec
    Hn.compare(fused, rows=Hn.sample_rows(w, 1 / 256), check_sentinel=False)

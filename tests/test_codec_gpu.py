"""The hidden-state codec on the GPU against the oracle, bit for bit: codes,
anchor scales and decoded values (in the storage dtype), for both dtypes,
device and pinned-host encoded stores, layer subranges that cross the
layer-group boundaries, and the full 7B shape on whole layers."""
import numpy as np
import pytest
import torch

from oracle import codec as K
from tests import harness as Hn
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

W = Workload("codec", ModelShape("cd", 6, 512, 4, 4, 128), (1, 200, 0, 77, 300, 13),
             (0, 5, 9, 1000, 31, 2), block_order="shuffled")
W16 = Workload("codec16", ModelShape("cd16", 3, 384, 3, 3, 128, norm="ln", rope=False,
                                     dtype="fp16", kv_bias=True), (250, 10), (0, 40))


def _encode(case, params, pinned=False):
    from kv_cache_restoration_gb300 import binding as B
    L, T, d = case.hidden.shape
    codes = torch.zeros((L, T, d), dtype=torch.int8)
    scales = torch.full((L, T), -1.0, dtype=torch.float32)
    if pinned:
        codes, scales = codes.pin_memory(), scales.pin_memory()
    else:
        codes, scales = codes.to(case.hidden.device), scales.to(case.hidden.device)
    B.hcr_encode_hidden(case.restorer.handle, params, case.hidden, case.layer_begin,
                        case.layer_end, int(case.start.numel()), T, case.cu, codes, scales,
                        torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert case.restorer.check()[0] == 0
    return codes, scales


def _decode(case, params, codes, scales):
    from kv_cache_restoration_gb300 import binding as B
    out = torch.empty_like(case.hidden)
    B.hcr_decode_hidden(case.restorer.handle, params, codes, scales, case.layer_begin,
                        case.layer_end, int(case.start.numel()), case.hidden.shape[1], case.cu,
                        out, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert case.restorer.check()[0] == 0
    return out


def _oracle(case, bins=K.DEFAULT_BINS, group=K.GROUP_TOKENS):
    dt = case.w.shape.dtype
    hs = [Hn.widen(case.hidden[i], dt).astype(np.float32)
          for i in range(case.layer_end - case.layer_begin)]
    codes, scales = K.encode(hs, case.layer_begin, case.w.shape.n_layers,
                             case.layout.cu_seqlens, bins, group)
    dec = K.decode(codes, scales, case.layer_begin, case.w.shape.n_layers,
                   case.layout.cu_seqlens, bins, group)
    return codes, scales, K.round_to_storage(dec, dt)


def _check(case, params, pinned=False, bins=K.DEFAULT_BINS, group=K.GROUP_TOKENS):
    codes, scales = _encode(case, params, pinned)
    want_codes, want_scales, want_dec = _oracle(case, bins, group)
    assert np.array_equal(codes.cpu().numpy(), want_codes)
    anchors = K.group_anchors(case.layout.cu_seqlens, group)
    is_anchor = anchors == np.arange(len(anchors))
    got_s = scales.cpu().numpy()
    assert np.array_equal(got_s[:, is_anchor], want_scales[:, is_anchor])
    assert (got_s[:, ~is_anchor] == -1.0).all(), "scales of non-anchor rows must stay untouched"
    dec = _decode(case, params, codes, scales)
    assert np.array_equal(Hn.bits_of(dec), want_dec)


@pytest.mark.parametrize("pinned", [False, True], ids=["device-store", "host-store"])
def test_codec_matches_oracle_bf16(cuda_device, pinned):
    from kv_cache_restoration_gb300 import binding as B
    _check(Hn.make_case(W, cuda_device), B.codec_params(), pinned)


def test_codec_matches_oracle_fp16_and_other_params(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W16, cuda_device)
    _check(case, B.codec_params())
    bins, group = (0.03, 0.07, 0.11), 7
    _check(case, B.codec_params(bins, group), bins=bins, group=group)


def test_codec_layer_subrange_uses_model_layer_bins(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    # layers 1..4 of 6: bins 0.5 (layer 1), 1.0 (2, 3), 1.5 (4)
    _check(Hn.make_case(W, cuda_device, 1, 5), B.codec_params())


def test_codec_full_size_7b_whole_layers(cuda_device):
    """7B shape, 4096 tokens: every row of one layer from each layer group."""
    from kv_cache_restoration_gb300 import binding as B
    w = C.get("llama2-7b")
    for layer in (0, 16, 31):
        case = Hn.make_case(w, cuda_device, layer, layer + 1, gen_device=cuda_device)
        _check(case, B.codec_params())
        del case
        torch.cuda.empty_cache()


def test_codec_rejects_bad_params(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    L, T, d = case.hidden.shape
    codes = torch.zeros((L, T, d), dtype=torch.int8, device=cuda_device)
    scales = torch.zeros((L, T), dtype=torch.float32, device=cuda_device)
    for p in (B.codec_params((0.5, 0.0, 1.5)), B.codec_params((0.5, float("nan"), 1.5)),
              B.codec_params(group_tokens=0)):
        st = B.hcr_encode_hidden(case.restorer.handle, p, case.hidden, 0, L,
                                 int(case.start.numel()), T, case.cu, codes, scales,
                                 torch.cuda.current_stream(), check=False)
        assert st == B.HCR_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not codes.any()


def _streamed_encoded(case, params, codes_host, scales_host, chunk, slots, overlap=False):
    from kv_cache_restoration_gb300 import binding as B
    lay = case.layout
    T, d = case.w.n_tokens, case.w.shape.d_model
    nl = case.layer_end - case.layer_begin
    c = min(chunk, nl)
    nbytes = B.encoded_staging_bytes(T, d, c, slots)
    dev = case.k_cache.device
    staging = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
    ws_layers = c * (min(slots, 8) if overlap else 1)   # overlap: statistics per slot
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, ws_layers) + 256,
                     dtype=torch.uint8, device=dev)
    st = B.hcr_restore_streamed_encoded(
        case.restorer.handle, params, codes_host, scales_host, case.layer_begin, case.layer_end,
        int(case.start.numel()), T, case.cu, case.start, case.table, lay.max_blocks,
        case.k_cache, case.v_cache, B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0),
        staging, nbytes, chunk, ws, ws.numel(), torch.cuda.current_stream(), check=False)
    torch.cuda.synchronize()
    return st


def _reference_from_decoded(w, device, params, layer_begin=0, layer_end=None, gen_device=None):
    """Encode on the GPU, decode on the GPU, restore the decoded hidden states."""
    src = Hn.make_case(w, device, layer_begin, layer_end, gen_device=gen_device)
    codes, scales = _encode(src, params)
    src.hidden = _decode(src, params, codes, scales)
    Hn.run(src)
    return src, codes.cpu().pin_memory(), scales.cpu().pin_memory()


@pytest.mark.parametrize("overlap", [False, True], ids=["in-order", "side-stream-stats"])
@pytest.mark.parametrize("chunk,slots", [(1, 2), (2, 3), (4, 1), (6, 2)])
def test_streamed_encoded_matches_restore_of_decoded(cuda_device, chunk, slots, overlap):
    from kv_cache_restoration_gb300 import binding as B
    params = B.codec_params()
    ref, codes_h, scales_h = _reference_from_decoded(W, cuda_device, params)
    case = Hn.make_case(W, cuda_device, params=ref.params, restorer=ref.restorer)
    assert _streamed_encoded(case, params, codes_h, scales_h, chunk, slots, overlap) == 0
    assert case.restorer.check()[0] == 0
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(case, c).view(torch.int16), getattr(ref, c).view(torch.int16))


def test_streamed_encoded_layer_subrange_and_full_7b(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    params = B.codec_params()
    ref, codes_h, scales_h = _reference_from_decoded(W, cuda_device, params, 2, 6)
    case = Hn.make_case(W, cuda_device, 2, 6, params=ref.params, restorer=ref.restorer)
    assert _streamed_encoded(case, params, codes_h, scales_h, 3, 2) == 0
    assert torch.equal(case.k_cache.view(torch.int16), ref.k_cache.view(torch.int16))
    del ref, case
    w = C.get("llama2-7b")
    ref, codes_h, scales_h = _reference_from_decoded(w, cuda_device, params,
                                                     gen_device=cuda_device)
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer,
                        gen_device=cuda_device)
    assert _streamed_encoded(case, params, codes_h, scales_h, 4, 3, overlap=True) == 0
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(case, c).view(torch.int16), getattr(ref, c).view(torch.int16))


def test_streamed_encoded_rejects_small_staging(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    params = B.codec_params()
    case = Hn.make_case(W, cuda_device)
    lay = case.layout
    T, d = W.n_tokens, W.shape.d_model
    need = B.encoded_staging_bytes(T, d, 2, 1)
    staging = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    ws = torch.empty(1 << 22, dtype=torch.uint8, device=cuda_device)
    codes = torch.zeros((6, T, d), dtype=torch.int8).pin_memory()
    scales = torch.zeros((6, T), dtype=torch.float32).pin_memory()
    st = B.hcr_restore_streamed_encoded(
        case.restorer.handle, params, codes, scales, 0, 6, int(case.start.numel()), T, case.cu,
        case.start, case.table, lay.max_blocks, case.k_cache, case.v_cache,
        B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0), staging, need - 256, 2, ws,
        ws.numel(), torch.cuda.current_stream(), check=False)
    assert st == B.HCR_ERR_WORKSPACE


def test_streamed_encoded_rejects_bad_params_before_enqueueing(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    lay = case.layout
    T, d = W.n_tokens, W.shape.d_model
    need = B.encoded_staging_bytes(T, d, 2, 2)
    staging = torch.full((need,), 0x5A, dtype=torch.uint8, device=cuda_device)
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, 2) + 256, dtype=torch.uint8,
                     device=cuda_device)
    codes = torch.ones((6, T, d), dtype=torch.int8).pin_memory()
    scales = torch.ones((6, T), dtype=torch.float32).pin_memory()
    for p in (B.codec_params((0.5, 0.0, 1.5)), B.codec_params(group_tokens=0)):
        st = B.hcr_restore_streamed_encoded(
            case.restorer.handle, p, codes, scales, 0, 6, int(case.start.numel()), T, case.cu,
            case.start, case.table, lay.max_blocks, case.k_cache, case.v_cache,
            B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0), staging, need, 2, ws,
            ws.numel(), torch.cuda.current_stream(), check=False)
        assert st == B.HCR_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((staging == 0x5A).all())          # no copy was enqueued
    assert bool((case.k_cache.view(torch.int16) == G.SENTINEL_BITS).all())

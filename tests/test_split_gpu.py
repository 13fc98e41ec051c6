"""The KV-offload side and the layer-split restore on the GPU.

* hcr_load_kv / hcr_save_kv against the oracle's placement, bit for bit
  (dense store in device memory and in pinned host memory);
* hcr_restore_streamed_split: hidden states for the lower layers, saved K/V
  for the upper ones, gives bit for bit the caches of hcr_restore over all
  layers, for every split, group size and staging ring tried;
* hcr_profile_layer_costs gives positive per-layer costs that the planner
  turns into a split.
"""
import numpy as np
import pytest
import torch

from oracle import split as SP
from tests import harness as Hn
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

W = Workload("kv", ModelShape("kv", 5, 512, 4, 4, 128), (1, 200, 0, 77, 300),
             (0, 5, 9, 1000, 31), block_order="shuffled", spare_blocks=3)


def _flat_bits(cache):
    """[L][num_blocks][B][H][dh] -> numpy uint16 [L][num_blocks * B][H * dh]."""
    b = Hn.bits_of(cache)
    return b.reshape(b.shape[0], b.shape[1] * b.shape[2], -1)


def _kv_call(fn, case, kv, layer_begin=None, layer_end=None, check=True):
    from kv_cache_restoration_gb300 import binding as B
    lay = case.layout
    lb = case.layer_begin if layer_begin is None else layer_begin
    le = case.layer_end if layer_end is None else layer_end
    T = case.w.n_tokens
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, 1) + 256, dtype=torch.uint8,
                     device=case.k_cache.device)
    st = fn(case.restorer.handle, kv, lb, le, int(case.start.numel()), T, case.cu, case.start,
            case.table, lay.max_blocks, case.k_cache, case.v_cache,
            B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0), ws, ws.numel(),
            torch.cuda.current_stream(), check=check)
    torch.cuda.synchronize()
    return st


def _dense_shape(case, n_layers):
    s = case.w.shape
    return (n_layers, 2, case.w.n_tokens, s.n_kv_heads * s.head_dim)


@pytest.mark.parametrize("pinned", [False, True], ids=["device-store", "host-store"])
def test_load_kv_matches_oracle_placement(cuda_device, pinned):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    L = case.layer_end - case.layer_begin
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 0x7F00, _dense_shape(case, L), dtype=np.uint16)
    kv = torch.from_numpy(bits.view(np.int16))
    kv = kv.pin_memory() if pinned else kv.to(cuda_device)
    before_k, before_v = _flat_bits(case.k_cache), _flat_bits(case.v_cache)
    assert _kv_call(B.hcr_load_kv, case, kv) == 0
    assert case.restorer.check()[0] == 0
    lay = case.layout
    want_k, want_v = SP.kv_rows_to_cache(bits, before_k, before_v, lay.cu_seqlens, lay.start_pos,
                                         lay.block_table, lay.block_size)
    assert np.array_equal(_flat_bits(case.k_cache), want_k)
    assert np.array_equal(_flat_bits(case.v_cache), want_v)


@pytest.mark.parametrize("pinned", [False, True], ids=["device-store", "host-store"])
def test_save_kv_matches_oracle(cuda_device, pinned):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.run(Hn.make_case(W, cuda_device))
    L = case.layer_end - case.layer_begin
    kv = torch.full(_dense_shape(case, L), G.SENTINEL_BITS, dtype=torch.int16)
    kv = kv.pin_memory() if pinned else kv.to(cuda_device)
    assert _kv_call(B.hcr_save_kv, case, kv) == 0
    lay = case.layout
    want = SP.kv_rows_from_cache(_flat_bits(case.k_cache), _flat_bits(case.v_cache),
                                 lay.cu_seqlens, lay.start_pos, lay.block_table, lay.block_size)
    assert np.array_equal(kv.cpu().numpy().view(np.uint16), want)


def test_save_then_load_round_trip_on_a_layer_subrange(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    ref = Hn.run(Hn.make_case(W, cuda_device))
    kv = torch.empty(_dense_shape(ref, 2), dtype=torch.int16, device=cuda_device)
    # layers 2..3 of the model: cache bases offset to layer 2
    sub = Hn.make_case(W, cuda_device, 2, 4, params=ref.params, restorer=ref.restorer)
    sub.k_cache, sub.v_cache = ref.k_cache[2:4], ref.v_cache[2:4]
    assert _kv_call(B.hcr_save_kv, sub, kv) == 0
    fresh = Hn.make_case(W, cuda_device, 2, 4, params=ref.params, restorer=ref.restorer)
    assert _kv_call(B.hcr_load_kv, fresh, kv) == 0
    assert torch.equal(fresh.k_cache.view(torch.int16), ref.k_cache[2:4].view(torch.int16))
    assert torch.equal(fresh.v_cache.view(torch.int16), ref.v_cache[2:4].view(torch.int16))


def _split_restore(case, hidden_host, kv_host, split, chunk, slots, check=False,
                   overlap=False):
    from kv_cache_restoration_gb300 import binding as B
    lay = case.layout
    s = case.w.shape
    T = case.w.n_tokens
    n_hid = split - case.layer_begin
    ch = max(1, min(chunk, n_hid))
    slot_bytes = max(ch * T * s.d_model * 2 if n_hid else 0,
                     2 * T * s.n_kv_heads * s.head_dim * 2 if case.layer_end > split else 0)
    dev = case.k_cache.device
    staging = torch.empty(slots * slot_bytes + 256, dtype=torch.uint8, device=dev)
    # overlap: statistics room for every slot's hidden-state group (side stream)
    ws_layers = ch * (min(slots, 8) if overlap else 1)
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, ws_layers) + 256,
                     dtype=torch.uint8, device=dev)
    st = B.hcr_restore_streamed_split(
        case.restorer.handle, hidden_host, kv_host, case.layer_begin, split, case.layer_end,
        int(case.start.numel()), T, case.cu, case.start, case.table, lay.max_blocks,
        case.k_cache, case.v_cache, B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0),
        staging, slots * slot_bytes, chunk, ws, ws.numel(), torch.cuda.current_stream(),
        check=check)
    torch.cuda.synchronize()
    return st


def _saved_kv_host(ref, layer_begin, layer_end):
    from kv_cache_restoration_gb300 import binding as B
    n = layer_end - layer_begin
    if n == 0:
        return None
    kv = torch.empty(_dense_shape(ref, n), dtype=torch.int16).pin_memory()
    if n:
        sub = Hn.make_case(ref.w, ref.k_cache.device, layer_begin, layer_end, params=ref.params,
                           restorer=ref.restorer)
        sub.k_cache = ref.k_cache[layer_begin - ref.layer_begin:layer_end - ref.layer_begin]
        sub.v_cache = ref.v_cache[layer_begin - ref.layer_begin:layer_end - ref.layer_begin]
        assert _kv_call(B.hcr_save_kv, sub, kv) == 0
    return kv


def _same(a, b):
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c


@pytest.mark.parametrize("split,chunk,slots", [(0, 2, 2), (1, 1, 2), (3, 2, 3), (4, 4, 1),
                                               (5, 2, 2), (2, 9, 3)])
def test_streamed_split_matches_restore(cuda_device, split, chunk, slots):
    ref = Hn.run(Hn.make_case(W, cuda_device))
    kv_host = _saved_kv_host(ref, split, 5)
    hidden_host = ref.hidden[:split].cpu().pin_memory() if split else None
    case = Hn.make_case(W, cuda_device, params=ref.params, restorer=ref.restorer)
    overlap = slots > 2   # side-stream statistics for the 3-slot cases
    assert _split_restore(case, hidden_host, kv_host, split, chunk, slots, overlap=overlap) == 0
    assert case.restorer.check()[0] == 0
    _same(case, ref)


def test_streamed_split_layer_subrange(cuda_device):
    ref = Hn.run(Hn.make_case(W, cuda_device, 1, 5))
    kv_host = _saved_kv_host(ref, 3, 5)
    hidden_host = ref.hidden[:2].cpu().pin_memory()
    case = Hn.make_case(W, cuda_device, 1, 5, params=ref.params, restorer=ref.restorer)
    assert _split_restore(case, hidden_host, kv_host, 3, 2, 2) == 0
    _same(case, ref)
    Hn.compare(case)


def test_streamed_split_full_size_7b(cuda_device):
    w = C.get("llama2-7b")
    ref = Hn.run(Hn.make_case(w, cuda_device, gen_device=cuda_device))
    kv_host = _saved_kv_host(ref, 28, 32)
    hidden_host = ref.hidden[:28].cpu().pin_memory()
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer,
                        gen_device=cuda_device)
    assert _split_restore(case, hidden_host, kv_host, 28, 4, 3, overlap=True) == 0
    _same(case, ref)


def test_streamed_split_rejects_bad_ranges(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    h = case.hidden.cpu().pin_memory()
    for lb, sp, le in [(2, 1, 5), (0, 6, 5), (0, 3, 6)]:
        case.layer_begin, case.layer_end = lb, le
        assert _split_restore(case, h, h, sp, 2, 2) == B.HCR_ERR_INVALID_ARG
    case.layer_begin, case.layer_end = 0, 5
    assert _split_restore(case, h, None, 3, 2, 2) == B.HCR_ERR_INVALID_ARG
    assert bool((case.k_cache.view(torch.int16) == G.SENTINEL_BITS).all())


def test_profile_and_plan(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    c = B.hcr_profile_layer_costs(case.restorer.handle, 512, 2, 2, torch.cuda.current_stream())
    for f in ("restore_s", "hidden_copy_s", "kv_copy_s", "kv_place_s"):
        assert 0 < getattr(c, f) < 1.0, f
    assert case.restorer.check()[0] == 0
    plan = B.hcr_plan_layer_split(c, 5)
    want = SP.plan_layer_split(SP.LayerCosts(c.restore_s, c.hidden_copy_s, c.kv_copy_s,
                                             c.kv_place_s), 5)
    assert (plan.hidden_layers, plan.kv_layers) == (want.hidden_layers, want.kv_layers)

"""hcr_restore_streamed_chunks: the restore half of the chunk store.  Layer
inputs saved by hcr_save_hidden into a pinned host store, then restored
straight from it with the layer-pipelined restore, give bit for bit the
caches hcr_restore gives from the original hidden states in HBM."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from tests import harness as Hn
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu


def _chunk_table(w, chunk_tokens, order=None):
    lay = G.request_layout(replace(w, block_size=chunk_tokens,
                                   block_order=order or w.block_order))
    return lay.block_table, lay.num_blocks


def _save_to_host(case, chunk_tokens, order=None):
    """Saves the case's layer inputs into a fresh pinned host chunk store."""
    from kv_cache_restoration_gb300 import binding as B
    table_np, n = _chunk_table(case.w, chunk_tokens, order)
    s = case.w.shape
    store = torch.full((n, s.n_layers, chunk_tokens, s.d_model), G.SENTINEL_BITS,
                       dtype=torch.int16).pin_memory()
    table = torch.as_tensor(table_np, device=case.hidden.device)
    B.hcr_save_hidden(case.restorer.handle, case.hidden, case.layer_begin, case.layer_end,
                      int(case.start.numel()), int(case.hidden.shape[1]), case.cu, case.start,
                      table, int(table.shape[1]), chunk_tokens, store, n,
                      torch.cuda.current_stream())
    torch.cuda.synchronize()
    return store, np.ascontiguousarray(table_np, dtype=np.int32), n


def _source(store, chunk_tokens, n, table_np, lay):
    from kv_cache_restoration_gb300 import binding as B
    cu = np.ascontiguousarray(lay.cu_seqlens, dtype=np.int32)
    start = np.ascontiguousarray(lay.start_pos, dtype=np.int32)
    src = B.hcr_chunk_source(store.data_ptr(), chunk_tokens, n, table_np.ctypes.data,
                             int(table_np.shape[1]), cu.ctypes.data, start.ctypes.data)
    src._keep = (store, table_np, cu, start)       # the host arrays outlive the call
    return src


def _restore_chunks(case, src, chunk, slots, check=False, overlap=False):
    from kv_cache_restoration_gb300 import binding as B
    lay = case.layout
    T, d = case.w.n_tokens, case.w.shape.d_model
    nl = case.layer_end - case.layer_begin
    chunk_bytes = min(chunk, nl) * T * d * 2
    dev = case.k_cache.device
    staging = torch.empty(slots * chunk_bytes + 256, dtype=torch.uint8, device=dev)
    # overlap: statistics room for every slot's group (computed on the side stream)
    ws_layers = min(chunk, nl) * (min(slots, 8) if overlap else 1)
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, ws_layers) + 256,
                     dtype=torch.uint8, device=dev)
    st = B.hcr_restore_streamed_chunks(
        case.restorer.handle, src, case.layer_begin, case.layer_end, int(case.start.numel()), T,
        case.cu, case.start, case.table, lay.max_blocks, case.k_cache, case.v_cache,
        B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0), staging, slots * chunk_bytes,
        chunk, ws, ws.numel(), torch.cuda.current_stream(), check=check)
    torch.cuda.synchronize()
    return st


def _same(a, b):
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c


W = Workload("sc", ModelShape("sc", 5, 512, 4, 4, 128), (1, 200, 0, 77, 300),
             (0, 5, 9, 1000, 31), block_order="shuffled", spare_blocks=3)


# Shuffled chunk ids make one copy per chunk; consecutive ids ("contiguous")
# make spans, copied per layer when a span outnumbers the group's layers.
@pytest.mark.parametrize("order", ["shuffled", "contiguous"])
@pytest.mark.parametrize("chunk_tokens", [64, 16, 1])
@pytest.mark.parametrize("chunk,slots", [(1, 2), (2, 3), (5, 1)])
def test_restore_from_chunk_store_matches_restore(cuda_device, chunk_tokens, chunk, slots,
                                                  order):
    ref = Hn.run(Hn.make_case(W, cuda_device))
    store, table_np, n = _save_to_host(ref, chunk_tokens, order)
    case = Hn.make_case(W, cuda_device, params=ref.params, restorer=ref.restorer)
    src = _source(store, chunk_tokens, n, table_np, case.layout)
    overlap = chunk_tokens == 16   # one third of the cases with side-stream statistics
    assert _restore_chunks(case, src, chunk, slots, overlap=overlap) == 0
    assert case.restorer.check()[0] == 0
    _same(case, ref)


def test_restore_from_chunk_store_layer_subrange(cuda_device):
    ref = Hn.run(Hn.make_case(W, cuda_device, 1, 4))
    store, table_np, n = _save_to_host(ref, 64)
    case = Hn.make_case(W, cuda_device, 1, 4, params=ref.params, restorer=ref.restorer)
    assert _restore_chunks(case, _source(store, 64, n, table_np, case.layout), 2, 2) == 0
    _same(case, ref)
    Hn.compare(case)


def test_restore_from_chunk_store_full_size_7b(cuda_device):
    w = C.get("llama2-7b")
    ref = Hn.run(Hn.make_case(w, cuda_device, gen_device=cuda_device))
    store, table_np, n = _save_to_host(ref, 64)
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer,
                        gen_device=cuda_device)
    assert _restore_chunks(case, _source(store, 64, n, table_np, case.layout), 4, 3,
                           overlap=True) == 0
    _same(case, ref)


def test_bad_chunk_table_is_rejected_on_the_host(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    ref = Hn.run(Hn.make_case(W, cuda_device))
    store, table_np, n = _save_to_host(ref, 64)
    case = Hn.make_case(W, cuda_device, params=ref.params, restorer=ref.restorer)
    bad = table_np.copy()
    bad[4, 1] = n + 5
    assert _restore_chunks(case, _source(store, 64, n, bad, case.layout), 2, 2) == \
        B.HCR_ERR_INVALID_ARG
    short = np.ascontiguousarray(table_np[:, :1])    # request 4 runs past its first chunk
    assert _restore_chunks(case, _source(store, 64, n, short, case.layout), 2, 2) == \
        B.HCR_ERR_INVALID_ARG
    assert bool((case.k_cache.view(torch.int16) == G.SENTINEL_BITS).all())
    assert bool((case.v_cache.view(torch.int16) == G.SENTINEL_BITS).all())

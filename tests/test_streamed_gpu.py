"""hcr_restore_streamed (the layer-pipelined restore from host memory) gives
bit for bit the caches hcr_restore gives from the same hidden states in HBM,
for any chunking and staging ring, including a single slot."""
import pytest
import torch

from tests import harness as Hn
from workloads import configs as C
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu


def _streamed(case, chunk, slots, stream=None, pinned=True, overlap=False):
    """overlap: a workspace with statistics room for every slot's group, so the
    statistics run on the handle's side stream; otherwise room for one group."""
    from kv_cache_restoration_gb300 import binding as B
    lay = case.layout
    T, d = case.w.n_tokens, case.w.shape.d_model
    nl = case.layer_end - case.layer_begin
    host = case.hidden.cpu()
    if pinned:
        host = host.pin_memory()
    chunk_bytes = min(chunk, nl) * T * d * 2
    staging = torch.empty(slots * chunk_bytes + 256, dtype=torch.uint8, device=case.hidden.device)
    ws_layers = min(chunk, nl) * (min(slots, 8) if overlap else 1)
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, ws_layers) + 256,
                     dtype=torch.uint8, device=case.hidden.device)
    st = B.hcr_restore_streamed(case.restorer.handle, host, case.layer_begin, case.layer_end,
                                int(case.start.numel()), T, case.cu, case.start, case.table,
                                lay.max_blocks, case.k_cache, case.v_cache,
                                B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0), staging,
                                slots * chunk_bytes, chunk, ws, ws.numel(),
                                stream or torch.cuda.current_stream(), check=False)
    torch.cuda.synchronize()
    return st


def _same(a, b):
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c


W4 = Workload("st4", ModelShape("st4", 5, 512, 4, 4, 128), (1, 200, 0, 77, 300),
              (0, 5, 9, 1000, 31), block_order="shuffled", spare_blocks=3)


@pytest.mark.parametrize("overlap", [False, True], ids=["in-order", "side-stream-stats"])
@pytest.mark.parametrize("chunk,slots", [(1, 2), (2, 2), (2, 3), (3, 1), (5, 8), (9, 2)])
def test_streamed_matches_restore(cuda_device, chunk, slots, overlap):
    ref = Hn.run(Hn.make_case(W4, cuda_device))
    assert ref.status == 0
    case = Hn.make_case(W4, cuda_device, params=ref.params, restorer=ref.restorer)
    assert _streamed(case, chunk, slots, overlap=overlap) == 0
    assert case.restorer.check()[0] == 0
    _same(case, ref)


# LayerNorm (mean and rstd per row), fp16, biases
WLN = Workload("stln", ModelShape("stln", 4, 384, 3, 3, 128, norm="ln", rope=False,
                                  dtype="fp16", kv_bias=True), (250, 10), (0, 40))


@pytest.mark.parametrize("overlap", [False, True], ids=["in-order", "side-stream-stats"])
def test_streamed_layernorm(cuda_device, overlap):
    ref = Hn.run(Hn.make_case(WLN, cuda_device))
    case = Hn.make_case(WLN, cuda_device, params=ref.params, restorer=ref.restorer)
    assert _streamed(case, 1, 3, overlap=overlap) == 0
    _same(case, ref)
    Hn.compare(case)


def test_streamed_layer_subrange_and_pageable_host(cuda_device):
    ref = Hn.run(Hn.make_case(W4, cuda_device, 1, 4))
    case = Hn.make_case(W4, cuda_device, 1, 4, params=ref.params, restorer=ref.restorer)
    assert _streamed(case, 2, 2, pinned=False) == 0
    _same(case, ref)
    Hn.compare(case)


def test_streamed_full_size_7b(cuda_device):
    w = C.get("llama2-7b")
    ref = Hn.run(Hn.make_case(w, cuda_device, gen_device=cuda_device))
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer,
                        gen_device=cuda_device)
    assert _streamed(case, 4, 3, overlap=True) == 0
    _same(case, ref)


def test_streamed_rejects_small_buffers(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W4, cuda_device)
    lay = case.layout
    host = case.hidden.cpu()
    T, d = W4.n_tokens, W4.shape.d_model
    staging = torch.empty(T * d * 2, dtype=torch.uint8, device=cuda_device)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=cuda_device)
    layout = B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0)
    args = (case.restorer.handle, host, 0, 5, 5, T, case.cu, case.start, case.table,
            lay.max_blocks, case.k_cache, case.v_cache, layout)
    # a 2-layer chunk does not fit a 1-layer staging buffer
    assert B.hcr_restore_streamed(*args, staging, staging.numel(), 2, ws, ws.numel(),
                                  check=False) == B.HCR_ERR_WORKSPACE
    # workspace too small for one chunk
    assert B.hcr_restore_streamed(*args, staging, staging.numel(), 1, ws, 64,
                                  check=False) == B.HCR_ERR_WORKSPACE
    assert B.hcr_restore_streamed(*args, staging, staging.numel(), 0, ws, ws.numel(),
                                  check=False) == B.HCR_ERR_INVALID_ARG
    torch.cuda.synchronize()
    from workloads import generate as G
    assert bool((case.k_cache.view(torch.int16) == G.SENTINEL_BITS).all())


def test_streamed_full_size_13b(cuda_device):
    """Llama2-13B shape, 16384 tokens, shuffled blocks: the single-CTA tiles
    (chosen for d_model > 4096) through the streamed pipeline at full size."""
    w = C.get("llama2-13b")
    ref = Hn.run(Hn.make_case(w, cuda_device, gen_device=cuda_device))
    assert ref.status == 0
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer,
                        gen_device=cuda_device)
    assert _streamed(case, 4, 3) == 0
    assert case.restorer.check()[0] == 0
    _same(case, ref)

"""Guard regions around every output buffer (GPU).

Each output is a view into a larger sentinel-filled allocation: the bytes
before and after the view must survive every call unchanged.  This covers
what a memory sanitizer would for the library's own writes: the workspace,
the K/V row store, the codec's codes, scales and decoded output, the chunk
store of the save side, and the staging ring of the streamed restores.
"""
import pytest
import torch

from tests import harness as Hn
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

W = Workload("guard", ModelShape("gd", 4, 512, 4, 4, 128), (1, 200, 0, 77, 300, 13),
             (0, 5, 9, 1000, 31, 2), block_order="shuffled", spare_blocks=3)
PAD = 4096          # guard bytes on each side (a multiple of 256 keeps the view aligned)
BYTE = 0xA5


class Guarded:
    """A byte buffer of `nbytes` with PAD guard bytes on both sides."""

    def __init__(self, nbytes, device, pinned=False):
        self.n = nbytes
        t = torch.full((nbytes + 2 * PAD,), BYTE, dtype=torch.uint8)
        self.raw = t.pin_memory() if pinned else t.to(device)

    def view(self, dtype=torch.uint8, shape=None):
        v = self.raw[PAD:PAD + self.n].view(dtype)
        return v if shape is None else v.view(shape)

    def intact(self):
        torch.cuda.synchronize()
        head, tail = self.raw[:PAD], self.raw[PAD + self.n:]
        return bool((head == BYTE).all()) and bool((tail == BYTE).all())


def _layout(case):
    from kv_cache_restoration_gb300 import binding as B
    lay = case.layout
    return B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0)


def test_restore_workspace_guard(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    L, T, _ = case.hidden.shape
    need = B.hcr_workspace_bytes(case.restorer.handle, T, L)
    ws = Guarded(need, cuda_device)
    B.hcr_restore(case.restorer.handle, case.hidden, 0, L, int(case.start.numel()), T, case.cu,
                  case.start, case.table, case.layout.max_blocks, case.k_cache, case.v_cache,
                  _layout(case), ws.view(), need, torch.cuda.current_stream())
    assert ws.intact()
    Hn.compare(case)


@pytest.mark.parametrize("pinned", [False, True], ids=["device", "host"])
def test_kv_store_guard(cuda_device, pinned):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.run(Hn.make_case(W, cuda_device))
    L, T, _ = case.hidden.shape
    row = W.shape.n_kv_heads * W.shape.head_dim
    kv = Guarded(L * 2 * T * row * 2, cuda_device, pinned)
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, 1) + 256, dtype=torch.uint8,
                     device=cuda_device)
    B.hcr_save_kv(case.restorer.handle, kv.view(torch.int16), 0, L, int(case.start.numel()), T,
                  case.cu, case.start, case.table, case.layout.max_blocks, case.k_cache,
                  case.v_cache, _layout(case), ws, ws.numel(), torch.cuda.current_stream())
    assert kv.intact()


@pytest.mark.parametrize("pinned", [False, True], ids=["device", "host"])
def test_codec_guards(cuda_device, pinned):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    L, T, d = case.hidden.shape
    params = B.codec_params()
    codes = Guarded(L * T * d, cuda_device, pinned)
    scales = Guarded(L * T * 4, cuda_device, pinned)
    out = Guarded(L * T * d * 2, cuda_device)
    n_req = int(case.start.numel())
    stream = torch.cuda.current_stream()
    B.hcr_encode_hidden(case.restorer.handle, params, case.hidden, 0, L, n_req, T, case.cu,
                        codes.view(torch.int8), scales.view(torch.float32), stream)
    assert codes.intact() and scales.intact()
    B.hcr_decode_hidden(case.restorer.handle, params, codes.view(torch.int8),
                        scales.view(torch.float32), 0, L, n_req, T, case.cu,
                        out.view(torch.bfloat16), stream)
    assert out.intact()


def test_chunk_store_guard(cuda_device):
    from dataclasses import replace

    from kv_cache_restoration_gb300 import binding as B
    from workloads import generate as G
    case = Hn.make_case(W, cuda_device)
    L, T, d = case.hidden.shape
    clay = G.request_layout(replace(W, block_size=64))
    store = Guarded(clay.num_blocks * W.shape.n_layers * 64 * d * 2, cuda_device)
    B.hcr_save_hidden(case.restorer.handle, case.hidden, 0, L, int(case.start.numel()), T,
                      case.cu, case.start, torch.as_tensor(clay.block_table, device=cuda_device),
                      int(clay.block_table.shape[1]), 64, store.view(torch.int16),
                      clay.num_blocks, torch.cuda.current_stream())
    assert store.intact()


def test_staging_guards_of_the_streamed_restores(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    L, T, d = case.hidden.shape
    lay = case.layout
    n_req = int(case.start.numel())
    ws = torch.empty(B.hcr_workspace_bytes(case.restorer.handle, T, 2) + 256, dtype=torch.uint8,
                     device=cuda_device)
    stream = torch.cuda.current_stream()
    # plain hidden states, 2-layer groups, 2 slots
    host = case.hidden.cpu().pin_memory()
    staging = Guarded(2 * 2 * T * d * 2, cuda_device)
    B.hcr_restore_streamed(case.restorer.handle, host, 0, L, n_req, T, case.cu, case.start,
                           case.table, lay.max_blocks, case.k_cache, case.v_cache, _layout(case),
                           staging.view(), staging.n, 2, ws, ws.numel(), stream)
    assert staging.intact()
    Hn.compare(case)
    # encoded form
    params = B.codec_params()
    codes = torch.empty((L, T, d), dtype=torch.int8, device=cuda_device)
    scales = torch.zeros((L, T), dtype=torch.float32, device=cuda_device)
    B.hcr_encode_hidden(case.restorer.handle, params, case.hidden, 0, L, n_req, T, case.cu,
                        codes, scales, stream)
    nbytes = B.encoded_staging_bytes(T, d, 2, 2)
    staging2 = Guarded(nbytes, cuda_device)
    B.hcr_restore_streamed_encoded(case.restorer.handle, params, codes.cpu().pin_memory(),
                                   scales.cpu().pin_memory(), 0, L, n_req, T, case.cu, case.start,
                                   case.table, lay.max_blocks, case.k_cache, case.v_cache,
                                   _layout(case), staging2.view(), nbytes, 2, ws, ws.numel(),
                                   stream)
    assert staging2.intact()
    assert case.restorer.check()[0] == 0

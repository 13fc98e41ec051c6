"""hcr_save_hidden (the save side: layer inputs into fixed-size chunks laid out
token-before-layer) against the oracle, bit for bit, on the GPU."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from oracle import save as S
from tests import harness as Hn
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu


def _store(n_chunks, L, Ct, d, device, pinned=False):
    t = torch.full((n_chunks, L, Ct, d), G.SENTINEL_BITS, dtype=torch.int16)
    t = t.pin_memory() if pinned else t.to(device)
    return t.view(torch.bfloat16)


def _save(case, chunk_tokens, store, table, n_chunks, hidden=None, cu=None, start=None,
          layer_begin=None, layer_end=None, check=True):
    from kv_cache_restoration_gb300 import binding as B
    hidden = case.hidden if hidden is None else hidden
    cu = case.cu if cu is None else cu
    start = case.start if start is None else start
    lb = case.layer_begin if layer_begin is None else layer_begin
    le = case.layer_end if layer_end is None else layer_end
    st = B.hcr_save_hidden(case.restorer.handle, hidden, lb, le, int(start.numel()),
                           int(hidden.shape[1]), cu, start, table, int(table.shape[1]),
                           chunk_tokens, store, n_chunks, torch.cuda.current_stream(),
                           check=check)
    torch.cuda.synchronize()
    return st


def _expect(case, chunk_tokens, table_np, n_chunks):
    s = case.w.shape
    lay = case.layout
    hid = [Hn.widen(case.hidden[i], s.dtype) for i in range(case.layer_end - case.layer_begin)]
    return S.save_chunks(hid, case.layer_begin, s.n_layers, lay.cu_seqlens, lay.start_pos,
                         table_np, chunk_tokens, n_chunks)


def _chunk_table(w, chunk_tokens):
    lay = G.request_layout(replace(w, block_size=chunk_tokens))
    return lay.block_table, lay.num_blocks


def _assert_store_equals(store, want, dtype):
    bits = Hn.bits_of(store)
    unwritten = np.isnan(want)
    assert np.all(bits[unwritten] == G.SENTINEL_BITS), "unwritten chunk slots changed"
    assert np.array_equal(Hn.widen(store, dtype)[~unwritten], want[~unwritten])


W = Workload("save", ModelShape("sv", 3, 256, 2, 2, 64), (1, 200, 0, 77, 300),
             (0, 5, 9, 1000, 31), block_order="shuffled", spare_blocks=3)


@pytest.mark.parametrize("chunk_tokens", [64, 16, 1])
@pytest.mark.parametrize("pinned", [False, True], ids=["device-store", "host-store"])
def test_save_matches_oracle(cuda_device, chunk_tokens, pinned):
    case = Hn.make_case(W, cuda_device)
    table_np, n = _chunk_table(W, chunk_tokens)
    table = torch.as_tensor(table_np, device=cuda_device)
    store = _store(n, 3, chunk_tokens, 256, cuda_device, pinned)
    assert _save(case, chunk_tokens, store, table, n) == 0
    assert case.restorer.check()[0] == 0
    _assert_store_equals(store, _expect(case, chunk_tokens, table_np, n), "bf16")


def test_save_layer_subrange(cuda_device):
    case = Hn.make_case(W, cuda_device, 1, 3)
    table_np, n = _chunk_table(W, 64)
    store = _store(n, 3, 64, 256, cuda_device)
    assert _save(case, 64, store, torch.as_tensor(table_np, device=cuda_device), n) == 0
    want = _expect(case, 64, table_np, n)
    assert np.isnan(want[:, 0]).all()
    _assert_store_equals(store, want, "bf16")


def test_decode_steps_fill_chunks_like_one_save(cuda_device):
    """Generation saves one token per request per step (every layer's input of
    that token); after N steps the chunks equal one save of all N tokens."""
    n_req, steps = 4, 70
    w = Workload("dec", ModelShape("dec", 2, 256, 2, 2, 64), (steps,) * n_req, (0, 5, 63, 200))
    case = Hn.make_case(w, cuda_device)
    table_np, n = _chunk_table(w, 64)
    table = torch.as_tensor(table_np, device=cuda_device)
    once = _store(n, 2, 64, 256, cuda_device)
    assert _save(case, 64, once, table, n) == 0
    stepwise = _store(n, 2, 64, 256, cuda_device)
    hid = case.hidden.view(2, n_req, steps, 256)
    one = torch.arange(n_req + 1, dtype=torch.int32, device=cuda_device)
    for s in range(steps):
        step_h = hid[:, :, s].contiguous()
        assert _save(case, 64, stepwise, table, n, hidden=step_h, cu=one,
                     start=case.start + s) == 0
    assert torch.equal(once.view(torch.int16), stepwise.view(torch.int16))


def test_bad_chunk_id_is_skipped_and_flagged(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(W, cuda_device)
    table_np, n = _chunk_table(W, 64)
    bad = table_np.copy()
    bad[4, 1] = n + 5                      # request 4: positions 64..127 (tokens 311..374)
    store = _store(n, 3, 64, 256, cuda_device)
    assert _save(case, 64, store, torch.as_tensor(bad, device=cuda_device), n) == 0
    st, flags = case.restorer.check()
    assert st == B.HCR_ERR_DEVICE_BOUNDS and flags & B.HCR_DEVERR_BLOCK_ID
    want = _expect(case, 64, table_np, n)
    want[table_np[4, 1]] = np.nan          # that chunk must stay untouched
    _assert_store_equals(store, want, "bf16")


def test_save_then_restore_round_trip(cuda_device):
    """Restoring from hidden states gathered out of the chunk store gives the
    same caches as restoring from the originals."""
    ref = Hn.run(Hn.make_case(W, cuda_device))
    table_np, n = _chunk_table(W, 64)
    store = _store(n, 3, 64, 256, cuda_device)
    assert _save(ref, 64, store, torch.as_tensor(table_np, device=cuda_device), n) == 0
    pl = S.chunk_placement(ref.layout.cu_seqlens, ref.layout.start_pos, table_np, 64, n)
    cid = torch.as_tensor(pl.chunk, device=cuda_device)
    off = torch.as_tensor(pl.offset, device=cuda_device)
    gathered = torch.stack([store[cid, l, off] for l in range(3)])
    case = Hn.make_case(W, cuda_device, params=ref.params, restorer=ref.restorer)
    case.hidden = gathered.contiguous()
    Hn.run(case)
    assert torch.equal(case.k_cache.view(torch.int16), ref.k_cache.view(torch.int16))
    assert torch.equal(case.v_cache.view(torch.int16), ref.v_cache.view(torch.int16))

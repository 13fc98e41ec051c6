"""Concurrent use of one handle (GPU): restores of different request batches
on different streams, each with its own workspace, issued from different host
threads at once, give bit for bit the caches of the same restores run one
after the other.  The streamed restore (whose copy stream and events belong
to the handle) is covered the same way."""
import threading

import torch
import pytest

from tests import harness as Hn
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

SHAPE = ModelShape("cc", 4, 512, 4, 4, 128)
WA = Workload("cc-a", SHAPE, (1, 200, 0, 77, 300), (0, 5, 9, 1000, 31), block_order="shuffled",
              spare_blocks=3)
# batch B stays inside the handle's RoPE table, which batch A sizes (1077 positions)
WB = Workload("cc-b", SHAPE, (513, 64, 129), (7, 0, 500), block_order="shuffled", seed=5)


def _same(a, b):
    for c in ("k_cache", "v_cache"):
        assert torch.equal(getattr(a, c).view(torch.int16), getattr(b, c).view(torch.int16)), c


def _run_threads(fns):
    errors = []

    def wrap(fn):
        try:
            fn()
        except Exception as e:   # re-raised in the main thread
            errors.append(e)
    ts = [threading.Thread(target=wrap, args=(f,)) for f in fns]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errors:
        raise errors[0]


def test_concurrent_restores_on_two_streams(cuda_device):
    ref_a = Hn.run(Hn.make_case(WA, cuda_device))
    r = ref_a.restorer
    ref_b = Hn.run(Hn.make_case(WB, cuda_device, params=ref_a.params, restorer=r))
    assert ref_a.status == 0 and ref_b.status == 0
    for _ in range(3):
        a = Hn.make_case(WA, cuda_device, params=ref_a.params, restorer=r)
        b = Hn.make_case(WB, cuda_device, params=ref_a.params, restorer=r)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        ws1 = torch.empty_like(r.workspace(WA.n_tokens, 4, cuda_device))
        ws2 = torch.empty(r.workspace(WB.n_tokens, 4, cuda_device).numel() + 4096,
                          dtype=torch.uint8, device=cuda_device)
        torch.cuda.synchronize()

        def go(case, stream, ws):
            def f():
                lay = case.layout
                case.restorer.restore(case.hidden, 0, 4, case.cu, case.start, case.table,
                                      case.k_cache, case.v_cache, lay.num_blocks, lay.block_size,
                                      stream=stream, workspace=ws)
            return f
        _run_threads([go(a, s1, ws1), go(b, s2, ws2)])
        torch.cuda.synchronize()
        assert r.check()[0] == 0
        _same(a, ref_a)
        _same(b, ref_b)


def test_concurrent_streamed_restores_share_the_handle(cuda_device):
    ref_a = Hn.run(Hn.make_case(WA, cuda_device))
    r = ref_a.restorer
    ref_b = Hn.run(Hn.make_case(WB, cuda_device, params=ref_a.params, restorer=r))
    # separate Restorer-style staging per thread: call the binding directly
    from kv_cache_restoration_gb300 import binding as B
    a = Hn.make_case(WA, cuda_device, params=ref_a.params, restorer=r)
    b = Hn.make_case(WB, cuda_device, params=ref_a.params, restorer=r)

    def go(case, stream):
        def f():
            lay = case.layout
            T, d = case.w.n_tokens, SHAPE.d_model
            host = case.hidden.cpu().pin_memory()
            staging = torch.empty(2 * 2 * T * d * 2, dtype=torch.uint8, device=cuda_device)
            ws = torch.empty(B.hcr_workspace_bytes(r.handle, T, 2) + 256, dtype=torch.uint8,
                             device=cuda_device)
            B.hcr_restore_streamed(r.handle, host, 0, 4, int(case.start.numel()), T, case.cu,
                                   case.start, case.table, lay.max_blocks, case.k_cache,
                                   case.v_cache,
                                   B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0),
                                   staging, staging.numel(), 2, ws, ws.numel(), stream)
            torch.cuda.synchronize()
        return f
    _run_threads([go(a, torch.cuda.Stream()), go(b, torch.cuda.Stream())])
    assert r.check()[0] == 0
    _same(a, ref_a)
    _same(b, ref_b)

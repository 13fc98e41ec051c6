"""hcr_restore_no_alloc: the restore entry point for callers that cannot
allocate device memory (an engine whose HBM is all handed to its KV pool, or
one that must not let cudaMalloc/cudaFree synchronise the device under
running decode work).  It takes its scratch from a fixed array built into
the library instead of a caller workspace.

Checked through the C ABI on two calls in a row of different shapes (the
second call reuses the array the first one left behind): the caches must be
bit-identical to hcr_restore's on the same inputs (the same kernels run; only
the scratch address differs), and within the parity tolerance of the oracle.
This file is collected last so a stop-at-first-failure run has already run
every other test.
"""
import pytest
import torch

from tests import harness as Hn
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu


def _no_alloc(case):
    from kv_cache_restoration_gb300 import binding as B
    lay = case.layout
    layout = B.hcr_cache_layout(lay.num_blocks, lay.block_size, 0)
    return B.hcr_restore_no_alloc(case.restorer.handle, case.hidden, case.layer_begin,
                                  case.layer_end, int(case.start.numel()), case.w.n_tokens,
                                  case.cu, case.start, case.table, lay.max_blocks, case.k_cache,
                                  case.v_cache, layout, torch.cuda.current_stream(),
                                  check=False)


def _assert_same_restore(got: torch.Tensor, ref: torch.Tensor):
    gb, rb = got.view(torch.int16), ref.view(torch.int16)
    diff = int((gb != rb).sum())
    assert diff == 0, f"{diff} cache elements differ from hcr_restore's"


WORKLOADS = [
    Workload("na-ragged", ModelShape("na1", 3, 512, 4, 4, 128), (1, 200, 0, 77, 300),
             (0, 5, 9, 1000, 31), block_order="shuffled", spare_blocks=3),
    C.get("tiny"),
]


def test_no_alloc_matches_restore_on_two_calls_in_a_row(cuda_device):
    for w in WORKLOADS:
        ref = Hn.run(Hn.make_case(w, cuda_device))          # hcr_restore, caller workspace
        assert ref.status == 0
        case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer)
        assert _no_alloc(case) == 0
        st, flags = case.restorer.check()
        assert st == 0, flags
        _assert_same_restore(case.k_cache, ref.k_cache)
        _assert_same_restore(case.v_cache, ref.v_cache)
        Hn.compare(case)          # every element against the oracle, every slot


def test_no_alloc_rejects_restores_beyond_its_scratch(cuda_device):
    from kv_cache_restoration_gb300 import binding as B
    case = Hn.make_case(C.get("tiny"), cuda_device)
    too_many = B.HCR_NO_ALLOC_SCRATCH_BYTES // 8          # needs > 16 B of scratch per token
    need = B.hcr_workspace_bytes(case.restorer.handle, too_many, 2)
    assert need > B.HCR_NO_ALLOC_SCRATCH_BYTES
    lay = case.layout
    st = B.hcr_restore_no_alloc(case.restorer.handle, case.hidden, 0, 2, 1, too_many, case.cu,
                                case.start, case.table, lay.max_blocks, case.k_cache,
                                case.v_cache, B.hcr_cache_layout(lay.num_blocks, 16, 0),
                                check=False)
    assert st == B.HCR_ERR_WORKSPACE
    assert "scratch" in B.hcr_last_error()
    torch.cuda.synchronize()
    assert bool((case.k_cache.view(torch.int16) == G.SENTINEL_BITS).all())

"""Failure detection on the GPU without faulting it: a pipeline wait that can
never complete gives up after its time limit, the kernel reports
HCR_ERR_TIMEOUT through the device error word, and the CUDA context stays
usable for the next restore."""
import time

import pytest

from tests import harness as Hn
from workloads import configs as C
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu


# the weight-row tiles need 128-wide heads: 1-layer cases with two of them,
# one with a single-MMA chunk (129 tokens) and one with a two-MMA chunk (300)
HEAD128 = {"weight-rows": Workload("stall128", ModelShape("s128", 1, 256, 2, 2, 128), (129,),
                                   (2,)),
           "weight-rows-2mma": Workload("stall128x2", ModelShape("s128", 1, 256, 2, 2, 128),
                                        (300,), (2,))}


@pytest.mark.parametrize("name", ["single", "pair", "weight-rows", "weight-rows-2mma"])
def test_stalled_pipeline_times_out_and_context_survives(cuda_device, name):
    from kv_cache_restoration_gb300 import binding as B
    variant = {"single": 1, "pair": 2}.get(name, 3)
    w = HEAD128[name] if variant == 3 else C.get("tiny")
    case = Hn.make_case(w, cuda_device)
    assert B.hcr_debug_set_variant(case.restorer.handle, variant) == B.HCR_OK
    assert B.hcr_debug_set_stall(case.restorer.handle, True) == B.HCR_OK
    t0 = time.monotonic()
    Hn.run(case)
    elapsed = time.monotonic() - t0
    assert case.status == B.HCR_ERR_TIMEOUT
    assert case.flags & B.HCR_DEVERR_TIMEOUT
    assert 1.5 < elapsed < 60.0
    # the record names the first wait that gave up: the MMA's wait for the
    # stage whose load was withheld (k-block 0), or the epilogue's wait for
    # that tile's accumulator (accumulator 0), on one of the 4 tiles
    st, rec = B.hcr_debug_timeout_record(case.restorer.handle)
    assert st == B.HCR_OK
    assert rec[0] in (4, 7) and rec[3] < 4 and rec[4] == 0, rec
    assert B.hcr_debug_timeout_record(case.restorer.handle)[1][0] == 0   # cleared
    assert B.hcr_debug_set_stall(case.restorer.handle, False) == B.HCR_OK
    again = Hn.run(Hn.make_case(w, cuda_device, params=case.params, restorer=case.restorer))
    assert again.status == 0
    Hn.compare(again)

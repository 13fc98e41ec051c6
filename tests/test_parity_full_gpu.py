"""The restore at the workloads' full sizes (GPU), in the launch configuration
bench.py times: every row of one layer against the oracle, a seeded sample
of rows (plus each request's first and last) in every layer, and the
bit-exact sentinel check on every slot of every layer."""
import numpy as np
import pytest
import torch

from tests import harness as Hn
from workloads import configs as C

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["llama2-7b", "llama2-13b", "opt-30b"])
def test_full_size(cuda_device, name):
    w = C.get(name)
    L = w.shape.n_layers
    case = Hn.make_case(w, cuda_device, gen_device=cuda_device)
    lay = case.layout
    # the two stages exactly as bench.py launches them
    for stage in ("prepare", "project"):
        case.restorer.restore(case.hidden, 0, L, case.cu, case.start, case.table, case.k_cache,
                              case.v_cache, lay.num_blocks, lay.block_size, stage=stage)
    case.status, case.flags = case.restorer.check()
    assert case.status == 0, (case.status, case.flags)
    Hn.compare(case, layers=[L - 1], check_sentinel=False)              # every row
    Hn.compare(case, rows=Hn.sample_rows(w, 1 / 64), check_sentinel=True)  # every layer


@pytest.mark.parametrize("name", ["llama2-7b-T300", "llama2-13b-T300", "opt-30b-T300",
                                  "llama2-7b-T794"])
def test_full_size_short_restores(cuda_device, name):
    """The short restores the bench times beside the headline, at full model
    size and in its launch configuration: 300 tokens run on the weight-row
    tiles (the automatic choice for 257..320 tokens), 794 on token-row tiles.
    Every row of every layer is checked (the oracle is cheap at 300-800 rows),
    plus the sentinel check on every slot."""
    from kv_cache_restoration_gb300 import binding as B
    w = C.get(name)
    L = w.shape.n_layers
    case = Hn.make_case(w, cuda_device, gen_device=cuda_device)
    want = 3 if w.n_tokens == 300 else None
    if want is not None:
        assert B.hcr_project_variant(case.restorer.handle, w.n_tokens, L) == want
    lay = case.layout
    for stage in ("prepare", "project"):
        case.restorer.restore(case.hidden, 0, L, case.cu, case.start, case.table, case.k_cache,
                              case.v_cache, lay.num_blocks, lay.block_size, stage=stage)
    case.status, case.flags = case.restorer.check()
    assert case.status == 0, (case.status, case.flags)
    Hn.compare(case, check_sentinel=True)


def test_ragged_batch_in_layer_windows(cuda_device):
    """64 requests, ~648K tokens, ragged lengths and starts, permuted block
    table.  Hidden states plus caches for all 32 layers exceed HBM, so the
    restore runs in four windows of 8 layers through layer_begin/layer_end;
    every window is checked before its buffers are reused."""
    w = C.get("ragged-7b")
    s = w.shape
    first = Hn.make_case(w, cuda_device, 0, 8, gen_device=cuda_device)
    params, restorer = first.params, first.restorer
    rows = Hn.sample_rows(w, 1 / 1024)
    del first
    for lb in range(0, s.n_layers, 8):
        torch.cuda.empty_cache()
        case = Hn.run(Hn.make_case(w, cuda_device, lb, lb + 8, params=params, restorer=restorer,
                                   gen_device=cuda_device))
        assert case.status == 0, (case.status, case.flags)
        Hn.compare(case, rows=rows, check_sentinel=True)
        del case


@pytest.mark.parametrize("name,variant", [("llama2-13b-T1024", 2), ("llama2-13b-T2048", 1),
                                          ("opt-30b-T512", 2), ("opt-30b-T384", 1)])
def test_full_width_mid_restores(cuda_device, name, variant):
    """Mid-size restores of the wider models at full size, in the variant the
    automatic choice takes for them (CTA pairs for calls of at most 6.5 TFLOP
    without a half tail tile, single CTAs otherwise; the norm statistics fused
    into the projection where it has at most 8 m-tiles per layer): every row
    of the last layer, a seeded row sample of every layer, the sentinel check
    on every slot."""
    from kv_cache_restoration_gb300 import binding as B
    w = C.get(name)
    L = w.shape.n_layers
    case = Hn.make_case(w, cuda_device, gen_device=cuda_device)
    assert B.hcr_project_variant(case.restorer.handle, w.n_tokens, L) == variant
    lay = case.layout
    for stage in ("prepare", "project"):
        case.restorer.restore(case.hidden, 0, L, case.cu, case.start, case.table, case.k_cache,
                              case.v_cache, lay.num_blocks, lay.block_size, stage=stage)
    case.status, case.flags = case.restorer.check()
    assert case.status == 0, (case.status, case.flags)
    Hn.compare(case, layers=[L - 1], check_sentinel=False)
    Hn.compare(case, rows=Hn.sample_rows(w, 1 / 32), check_sentinel=True)

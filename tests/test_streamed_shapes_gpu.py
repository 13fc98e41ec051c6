"""The streamed entry points on other model shapes (GPU): fp16 with LayerNorm,
K/V bias and no RoPE (the OPT family), grouped-query heads, 64- and 256-wide
heads.  From plain host hidden states, from the saved chunk store and as a
layer split with saved K/V, each gives bit for bit the caches hcr_restore
gives from the same hidden states in HBM, which the oracle checks."""
import pytest

from tests import harness as Hn
from tests.test_split_gpu import _saved_kv_host, _split_restore
from tests.test_streamed_chunks_gpu import _restore_chunks, _save_to_host, _source
from tests.test_streamed_gpu import _same, _streamed
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

LENS, STARTS = (1, 150, 0, 77, 200), (0, 5, 9, 400, 31)
SHAPES = [
    ModelShape("opt", 4, 384, 6, 6, 64, norm="ln", rope=False, dtype="fp16", kv_bias=True),
    ModelShape("gqa", 4, 512, 8, 2, 128),
    ModelShape("dh64", 4, 256, 4, 4, 64, rope_theta=5e5),
    ModelShape("dh256", 4, 512, 2, 2, 256),
]


def _workload(s):
    return Workload(f"st-{s.name}", s, LENS, STARTS, block_order="shuffled", spare_blocks=2)


def _reference(w, device):
    ref = Hn.run(Hn.make_case(w, device))
    assert ref.status == 0
    Hn.compare(ref)
    return ref


@pytest.mark.parametrize("s", SHAPES, ids=[s.name for s in SHAPES])
def test_streamed_from_host_hidden_states(cuda_device, s):
    w = _workload(s)
    ref = _reference(w, cuda_device)
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer)
    assert _streamed(case, 2, 2) == 0
    assert case.restorer.check()[0] == 0
    _same(case, ref)


@pytest.mark.parametrize("s", SHAPES, ids=[s.name for s in SHAPES])
def test_streamed_from_the_chunk_store(cuda_device, s):
    w = _workload(s)
    ref = _reference(w, cuda_device)
    store, table_np, n = _save_to_host(ref, 16)
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer)
    assert _restore_chunks(case, _source(store, 16, n, table_np, case.layout), 3, 2) == 0
    assert case.restorer.check()[0] == 0
    _same(case, ref)


@pytest.mark.parametrize("s", SHAPES, ids=[s.name for s in SHAPES])
def test_streamed_layer_split(cuda_device, s):
    w = _workload(s)
    ref = _reference(w, cuda_device)
    split = 2
    kv_host = _saved_kv_host(ref, split, s.n_layers)
    hidden_host = ref.hidden[:split].cpu().pin_memory()
    case = Hn.make_case(w, cuda_device, params=ref.params, restorer=ref.restorer)
    assert _split_restore(case, hidden_host, kv_host, split, 1, 2) == 0
    assert case.restorer.check()[0] == 0
    _same(case, ref)

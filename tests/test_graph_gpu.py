"""hcr_restore inside a CUDA graph, and a clean out-of-memory failure (GPU)."""
import pytest
import torch

from tests import harness as Hn
from workloads import configs as C
from workloads import generate as G
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

W = Workload("graph", ModelShape("gr", 3, 512, 4, 4, 128), (1, 200, 0, 77, 300),
             (0, 5, 9, 1000, 31), block_order="shuffled", spare_blocks=3)


def test_restore_captured_in_a_cuda_graph(cuda_device):
    """Capture one restore (both stages) and replay it on new hidden states
    copied into the captured buffers: each replay equals a direct restore."""
    ref = Hn.make_case(W, cuda_device)
    lay = ref.layout
    r = ref.restorer
    ws = r.workspace(W.n_tokens, 3, cuda_device)
    hidden = ref.hidden.clone()
    kc, vc = ref.k_cache.clone(), ref.v_cache.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):      # warm-up outside capture (loads modules, sets attributes)
        r.restore(hidden, 0, 3, ref.cu, ref.start, ref.table, kc, vc, lay.num_blocks,
                  lay.block_size, workspace=ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        r.restore(hidden, 0, 3, ref.cu, ref.start, ref.table, kc, vc, lay.num_blocks,
                  lay.block_size, workspace=ws, stream=torch.cuda.current_stream())
    for seed in (5, 6, 7):
        w = Workload(W.name, W.shape, W.seq_lens, W.start_pos, block_order="shuffled",
                     spare_blocks=3, seed=seed)
        fresh = G.device_inputs(w, cuda_device, params=ref.params)
        hidden.copy_(fresh.hidden)
        kc.fill_(0)
        vc.fill_(0)
        graph.replay()
        direct = Hn.make_case(W, cuda_device, params=ref.params, restorer=r)
        direct.hidden = fresh.hidden
        Hn.run(direct)
        torch.cuda.synchronize()
        written = direct.k_cache.view(torch.int16) != G.SENTINEL_BITS
        assert torch.equal(kc.view(torch.int16)[written], direct.k_cache.view(torch.int16)[written])
        assert torch.equal(vc.view(torch.int16)[written], direct.v_cache.view(torch.int16)[written])
    assert r.check()[0] == 0


def test_create_out_of_memory_fails_cleanly(cuda_device):
    """A model whose packed weights cannot fit is refused with HCR_ERR_OOM,
    nothing leaks, and the context keeps working."""
    from kv_cache_restoration_gb300 import binding as B, make_dims
    d = 16384
    g = torch.ones(d, dtype=torch.bfloat16, device=cuda_device)
    w = torch.zeros(128 * 128, d, dtype=torch.bfloat16, device=cuda_device)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    per_layer = 2 * d * d * 2                             # packed [W_k; W_v] of one layer, bytes
    L = int(free_before // per_layer) + 64                # layers beyond the free memory
    dims = make_dims(L, d, 128, 128, 128, max_position=16)
    st, h = B.hcr_create(dims, [g] * L, None, [w] * L, [w] * L, check=False)
    if h is not None:
        B.hcr_destroy(h)
    assert st == B.HCR_ERR_OOM and h is None, (st, B.hcr_last_error())
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free_before - (64 << 20)
    case = Hn.run(Hn.make_case(C.get("tiny"), cuda_device))
    assert case.status == 0
    Hn.compare(case)

"""The Restorer convenience methods over the C ABI (GPU): each gives what the
entry point it wraps gives."""
import pytest
import torch

from tests import harness as Hn
from workloads.configs import ModelShape, Workload

pytestmark = pytest.mark.gpu

W = Workload("rs", ModelShape("rs", 4, 512, 4, 4, 128), (1, 200, 0, 77, 300),
             (0, 5, 9, 1000, 31), block_order="shuffled", spare_blocks=3)


def test_restorer_methods(cuda_device):
    ref = Hn.run(Hn.make_case(W, cuda_device))
    r, lay = ref.restorer, ref.layout
    n_req = int(ref.start.numel())
    # streamed restore == restore
    case = Hn.make_case(W, cuda_device, params=ref.params, restorer=r)
    assert r.restore_streamed(ref.hidden.cpu().pin_memory(), 0, 4, ref.cu, ref.start, ref.table,
                              case.k_cache, case.v_cache, lay.num_blocks, lay.block_size,
                              layers_per_chunk=2, slots=2) == 0
    torch.cuda.synchronize()
    assert torch.equal(case.k_cache.view(torch.int16), ref.k_cache.view(torch.int16))
    # K/V rows out and back
    kv = torch.empty((4, 2, W.n_tokens, 512), dtype=torch.bfloat16, device=cuda_device)
    r.save_kv(kv, 0, 4, ref.cu, ref.start, ref.table, ref.k_cache, ref.v_cache, lay.num_blocks,
              lay.block_size)
    fresh = Hn.make_case(W, cuda_device, params=ref.params, restorer=r)
    r.load_kv(kv, 0, 4, ref.cu, ref.start, ref.table, fresh.k_cache, fresh.v_cache,
              lay.num_blocks, lay.block_size)
    torch.cuda.synchronize()
    assert torch.equal(fresh.v_cache.view(torch.int16), ref.v_cache.view(torch.int16))
    # codec round trip: decode(encode(h)) stays within half a bin (layers 0, 1
    # use bin 0.5, layer 2 bin 1, layer 3 bin 1.5 of 4 layers) plus the final
    # rounding to bf16 (half an ulp of values below 8: 0.016)
    codes, scales = r.encode(ref.hidden, 0, 4, ref.cu, n_req)
    dec = r.decode(codes, scales, 0, 4, ref.cu, n_req)
    torch.cuda.synchronize()
    err = (dec.float() - ref.hidden.float()).abs().amax(dim=(1, 2))
    bound = torch.tensor([0.25, 0.25, 0.5, 0.75], device=cuda_device) + 0.016
    assert (err <= bound).all(), err
    # split planning
    costs, split = r.plan_split(256, layers_per_chunk=2, reps=2)
    assert costs.restore_s > 0 and split.hidden_layers + split.kv_layers == 4
    assert r.check()[0] == 0

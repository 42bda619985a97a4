"""The allocation-free layer entry point (collected last on purpose).

bqe_moe_layer_forward_noalloc serves callers that cannot allocate device
memory where they run a layer (a plugin whose host framework owns all device
memory, a service that forbids allocation after start-up).  It must give the
same results as bqe_moe_layer_forward with a caller-allocated workspace, call
after call, although every call reuses one fixed array inside the library."""
import numpy as np
import pytest

import synth
from gpu_util import DeviceLayer, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.mark.parametrize("M", [1, 2])
def test_noalloc_matches_workspace_call(dev, M):
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    fm = [synth.TQ1, synth.Q2_0, synth.Q3_K, synth.MXFP4] * 6 + [synth.Q2_0]
    L = synth.small_layer(90 + M, fm, 1024, 768, 24, 3, M, bias_std=0.25)
    DL = DeviceLayer(L, dev)
    want, want_idx, want_w = DL.forward(L["x"])  # reference: caller-allocated workspace
    x = torch.from_numpy(np.ascontiguousarray(L["x"]).view(np.int16)).to(dev)
    for call in range(2):  # two calls in a row share the fixed array
        out = torch.full((M, 1024), float("nan"), device=dev)
        idx = torch.zeros(M, 3, dtype=torch.int32, device=dev)
        w = torch.zeros(M, 3, dtype=torch.float32, device=dev)
        status = torch.full((2,), -1, dtype=torch.int32, device=dev)
        A.bqe_moe_layer_forward_noalloc(DL.d, M, x, DL.wr, DL.bias, DL.pool.cstruct(), DL.table, None, out, 0,
                                        idx, w, status)
        torch.cuda.synchronize()
        assert status.cpu().tolist() == [0, 0], (call, status.cpu().tolist())
        assert np.array_equal(idx.cpu().numpy(), want_idx), call
        check_out(out.double().cpu().numpy(), want, what="no-alloc call %d" % call)


def test_noalloc_rejects_layers_beyond_its_array(dev):
    from bit_quantised_expert_gb300 import _abi as A
    d = A.desc(5120, 2304, 384, 6)
    assert A.bqe_workspace_bytes(d, 3) > 8 << 20
    with pytest.raises(A.BqeError) as e:
        A.bqe_moe_layer_forward_noalloc(d, 3, 1, 1, None, A.bqe_pool(1, 1, 1, 1, 1, 0), 1, None, 1, 0, None,
                                        None, None)
    assert e.value.status == A.BQE_ENOSPC

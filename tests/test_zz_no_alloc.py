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
    # every row count of the DeepSeek-V4.1-Flash layer fits; a wider layer at 8 rows does not
    assert A.bqe_workspace_bytes(A.desc(5120, 2304, 384, 6), 8) <= 8 << 20
    d = A.desc(7168, 2304, 384, 6)
    assert A.bqe_workspace_bytes(d, 8) > 8 << 20
    with pytest.raises(A.BqeError) as e:
        A.bqe_moe_layer_forward_noalloc(d, 8, 16, 16, None, A.bqe_pool(16, 1, 16, 16, 1, 0), 16, None, 16, 0, None,
                                        None, None)
    assert e.value.status == A.BQE_ENOSPC


def test_noalloc_timeout_then_recovery(dev):
    """A call whose work item never lands (the host tells the first CTA's
    producers to skip its copies, with a short wait limit) reports
    BQE_ETIMEOUT through status_out and through bqe_check_noalloc; the next
    clean call clears the array's state and matches the workspace call."""
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    M = 2
    fm = [synth.MXFP4] * 33
    L = synth.small_layer(13, fm, 2048, 1024, 32, 4, M)
    DL = DeviceLayer(L, dev)
    want, want_idx, _ = DL.forward(L["x"])
    x = torch.from_numpy(np.ascontiguousarray(L["x"]).view(np.int16)).to(dev)
    out = torch.zeros(M, 2048, device=dev)
    status = torch.full((2,), -1, dtype=torch.int32, device=dev)
    A.bqe_set_wait_limit_ns(20_000_000)  # 20 ms
    A.bqe_set_test_drop_item(0)
    try:
        A.bqe_moe_layer_forward_noalloc(DL.d, M, x, DL.wr, DL.bias, DL.pool.cstruct(), DL.table, None, out, 0,
                                        None, None, status)
        torch.cuda.synchronize()
    finally:
        A.bqe_set_test_drop_item(-1)
        A.bqe_set_wait_limit_ns(2_000_000_000)
    st = status.cpu().tolist()
    assert st[0] == A.BQE_ETIMEOUT and st[1] in (4, 5), st
    rc, det = A.bqe_check_noalloc()
    assert rc == A.BQE_ETIMEOUT and det in (4, 5), (A.status_name(rc), det)
    assert A.bqe_check_noalloc() == (A.BQE_OK, 0)  # read and cleared
    for call in range(2):
        out = torch.full((M, 2048), float("nan"), device=dev)
        idx = torch.zeros(M, 4, dtype=torch.int32, device=dev)
        status.fill_(-1)
        A.bqe_moe_layer_forward_noalloc(DL.d, M, x, DL.wr, DL.bias, DL.pool.cstruct(), DL.table, None, out, 0,
                                        idx, None, status)
        torch.cuda.synchronize()
        assert status.cpu().tolist() == [0, 0], (call, status.cpu().tolist())
        assert np.array_equal(idx.cpu().numpy(), want_idx)
        check_out(out.double().cpu().numpy(), want, what="no-alloc after timeout, call %d" % call)
    assert A.bqe_check_noalloc() == (A.BQE_OK, 0)

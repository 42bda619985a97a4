"""GPU parity of the decode path against the fp64 oracle, through the C ABI.

Bars: dequantised weights and top-k indices bit-exact (rows whose k-th and
(k+1)-th keys are within 1e-6 excepted); fp32 layer outputs within relative
L2 1e-4 and max-abs 1e-3 x max|reference|."""
import numpy as np
import pytest

import synth
from oracle import formats as F
from oracle import moe as O

from gpu_util import DeviceLayer, check_out, check_routing, oracle_layer_sampled, torch_dev

pytestmark = pytest.mark.gpu

ALL = [synth.TQ1, synth.Q2_0, synth.Q3_K, synth.MXFP4, synth.NVFP4]


@pytest.fixture(scope="module")
def dev():
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    d = torch_dev()
    torch.cuda.set_device(d)
    return d


# ------------------------------------------------------------------ dequant
@pytest.mark.parametrize("fmt", ALL)
@pytest.mark.parametrize("shape", [(512, 256), (2304, 5120)])
def test_dequant_bit_exact(dev, fmt, shape):
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    from bit_quantised_expert_gb300.pool import SlotPool
    H, I = shape
    rng = np.random.default_rng(100 + fmt)
    canon = synth.random_expert(rng, fmt, H, I)
    # exercise every code and extreme scales in the first blocks
    d = A.desc(H, I, 8, 2)
    pool = SlotPool(d, [fmt], dev)
    pool.upload(0, canon)
    p1, p3, p2 = F.split_expert(fmt, canon, H, I)
    base = pool.slot_ptr(0)
    for k, (p, rows, cols) in enumerate([(p1, I, H), (p3, I, H), (p2, H, I)]):
        out = torch.empty(rows * cols, dtype=torch.float32, device=dev)
        A.bqe_dequant(fmt, rows, cols, base + k * p1.size, out)
        got = out.cpu().numpy().reshape(rows, cols)
        want = F.dequant_matrix(fmt, p, rows, cols).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (fmt, k)


def test_dequant_special_values(dev):
    """Signed zeros, subnormal fp16 d, extreme UE8M0 exponents survive exactly."""
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    from bit_quantised_expert_gb300.pool import SlotPool
    H, I = 256, 256
    rng = np.random.default_rng(5)
    for fmt in ALL:
        canon = synth.random_expert(rng, fmt, H, I)
        bw, bb = F.BLOCK[fmt]
        blk = canon.reshape(-1, bb)
        if fmt == synth.MXFP4:
            blk[0, 16] = 0        # 2^-127 (subnormal in fp32)
            blk[1, 16] = 254      # 2^127
            blk[2, :16] = 0x88    # -0.0 codes
        elif fmt == synth.NVFP4:
            blk[0, 8] = 0x01      # smallest E4M3 subnormal, 2^-9
            blk[1, 8] = 0x7E      # largest E4M3, 448
            blk[2, 8] = 0xFE      # -448
            blk[3, :8] = 0x88     # -0.0 codes
            blk[4, 8] = 0x00      # scale +0
        else:
            dpos = {synth.Q2_0: 16, synth.TQ1: 52, synth.Q3_K: 108}[fmt]
            blk[0, dpos:dpos + 2] = (0x01, 0x00)   # smallest fp16 subnormal
            blk[1, dpos:dpos + 2] = (0x00, 0x00)   # d = +0: products keep their signs
            blk[2, dpos:dpos + 2] = (0x00, 0x80)   # d = -0
            blk[3, dpos:dpos + 2] = (0xff, 0x7b)   # largest finite fp16
        d = A.desc(H, I, 4, 1)
        pool = SlotPool(d, [fmt], dev)
        pool.upload(0, canon)
        out = torch.empty(I * H, dtype=torch.float32, device=dev)
        A.bqe_dequant(fmt, I, H, pool.slot_ptr(0), out)
        got = out.cpu().numpy()
        want = F.dequant_matrix(fmt, F.split_expert(fmt, canon, H, I)[0], I, H).astype(np.float32).reshape(-1)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), fmt


# ------------------------------------------------------------ small layers
@pytest.mark.parametrize("M", [1, 4])
def test_tiny_q2_0_layer(dev, M):
    """Tiny layer: hidden 512, inter 256, 16 routed + 1 shared, top-2, all Q2_0."""
    L = synth.tiny_layer(seed=0, m=M)
    DL = DeviceLayer(L, dev)
    out, idx, w = DL.forward(L["x"])
    ref = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 512, 256, 2, 16)
    check_routing(ref, idx, w)
    ref2 = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 512, 256, 2, 16, forced_idx=idx)
    assert np.allclose(w, ref2["w"], rtol=2e-6, atol=0)
    check_out(out, ref2["out"], what="tiny M=%d" % M)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 6, 8])
def test_mixed_small_layer(dev, M):
    """All four formats in one layer, selection bias N(0, 0.25), independent rows."""
    fm = [ALL[(3 * e + 1) % len(ALL)] for e in range(24)] + [synth.Q2_0]
    L = synth.small_layer(20 + M, fm, 1024, 768, 24, 3, M, bias_std=0.25)
    DL = DeviceLayer(L, dev)
    out, idx, w = DL.forward(L["x"])
    ref = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 1024, 768, 3, 24)
    check_routing(ref, idx, w)
    ref2 = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 1024, 768, 3, 24, forced_idx=idx)
    check_out(out, ref2["out"], what="mixed M=%d" % M)
    # the routing-only entry point selects the same experts with the same weights
    idx2, w2 = DL.route(L["x"])
    assert np.array_equal(idx, idx2) and np.allclose(w, w2, rtol=1e-6, atol=0)


@pytest.mark.parametrize("fmt", ALL)
def test_single_format_layer(dev, fmt):
    fm = [fmt] * 9
    L = synth.small_layer(40 + fmt, fm, 512, 512, 8, 2, 3, bias_std=0.0)
    # activations spanning many binades exercise the per-row f16 scaling
    L["x"][1] = synth.x_bf16(np.random.default_rng(3), 1, 512, std=1e-3)[0]
    L["x"][2] = synth.x_bf16(np.random.default_rng(4), 1, 512, std=20.0)[0]
    DL = DeviceLayer(L, dev)
    out, idx, w = DL.forward(L["x"], forced=np.array([[0, 1], [2, 3], [4, 5]], np.int32))
    ref2 = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 512, 512, 2, 8, forced_idx=idx)
    for m in range(3):  # rows differ by orders of magnitude: check each on its own scale
        check_out(out[m], ref2["out"][m], what="fmt %d row %d" % (fmt, m))


def test_bias_changes_selection_not_weights(dev):
    fm = [synth.Q2_0] * 17
    L = synth.small_layer(7, fm, 512, 256, 16, 2, 4, bias_std=0.0)
    DL = DeviceLayer(L, dev)
    _, idx0, w0 = DL.forward(L["x"], use_bias=False)
    # a large bias on the experts nobody chose moves the selection to them
    import torch
    b = np.zeros(16, np.float32)
    unchosen = sorted(set(range(16)) - set(idx0.reshape(-1).tolist()))[:2]
    b[unchosen] = 5.0
    DL.bias = torch.from_numpy(b).to(dev)
    out, idx1, w1 = DL.forward(L["x"])
    assert all(sorted(r.tolist()) == sorted(unchosen) for r in idx1)
    ref = O.moe_layer(L["x"], L["router"], b, L["experts"], L["fmts"], 512, 256, 2, 16)
    assert np.allclose(w1, ref["w"], rtol=2e-6)
    check_out(out, ref["out"], what="biased")


def test_scores_underflow_keep_weights_finite(dev):
    """Huge activations push every selected router logit below the fp32
    sigmoid's range; the mixing weights (ratios of scores) must still come out
    finite and equal to the fp64 statement."""
    fm = [synth.MXFP4] * 9
    L = synth.small_layer(44, fm, 512, 512, 8, 2, 3, bias_std=0.0)
    L["x"][2] = synth.x_bf16(np.random.default_rng(4), 1, 512, std=3e3)[0]
    DL = DeviceLayer(L, dev)
    forced = np.array([[7, 1], [1, 7], [0, 1]], np.int32)
    out, idx, w = DL.forward(L["x"], forced=forced)
    ref = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 512, 512, 2, 8, forced_idx=forced)
    assert np.isfinite(w).all() and np.isfinite(out).all()
    assert np.allclose(w, ref["w"], rtol=2e-6, atol=1e-30)
    for m in range(3):
        check_out(out[m], ref["out"][m], what="row %d" % m)


def test_forced_idx_with_repeats_and_accumulate(dev):
    import torch
    fm = [synth.MXFP4, synth.TQ1, synth.Q3_K, synth.Q2_0] * 4 + [synth.Q3_K]
    L = synth.small_layer(8, fm, 512, 256, 16, 3, 5, bias_std=0.0)
    DL = DeviceLayer(L, dev)
    forced = np.array([[0, 1, 2], [2, 2, 2], [15, 0, 7], [3, 3, 4], [9, 10, 11]], dtype=np.int32)
    prior = torch.randn(5, 512, device=dev)
    keep = prior.double().cpu().numpy()
    out, idx, w = DL.forward(L["x"], forced=forced, accumulate_into=prior)
    assert np.array_equal(idx, forced)
    ref = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 512, 256, 3, 16, forced_idx=forced)
    assert np.allclose(w, ref["w"], rtol=2e-6)
    # out = prior + layer, against the same sum in fp64 at the decode bar
    check_out(out, keep + ref["out"], what="accumulate")


@pytest.mark.parametrize("M", [1, 2, 6, 8])
def test_repeated_calls_consistent(dev, M):
    """Consecutive calls on one workspace (the call epoch and the arrival
    counters advance from call to call) choose the same experts with the
    same weights, and every call meets the decode bar against the oracle
    (the output rows are sums of fp32 atomic additions, whose order may
    differ from call to call)."""
    fm = [ALL[(3 * e + 2) % 4] for e in range(24)] + [synth.MXFP4]
    L = synth.small_layer(60 + M, fm, 1024, 768, 24, 3, M, bias_std=0.25)
    DL = DeviceLayer(L, dev)
    out, idx, w = DL.forward(L["x"])
    ref = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 1024, 768, 3, 24)
    check_routing(ref, idx, w)
    ref2 = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 1024, 768, 3, 24, forced_idx=idx)
    check_out(out, ref2["out"], what="M=%d" % M)
    for _ in range(5):
        out2, idx2, w2 = DL.forward(L["x"])
        assert np.array_equal(idx, idx2) and np.array_equal(w, w2)
        check_out(out2, ref2["out"], what="M=%d repeat" % M)
        assert np.allclose(out2, out, rtol=1e-5, atol=1e-5 * float(np.abs(out).max()))


def test_layer_stats(dev):
    """bqe_layer_stats reports the distinct experts the call streamed and
    their bytes, which the oracle's byte count states independently."""
    from bit_quantised_expert_gb300 import _abi as A
    fm = [ALL[e % len(ALL)] for e in range(24)] + [synth.Q2_0]
    L = synth.small_layer(71, fm, 1024, 768, 24, 3, 4, bias_std=0.25)
    DL = DeviceLayer(L, dev)
    _, idx, _ = DL.forward(L["x"])
    ws, _ = DL.workspace(4)
    st = A.bqe_layer_stats(DL.d, 4, ws)
    distinct = set(idx.reshape(-1).tolist())
    assert st["rows"] == 4 and st["experts_streamed"] == len(distinct) + 1
    assert st["expert_bytes"] == O.expert_bytes_streamed(idx, L["fmts"], 1024, 768, 24)
    assert st["router_bytes"] == 24 * 1024 * 4
    per = [0] * 6
    for e in distinct | {24}:
        per[int(L["fmts"][e])] += 1
    assert st["per_format"] == per
    # every row chose 3 distinct experts, and the shared expert serves all 4
    assert st["row_uses"] == 4 * 3 + 4


# ------------------------------------------------------- error reporting
def test_bad_slot_is_reported(dev):
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    L = synth.tiny_layer(seed=1, m=1)
    DL = DeviceLayer(L, dev)
    DL.table = torch.full((17,), 999, dtype=torch.int32, device=dev)  # no such slot
    ws, nb = DL.workspace(1)
    x = torch.from_numpy(L["x"].view(np.int16)).to(dev)
    out = torch.zeros(1, 512, device=dev)
    A.bqe_moe_layer_forward(DL.d, 1, x, DL.wr, None, DL.pool.cstruct(), DL.table, None, out, 0, None, None, ws, nb)
    rc, det = A.bqe_check(ws)
    assert rc == A.BQE_EDEVICE and det == 1
    A.bqe_workspace_init(ws, nb)
    DL.table = torch.arange(17, dtype=torch.int32, device=dev)
    o2, _, _ = DL.forward(L["x"])  # the context and the workspace are usable again
    assert np.isfinite(o2).all()


def test_pool_format_mask_selects_and_guards(dev):
    """bqe_pool_init records the slots' formats; a mask that leaves out a
    format in use is reported like an invalid slot (BQE_EDEVICE, slot-format
    detail), not computed with the wrong loops; mask 0 runs every format."""
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    L = synth.tiny_layer(seed=2, m=1)
    DL = DeviceLayer(L, dev)
    assert DL.pool.cstruct().fmt_mask == 1 << synth.Q2_0
    ref, _, _ = DL.forward(L["x"])
    ws, nb = DL.workspace(1)
    x = torch.from_numpy(L["x"].view(np.int16)).to(dev)
    for mask, ok in ((1 << synth.MXFP4, False), (0, True), ((1 << synth.Q2_0) | (1 << synth.TQ1), True)):
        p = A.bqe_pool.from_buffer_copy(DL.pool.cstruct())
        p.fmt_mask = mask
        A.bqe_workspace_init(ws, nb)
        out = torch.zeros(1, 512, device=dev)
        A.bqe_moe_layer_forward(DL.d, 1, x, DL.wr, DL.bias, p, DL.table, None, out, 0, None, None, ws, nb)
        rc, det = A.bqe_check(ws)
        if ok:
            assert rc == A.BQE_OK, (mask, A.status_name(rc), det)
            check_out(out.double().cpu().numpy(), ref, rel=1e-5, mabs=1e-5, what="mask %#x" % mask)
        else:
            assert rc == A.BQE_EDEVICE and det == 2, (mask, A.status_name(rc), det)
    A.bqe_workspace_init(ws, nb)


def test_host_argument_errors(dev):
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    L = synth.tiny_layer(seed=1, m=1)
    DL = DeviceLayer(L, dev)
    ws, nb = DL.workspace(1)
    x = torch.from_numpy(L["x"].view(np.int16)).to(dev)
    out = torch.zeros(1, 512, device=dev)
    for M in (0, 9):
        with pytest.raises(A.BqeError) as e:
            A.bqe_moe_layer_forward(DL.d, M, x, DL.wr, None, DL.pool.cstruct(), DL.table, None, out, 0, None, None,
                                    ws, nb)
        assert e.value.status == A.BQE_EINVAL
    with pytest.raises(A.BqeError) as e:
        A.bqe_moe_layer_forward(DL.d, 1, x, DL.wr, None, DL.pool.cstruct(), DL.table, None, out, 0, None, None,
                                ws, 64)
    assert e.value.status == A.BQE_ENOSPC


def test_wait_timeout_is_reported_and_recoverable(dev):
    """A work item that never lands (the host tells CTA 0's producers to skip
    its copies) makes the bounded waits run out: the call reports
    BQE_ETIMEOUT, and after re-initialising the workspace the next call is
    correct.  No GPU fault is involved."""
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    fm = [synth.MXFP4] * 33
    L = synth.small_layer(12, fm, 2048, 1024, 32, 4, 2)
    DL = DeviceLayer(L, dev)
    good, _, _ = DL.forward(L["x"])
    ws, nb = DL.workspace(2)
    x = torch.from_numpy(L["x"].view(np.int16)).to(dev)
    out = torch.zeros(2, 2048, device=dev)
    A.bqe_set_wait_limit_ns(20_000_000)  # 20 ms
    A.bqe_set_test_drop_item(0)
    try:
        A.bqe_moe_layer_forward(DL.d, 2, x, DL.wr, None, DL.pool.cstruct(), DL.table, None, out, 0, None, None,
                                ws, nb)
        rc, det = A.bqe_check(ws)
    finally:
        A.bqe_set_test_drop_item(-1)
        A.bqe_set_wait_limit_ns(2_000_000_000)
    assert rc == A.BQE_ETIMEOUT and det in (4, 5), (A.status_name(rc), det)
    A.bqe_workspace_init(ws, nb)
    again, _, _ = DL.forward(L["x"])
    check_out(again, good, what="after the timeout")

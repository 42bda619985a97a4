"""GPU parity at the full DeepSeek-V4.1-Flash layer sizes (hidden 5120,
inter 2304, 384 routed + 1 shared, top-6), in the launch configuration the
benchmark times: every output element of the decode layers against the fp64
oracle, and of the prefill layer on sampled tokens and 1024 columns."""
import numpy as np
import pytest

import synth
from oracle import moe as O

from gpu_util import check_out, check_routing, oracle_layer_sampled

pytestmark = pytest.mark.gpu

H, I, E, K = 5120, 2304, 384, 6


@pytest.fixture(scope="module")
def dev():
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _run_layer(W, dev, xi, M):
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    nb = A.bqe_workspace_bytes(W.d, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    A.bqe_workspace_init(ws, nb)
    out = torch.zeros(M, H, device=dev)
    idx = torch.zeros(M, K, dtype=torch.int32, device=dev)
    wts = torch.zeros(M, K, dtype=torch.float32, device=dev)
    x = W.xs[xi]
    A.bqe_moe_layer_forward(W.d, M, x, W.wr, W.bias, W.pool.cstruct(), W.table, None, out, 0, idx, wts, ws, nb)
    rc, det = A.bqe_check(ws)
    assert rc == A.BQE_OK, (A.status_name(rc), det)
    x_bits = x.cpu().numpy().view(np.uint16)
    return out.double().cpu().numpy(), idx.cpu().numpy(), wts.cpu().numpy(), x_bits


def _check_layer(W, dev, M, xi):
    out, idx, wts, x_bits = _run_layer(W, dev, xi, M)
    router = W.wr.cpu().numpy()
    bias = None if W.bias is None else W.bias.cpu().numpy()
    ref = O.route(O.bf16_bits_to_f64(x_bits), router, bias, K)
    assert check_routing(ref, idx, wts) > 0  # at least one row's selection is compared (not all near-ties)
    cols = None  # every column
    cache = {}

    def canon(e):
        if e not in cache:
            cache[e] = W.canon(e).cpu().numpy()
        return cache[e]
    oref, r2 = oracle_layer_sampled(W.fmts, canon, x_bits, router, bias, idx, H, I, E, K, cols)
    assert np.allclose(wts, r2["w"], rtol=2e-6, atol=0)
    return check_out(out, oref, what="full M=%d" % M)


@pytest.mark.parametrize("M", [1, 6, 8])
def test_fp4_layer(dev, M):
    from synth import workloads as WL
    W = WL.fp4_layer(dev, m=M, n_x=3)
    for xi in range(2 if M == 1 else 1):
        _check_layer(W, dev, M, xi)


@pytest.mark.parametrize("M", [1, 6])
def test_nvfp4_layer(dev, M):
    """The NVFP4 variant (blocks of 16 with E4M3 scales) at full size."""
    from synth import workloads as WL
    W = WL.fp4_layer(dev, seed=5, m=M, n_x=2, fmt=synth.NVFP4)
    _check_layer(W, dev, M, 0)


@pytest.mark.parametrize("M", [1, 6, 8])
def test_mixed_layer(dev, M):
    from synth import workloads as WL
    W = WL.mixed_layer(dev, m=M, n_x=2)
    _check_layer(W, dev, M, 0)


def test_step40_teacher_forced(dev):
    """40 chained layers over the 4288-slot pool (Zipf-forced routing): the
    whole step equals the layer-by-layer run bit for bit, each layer's input
    is the bf16 RMS-normalised residual, and sampled layers match the oracle
    when fed the GPU's own layer inputs (teacher forcing)."""
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    from synth import workloads as WL
    M = 1
    S = WL.Step40(dev, m=M, n_steps_forced=1)
    L = S.n_layers
    nb = A.bqe_workspace_bytes(S.d, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    A.bqe_workspace_init(ws, nb)
    pool = S.pool.cstruct()
    forced = S.forced[0].contiguous()                       # (L, M, K)
    t_all = torch.zeros(L, M, H, dtype=torch.int16, device=dev)
    resid = S.x0[0].clone()
    snaps = [resid.double().cpu().numpy()]
    EH = E * H
    for l in range(L):
        A.bqe_moe_step(S.d, 1, M, resid, S.wr[l], None, pool, S.tables[l], forced[l], t_all[l], ws, nb)
        snaps.append(resid.double().cpu().numpy())
    rc, det = A.bqe_check(ws)
    assert rc == A.BQE_OK, (A.status_name(rc), det)
    # the whole step as one call: its first layer sees the same input; after
    # 40 chained layers the residual agrees only loosely (the layers add their
    # outputs with fp32 atomics, and bf16 rounding of each layer's input
    # amplifies the different last bits), while a skipped or repeated layer
    # (each moves the residual by ~20 % of its norm) would be far off
    whole = S.x0[0].clone()
    t_whole = torch.zeros(L, M, H, dtype=torch.int16, device=dev)
    A.bqe_moe_step(S.d, L, M, whole, S.wr, None, pool, S.tables, forced, t_whole, ws, nb)
    assert A.bqe_check(ws)[0] == A.BQE_OK
    assert torch.equal(t_whole[0], t_all[0])
    wn = whole.double().cpu().numpy()
    rel = np.linalg.norm(wn - snaps[-1]) / np.linalg.norm(snaps[-1])
    assert rel < 0.1, rel
    step = np.linalg.norm(snaps[-1] - snaps[-2]) / np.linalg.norm(snaps[-1])
    assert step > 3 * rel, (step, rel)
    t_np = t_all.cpu().numpy().view(np.uint16)
    # layer inputs: bf16(rmsnorm(r_l)), within one bf16 step of the fp64 statement
    for l in range(L):
        want = O.rmsnorm_to_bf16(snaps[l])
        diff = np.abs(t_np[l].astype(np.int64) - want.astype(np.int64))
        assert diff.max() <= 1 and (diff > 0).mean() < 0.01, l
    router_all = S.wr.cpu().numpy()
    # eight of the 40 layers, every column: each layer's own output (the
    # residual difference) against the oracle fed that layer's GPU input
    for l in (0, 5, 11, 17, 23, 29, 34, 39):
        table = S.tables_np[l]
        fm = np.array([S.fmts[table[e]] for e in range(E + 1)], dtype=np.int32)
        oref, _ = oracle_layer_sampled(fm, lambda e: S.canon(int(table[e])).cpu().numpy(), t_np[l], router_all[l],
                                       None, S.forced_np[0, l], H, I, E, K, None)
        got = snaps[l + 1] - snaps[l]
        check_out(got, oref, rel=1e-4, what="layer %d" % l)


PF_TOL = 5e-3


def _prefill_sample(forced, cnt, budget):
    """Tokens whose outputs the oracle checks at the full prefill size: the
    rows at the tile boundaries of the most loaded expert, one token of each
    of the next three most and the four least loaded experts (the one adding
    the fewest new experts), then tokens adding at most one new expert while
    the set of experts to dequantise stays within `budget`."""
    T = forced.shape[0]
    sets = [set(r.tolist()) for r in forced]
    order = np.argsort(-cnt, kind="stable")
    most = [int(e) for e in order[:4]]
    least = [int(e) for e in order[::-1] if cnt[e] > 0][:4]
    S, sel = {E}, []

    def group(e):
        return [t for t in range(T) if e in sets[t]]
    g = group(most[0])
    for p in (0, 255, 256, 511, 512, len(g) - 1):
        if 0 <= p < len(g) and g[p] not in sel:
            sel.append(g[p])
            S |= sets[g[p]]
    for e in most[1:] + least:
        t = min(group(e), key=lambda t: len(sets[t] - S))
        if t not in sel:
            sel.append(t)
            S |= sets[t]
    rng = np.random.default_rng(9)
    for t in rng.permutation(T):
        t = int(t)
        if len(sel) >= 96:
            break
        new = sets[t] - S
        if t not in sel and (not new or (len(new) == 1 and len(S) < budget)):
            sel.append(t)
            S |= new
    return np.array(sel), most, least


def test_prefill_dsv4_zipf(dev):
    """8192 tokens, Zipf(0.8) forced routing over the mixed-format layer: the
    selection and mixing weights of every token, and sampled outputs (tile
    boundaries of the most loaded expert, the least loaded experts) against
    the oracle."""
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    from synth import workloads as WL
    W = WL.Prefill(dev)
    T = W.T
    nb = A.bqe_prefill_workspace_bytes(W.d, T)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = torch.full((T, H), float("nan"), device=dev)
    idx = torch.zeros(T, K, dtype=torch.int32, device=dev)
    wts = torch.zeros(T, K, dtype=torch.float32, device=dev)
    A.bqe_moe_prefill(W.d, T, W.x, W.wr, W.bias, W.pool.cstruct(), W.table, W.forced, out, 0, idx, wts, ws, nb)
    rc, det = A.bqe_check(ws)
    assert rc == A.BQE_OK, (A.status_name(rc), det)
    out = out.double().cpu().numpy()
    assert np.isfinite(out).all()
    assert np.array_equal(idx.cpu().numpy(), W.forced_np)
    x_bits = W.x.cpu().numpy().view(np.uint16)
    router = W.wr.cpu().numpy()
    ref = O.route(O.bf16_bits_to_f64(x_bits), router, None, K, W.forced_np)
    np.testing.assert_allclose(wts.cpu().numpy(), ref["w"], rtol=1e-5, atol=1e-7)
    cnt = W.counts()
    assert cnt.sum() == T * K and cnt.max() > 512
    sample, most, least = _prefill_sample(W.forced_np, cnt, budget=48)
    cols = np.random.default_rng(3).choice(H, 1024, replace=False)
    cache = {}

    def canon(e):
        if e not in cache:
            cache[e] = W.canon(e).cpu().numpy()
        return cache[e]
    oref, _ = oracle_layer_sampled(W.fmts, canon, x_bits[sample], router, None, W.forced_np[sample], H, I, E, K,
                                   cols)
    check_out(out[sample][:, cols], oref, PF_TOL, PF_TOL, "prefill T=8192")

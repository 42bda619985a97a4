"""GPU parity of the prefill path (bqe_moe_prefill) against the fp64 oracle.

Prefill regroups the tokens of one layer by expert and runs the experts as
grouped GEMMs on the bf16 tensor cores (Strata 4090 post, sections 4 and 5.3:
tensor-core experts must leave the per-token result unchanged), so the oracle
is the decode layer's, evaluated per token.  Bars: top-k indices exact (rows
whose k-th and (k+1)-th keys are within 1e-6 excepted), mixing weights within
1e-5 relative, fp32 outputs within relative L2 5e-3 and max-abs 5e-3 x
max|reference| (the bound set for the bf16 tensor-core path: weights and h
rounded to bf16 once each, fp32 accumulation)."""
import numpy as np
import pytest

import synth
from oracle import moe as O

from gpu_util import DeviceLayer, check_out, check_routing, torch_dev

pytestmark = pytest.mark.gpu

PF_TOL = 5e-3
ALL = [synth.TQ1, synth.Q2_0, synth.Q3_K, synth.MXFP4, synth.NVFP4]


@pytest.fixture(scope="module")
def dev():
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    d = torch_dev()
    torch.cuda.set_device(d)
    return d


def prefill(dl, x_bits, forced=None, use_bias=True, out_init=None, slot_table=None, expect=0):
    """Run bqe_moe_prefill on T = len(x_bits) rows; returns out, idx, w (numpy)."""
    import torch
    A = dl.A
    T = x_bits.shape[0]
    nb = A.bqe_prefill_workspace_bytes(dl.d, T)
    assert nb > 0
    ws = torch.empty(nb, dtype=torch.uint8, device=dl.dev)
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(dl.dev)
    out = (torch.from_numpy(out_init.astype(np.float32)).to(dl.dev) if out_init is not None
           else torch.full((T, dl.H), float("nan"), device=dl.dev))
    idx = torch.zeros(T, dl.K, dtype=torch.int32, device=dl.dev)
    w = torch.zeros(T, dl.K, dtype=torch.float32, device=dl.dev)
    fi = None if forced is None else torch.from_numpy(np.ascontiguousarray(forced, dtype=np.int32)).to(dl.dev)
    table = dl.table if slot_table is None else slot_table
    A.bqe_moe_prefill(dl.d, T, x, dl.wr, dl.bias if use_bias else None, dl.pool.cstruct(), table, fi, out,
                      out_init is not None, idx, w, ws, nb)
    rc, det = A.bqe_check(ws)
    assert rc == expect, (A.status_name(rc), det)
    return out.double().cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def oracle_full(L, x_bits, forced=None, use_bias=True):
    return O.moe_layer(x_bits, L["router"], L["bias"] if use_bias else None, L["experts"], L["fmts"],
                       L["hidden"], L["inter"], L["top_k"], L["n_experts"], forced_idx=forced)


def check_all(L, dl, x_bits, forced=None, use_bias=True):
    out, idx, w = prefill(dl, x_bits, forced, use_bias)
    ref = oracle_full(L, x_bits, forced, use_bias)
    n = check_routing(ref, idx, w, forced)
    assert n >= 0.9 * x_bits.shape[0]
    ok = np.array([forced is not None or ref["gap"][m] >= 1e-6 for m in range(x_bits.shape[0])])
    np.testing.assert_allclose(w[ok], ref["w"][ok], rtol=1e-5, atol=1e-7)
    # rows whose selection is a near-tie may legitimately pick the other expert
    return check_out(out[ok], ref["out"][ok], PF_TOL, PF_TOL, "prefill")


@pytest.mark.parametrize("T", [1, 37, 300])
def test_prefill_tiny_q2_0(dev, T):
    L = synth.tiny_layer(seed=0, m=T)
    check_all(L, DeviceLayer(L, dev), L["x"])


@pytest.mark.parametrize("T", [129, 700])
def test_prefill_mixed_formats_with_bias(dev, T):
    E = 16
    fm = [ALL[e % len(ALL)] for e in range(E)] + [synth.Q3_K]
    L = synth.small_layer(31, fm, 512, 512, E, 3, T, bias_std=0.25)
    check_all(L, DeviceLayer(L, dev), L["x"])


@pytest.mark.parametrize("fmt", ALL)
def test_prefill_single_format_forced(dev, fmt):
    E, K, T = 8, 2, 200
    L = synth.small_layer(40 + fmt, [fmt] * (E + 1), 768, 256, E, K, T)
    rng = np.random.default_rng(fmt)
    forced = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    check_all(L, DeviceLayer(L, dev), L["x"], forced)


def test_prefill_tile_boundaries_and_empty_experts(dev):
    """Expert 0 takes every token (600 rows: tiles of 256, 256, 88), expert 1
    exactly 256, expert 2 257, expert 3 the rest; experts 4..7 none; one token
    picks the same expert twice (two pairs, both counted)."""
    E, K, T = 8, 2, 600
    fm = [synth.Q2_0, synth.TQ1, synth.Q3_K, synth.MXFP4, synth.Q2_0, synth.TQ1, synth.Q3_K, synth.MXFP4, synth.Q2_0]
    L = synth.small_layer(55, fm, 512, 256, E, K, T)
    forced = np.zeros((T, K), np.int32)
    forced[:, 1] = np.where(np.arange(T) < 256, 1, np.where(np.arange(T) < 513, 2, 3))
    forced[599] = [3, 3]
    check_all(L, DeviceLayer(L, dev), L["x"], forced)


def test_prefill_medium_zipf_all_outputs(dev):
    """2048 tokens, 64 experts, Zipf(0.8) routing in the mixed formats: every
    output element against the oracle (several tiles per popular expert,
    ragged tails everywhere)."""
    E, K, T, H, I = 64, 4, 2048, 1024, 512
    rng = np.random.default_rng(77)
    fm = list(synth.assign_formats(rng, E)) + [synth.Q2_0]
    L = synth.small_layer(78, fm, H, I, E, K, T, bias_std=0.25)
    forced = synth.zipf_forced_idx(rng, T, E, K, 0.8, rng.permutation(E))
    cnt = np.bincount(forced.reshape(-1), minlength=E)
    assert cnt.max() > 256
    check_all(L, DeviceLayer(L, dev), L["x"], forced)


def test_prefill_accumulates(dev):
    L = synth.tiny_layer(seed=3, m=50)
    dl = DeviceLayer(L, dev)
    init = np.random.default_rng(1).standard_normal((50, L["hidden"])).astype(np.float32)
    out, _, _ = prefill(dl, L["x"], out_init=init)
    ref = oracle_full(L, L["x"])
    check_out(out - init, ref["out"], PF_TOL, PF_TOL, "accumulate")


def test_prefill_bad_slot_reports_device_error(dev):
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    L = synth.tiny_layer(seed=4, m=20)
    dl = DeviceLayer(L, dev)
    table = dl.table.clone()
    table[0] = 10_000
    forced = np.zeros((20, 2), np.int32)
    forced[:, 1] = 1
    prefill(dl, L["x"], forced, slot_table=table, expect=A.BQE_EDEVICE)
    # the next call with a good table succeeds on a fresh workspace
    prefill(dl, L["x"], forced)
    assert torch.cuda.is_available()


def test_prefill_deterministic(dev):
    L = synth.tiny_layer(seed=6, m=333)
    dl = DeviceLayer(L, dev)
    a = prefill(dl, L["x"])[0]
    b = prefill(dl, L["x"])[0]
    assert np.array_equal(a, b)


def test_prefill_host_argument_errors(dev):
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    L = synth.tiny_layer(seed=7, m=4)
    dl = DeviceLayer(L, dev)
    assert A.bqe_prefill_workspace_bytes(dl.d, 0) == 0
    nb = A.bqe_prefill_workspace_bytes(dl.d, 4)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    x = torch.zeros(4, L["hidden"], dtype=torch.int16, device=dev)
    out = torch.zeros(4, L["hidden"], device=dev)
    with pytest.raises(A.BqeError) as e:
        A.bqe_moe_prefill(dl.d, 4, x, dl.wr, None, dl.pool.cstruct(), dl.table, None, out, 0, None, None, ws,
                          nb - 256)
    assert e.value.status == A.BQE_ENOSPC
    with pytest.raises(A.BqeError) as e:
        A.bqe_moe_prefill(dl.d, 4, None, dl.wr, None, dl.pool.cstruct(), dl.table, None, out, 0, None, None, ws, nb)
    assert e.value.status == A.BQE_EINVAL


@pytest.mark.parametrize("T", [37, 300])
def test_prefill_bf16_operands(dev, T):
    """bf16 for every expert (the operand type the pages' workload names):
    weights and h keep 8 significant bits, so the bound is the relative L2
    5e-3 and max-abs 1e-2 x max|reference| (its inherent rounding reaches
    about 5e-3 in max-abs on these inputs)."""
    from bit_quantised_expert_gb300 import _abi as A
    L = synth.tiny_layer(seed=0, m=T)
    dl = DeviceLayer(L, dev)
    A.bqe_set_prefill_f16(False)
    try:
        out, idx, w = prefill(dl, L["x"])
    finally:
        A.bqe_set_prefill_f16(True)
    ref = oracle_full(L, L["x"])
    ok = ref["gap"] >= 1e-6
    check_routing(ref, idx, w)
    check_out(out[ok], ref["out"][ok], PF_TOL, 2 * PF_TOL, "prefill bf16")


def test_prefill_f16_range_is_reported(dev):
    """A Q2_0 block scale with 3|d| above the fp16 maximum cannot be held as
    fp16 weights: the call reports BQE_EUNSUPPORTED (detail 11); with bf16
    operands the same layer runs."""
    from bit_quantised_expert_gb300 import _abi as A
    L = synth.tiny_layer(seed=8, m=8)
    canon = L["experts"][3].copy()
    canon[16:18] = np.frombuffer(np.float16(30000.0).tobytes(), np.uint8)  # d of W1's first block
    L["experts"][3] = canon
    dl = DeviceLayer(L, dev)
    forced = np.tile(np.array([[3, 5]], np.int32), (8, 1))
    prefill(dl, L["x"], forced, expect=A.BQE_EUNSUPPORTED)
    A.bqe_set_prefill_f16(False)
    try:
        prefill(dl, L["x"], forced)
    finally:
        A.bqe_set_prefill_f16(True)

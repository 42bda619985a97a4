"""Expert cache (least-recently-used slot replacement in a pool smaller than
the set of experts; Strata 4090 post, section 5, second paragraph; field
report, section 3B).  CPU: the oracle on hand-worked sequences, then the
library's slot choice against it.  GPU: layers served from an undersized
pool, uploads on their own stream (also one layer ahead), against the
all-resident pool and the fp64 oracle."""
import ctypes

import numpy as np
import pytest

import synth
from oracle import cache as OC

TQ1, Q2_0, Q3_K, MXFP4 = 1, 2, 3, 4


# ---------------------------------------------------------------------------
# oracle pins: hand-worked sequences
# ---------------------------------------------------------------------------
def test_oracle_lru_by_hand():
    # one layer, 4 experts of one format, 2 slots
    c = OC.LruCache(1, 4, [Q2_0, Q2_0], [Q2_0] * 4)
    assert c.plan(0, [0]) == [(0, True, -1)]          # plan 0: the never-used slot 0
    assert c.plan(0, [1]) == [(1, True, -1)]          # plan 1: slot 1 (slot 0 used by the previous plan)
    assert c.plan(0, [2]) == [(0, True, 0)]           # plan 2: slot 0 (used at 0) evicts expert 0
    assert c.plan(0, [1]) == [(1, False, -1)]         # plan 3: hit
    assert c.plan(0, [3]) == [(0, True, 2)]           # plan 4: slot 1 used by plan 3 is held back
    assert c.plan(0, [3, 3]) == [(0, False, -1), (0, False, -1)]  # a repeat is a hit
    # two misses, one free slot: refused, nothing changes
    assert c.plan(0, [0, 2]) is None
    assert c.plan(0, [0]) == [(1, True, 1)]           # the same plan number as the refused one


def test_oracle_formats_and_pins():
    # slots: 0 ternary, 1 Q3_K, 2 ternary; experts 0..2 ternary, 3 Q3_K (both layers)
    c = OC.LruCache(2, 4, [TQ1, Q3_K, TQ1], [TQ1, TQ1, TQ1, Q3_K] * 2)
    assert c.plan(0, [3, 0]) == [(1, True, -1), (0, True, -1)]
    assert c.plan(1, [3]) is None                # the only Q3_K slot is held by the previous plan
    assert c.plan(1, [0]) == [(2, True, -1)]     # a ternary expert never lands in the Q3_K slot
    assert c.plan(1, [3]) == [(1, True, 3)]      # two plans later: layer 1's expert 3 evicts layer 0's


# ---------------------------------------------------------------------------
# the library's slot choice against the oracle
# ---------------------------------------------------------------------------
def _fake_pool(A, d, fmts):
    p = A.bqe_pool()
    p.base = 1 << 20
    p.base_bytes = 1 << 40
    p.slot_off = 1 << 21
    p.slot_fmt = 1 << 22
    p.n_slots = len(fmts)
    return p


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_library_lru_matches_oracle(seed):
    from bit_quantised_expert_gb300 import _abi as A
    rng = np.random.default_rng(seed)
    L, E = 3, 16
    d = A.desc(1024, 768, E, 4)
    expert_fmt = rng.choice([TQ1, Q2_0, Q3_K], size=(L, E)).astype(np.int32)
    shared = [Q2_0] * L
    managed = [TQ1] * 5 + [Q2_0] * 4 + [Q3_K] * 3
    rng.shuffle(managed)
    pool_fmt = np.array(shared + managed, np.int32)
    first = L
    h = A.bqe_cache_create(d, L, expert_fmt, _fake_pool(A, d, pool_fmt), pool_fmt, first, len(managed), 1 << 23)
    try:
        ref = OC.LruCache(L, E, managed, expert_fmt.reshape(-1).tolist())
        zipf = synth.zipf_probs(E, 1.0)
        n_req = n_hit = n_miss = n_ev = 0
        for step in range(200):
            layer = int(rng.integers(L))
            req = rng.choice(E, size=int(rng.integers(1, 6)), p=zipf).astype(np.int32)
            want = ref.plan(layer, req.tolist())
            if want is None:
                with pytest.raises(A.BqeError) as ex:
                    A.bqe_cache_plan(h, layer, req)
                assert ex.value.status == A.BQE_ENOSPC
                continue
            slots, miss, ev = A.bqe_cache_plan(h, layer, req)
            assert [(int(s) - first, bool(m), int(e)) for s, m, e in zip(slots, miss, ev)] == want, step
            for s, m, e in want:
                n_req += 1
                n_hit += not m
                n_miss += m
                n_ev += m and e >= 0
        st = A.bqe_cache_stats_get(h)
        assert (st["requests"], st["hits"], st["misses"], st["evictions"]) == (n_req, n_hit, n_miss, n_ev)
        assert n_miss > 20 and n_hit > 20
    finally:
        A.bqe_cache_destroy(h)


def test_library_cache_rejects_bad_arguments():
    from bit_quantised_expert_gb300 import _abi as A
    d = A.desc(1024, 768, 8, 2)
    fm = np.full(6, Q2_0, np.int32)
    pool = _fake_pool(A, d, fm)
    with pytest.raises(A.BqeError):
        A.bqe_cache_create(d, 2, np.full((2, 8), Q2_0, np.int32), pool, fm, 2, 5, 1 << 23)  # slots past the pool
    with pytest.raises(A.BqeError):
        A.bqe_cache_create(d, 2, np.full((2, 8), 9, np.int32), pool, fm, 2, 4, 1 << 23)  # bad format
    h = A.bqe_cache_create(d, 2, np.full((2, 8), Q2_0, np.int32), pool, fm, 2, 4, 1 << 23)
    try:
        with pytest.raises(A.BqeError):
            A.bqe_cache_plan(h, 2, np.array([0], np.int32))  # layer out of range
        with pytest.raises(A.BqeError):
            A.bqe_cache_plan(h, 0, np.array([8], np.int32))  # expert out of range
    finally:
        A.bqe_cache_destroy(h)


# ---------------------------------------------------------------------------
# GPU: layers served through the cache
# ---------------------------------------------------------------------------
@pytest.mark.gpu
@pytest.mark.parametrize("ahead", [False, True])
def test_layers_through_an_undersized_pool(ahead):
    """4 layers x 32 routed experts (plus one shared each) served from 40
    managed slots: every output equals the all-resident pool's (same
    kernels, same inputs) and the oracle's; with `ahead`, layer l + 1's
    experts are fetched before layer l runs (the routing is given)."""
    import torch
    from bit_quantised_expert_gb300 import _abi as A
    from bit_quantised_expert_gb300.pool import SlotPool
    from oracle import moe as O
    from gpu_util import check_out
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(7)
    L, H, I, E, K, M = 4, 1024, 768, 32, 4, 2
    d = A.desc(H, I, E, K)
    efmt = rng.choice([TQ1, Q2_0, Q3_K, MXFP4], size=(L, E)).astype(np.int32)
    canon = [[synth.random_expert(rng, int(efmt[l, e]), H, I) for e in range(E)] for l in range(L)]
    shared = [synth.random_expert(rng, Q2_0, H, I) for _ in range(L)]
    routers = [torch.from_numpy(synth.router_weights(rng, E, H)).to(dev) for _ in range(L)]
    # pinned host copies of every routed expert's canonical bytes
    host = [[torch.from_numpy(canon[l][e]).pin_memory() for e in range(E)] for l in range(L)]
    src = (ctypes.c_void_p * (L * E))(*[host[l][e].data_ptr() for l in range(L) for e in range(E)])
    # the all-resident pool: slot l * (E + 1) + e, shared last in each layer
    full = SlotPool(d, [int(f) for l in range(L) for f in list(efmt[l]) + [Q2_0]], dev)
    for l in range(L):
        for e in range(E):
            full.upload(l * (E + 1) + e, canon[l][e])
        full.upload(l * (E + 1) + E, shared[l])
    full_tab = torch.arange(L * (E + 1), dtype=torch.int32, device=dev)
    # the cache: shared experts in slots 0..L-1, then 40 managed slots
    managed = [TQ1] * 10 + [Q2_0] * 10 + [Q3_K] * 10 + [MXFP4] * 10
    cfmt = np.array([Q2_0] * L + managed, np.int32)
    small = SlotPool(d, cfmt, dev)
    for l in range(L):
        small.upload(l, shared[l])
    tab = torch.full((L, E + 1), -1, dtype=torch.int32, device=dev)
    tab[:, E] = torch.arange(L, dtype=torch.int32, device=dev)
    h = A.bqe_cache_create(d, L, efmt, small.cstruct(), cfmt, L, len(managed), tab)
    staging = torch.empty(32 << 20, dtype=torch.uint8, device=dev)
    up = torch.cuda.Stream()
    cs = torch.cuda.current_stream()
    nb = A.bqe_workspace_bytes(d, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    A.bqe_workspace_init(ws, nb)
    zipf = synth.zipf_probs(E, 1.0)
    try:
        seq = []
        for step in range(12):  # three passes over the 4 layers
            l = step % L
            forced = np.stack([rng.choice(E, size=K, replace=False, p=zipf) for _ in range(M)]).astype(np.int32)
            x_bits = synth.x_bf16(rng, M, H)
            seq.append((l, forced, x_bits))
        plans = {}

        def fetch(i):
            l, forced, _ = seq[i]
            plans[i] = A.bqe_cache_fetch(h, l, forced.reshape(-1), src, staging, up, cs)[0]

        outs = []
        if not ahead:
            for i in range(len(seq)):
                fetch(i)
                A.bqe_cache_ready(h, plans[i], cs)
                outs.append(_run(A, d, seq[i], small, tab[seq[i][0]], routers, ws, nb, dev))
                A.bqe_cache_done(h, plans[i], cs)
        else:
            fetch(0)
            for i in range(len(seq)):
                if i + 1 < len(seq):
                    fetch(i + 1)  # its uploads run while layer i computes
                A.bqe_cache_ready(h, plans[i], cs)
                outs.append(_run(A, d, seq[i], small, tab[seq[i][0]], routers, ws, nb, dev))
                A.bqe_cache_done(h, plans[i], cs)
        torch.cuda.synchronize()
        st = A.bqe_cache_stats_get(h)
        assert st["misses"] > 20 and st["hits"] > 5 and st["evictions"] > 0
        assert st["requests"] == len(seq) * M * K
        for i, (l, forced, x_bits) in enumerate(seq):
            ref = _run(A, d, seq[i], full, full_tab[l * (E + 1):(l + 1) * (E + 1)], routers, ws, nb, dev)
            check_out(outs[i], ref, rel=1e-5, mabs=1e-5, what="cache step %d" % i)
        # one step against the oracle
        l, forced, x_bits = seq[-1]
        fm_l = [int(f) for f in efmt[l]] + [Q2_0]
        experts_l = canon[l] + [shared[l]]
        r = O.moe_layer(x_bits, routers[l].cpu().numpy(), None, experts_l, fm_l, H, I, K, E, forced_idx=forced)
        check_out(outs[-1], r["out"], what="cache vs oracle")
    finally:
        A.bqe_cache_destroy(h)


def _run(A, d, item, pool, table, routers, ws, nb, dev):
    import torch
    l, forced, x_bits = item
    M = x_bits.shape[0]
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(dev)
    out = torch.zeros(M, d.hidden, device=dev)
    fi = torch.from_numpy(forced).to(dev)
    A.bqe_moe_layer_forward(d, M, x, routers[l], None, pool.cstruct(), table, fi, out, 0, None, None, ws, nb)
    rc, det = A.bqe_check(ws)
    assert rc == A.BQE_OK, (A.status_name(rc), det)
    return out.double().cpu().numpy()

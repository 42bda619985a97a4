"""Full-size seeded workloads built on the device.

Inputs only: every byte comes from synth's seeded generators (torch backend,
one generator per slot so any slot can be regenerated for the oracle); the
library's own bqe_pool_pack_slot lays the slots out.  Shapes are those of a
DeepSeek-V4.1-Flash MoE layer (field report, sections 1-2): hidden 5120,
expert intermediate 2304, 384 routed experts + 1 shared, top-6.

  fp4_layer    one layer, every expert MXFP4 (4.25 bpw), zero bias
  mixed_layer  one layer, experts ternary / Q2_0 / Q3_K in the weight shares
               42.8 / 39.2 / 18.0 % (Strata 4090 post, section 5.1), shared
               expert Q2_0, selection bias N(0, 0.25)
  step40       40 layers over a 4288-slot pool (field report, section 3B:
               4288 expert slots) in the same mixed shares, Zipf(1.0)
               popularity, slot aliasing for cold experts
"""
from __future__ import annotations

import numpy as np

from . import (MXFP4, NVFP4, Q2_0, assign_formats, expert_bytes, largest_remainder_counts, torch_random_expert,
               zipf_forced_idx, MIX_SHARES)

H, I, E, K = 5120, 2304, 384, 6


def slot_generator(device, seed: int, slot: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(slot))
    return g


def canon_slot(device, seed: int, slot: int, fmt: int, hidden=H, inter=I):
    """Canonical bytes of one slot (uint8 device tensor), reproducible from (seed, slot)."""
    return torch_random_expert(slot_generator(device, seed, slot), fmt, hidden, inter, device)


def build_pool(device, seed: int, fmts, hidden=H, inter=I, n_experts=E, top_k=K):
    from bit_quantised_expert_gb300 import _abi as A
    from bit_quantised_expert_gb300.pool import SlotPool
    d = A.desc(hidden, inter, n_experts, top_k)
    pool = SlotPool(d, fmts, device)
    for s, f in enumerate(fmts):
        pool.upload(s, canon_slot(device, seed, s, int(f), hidden, inter))
    return d, pool


def router_and_inputs(device, seed: int, n_layers: int, m: int, n_x: int, bias_std: float, n_experts=E):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 7919 + 17)
    wr = torch.randn(n_layers, n_experts, H, generator=g, device=device) / np.sqrt(H)
    bias = None
    if bias_std > 0:
        bias = torch.randn(n_layers, n_experts, generator=g, device=device) * bias_std
    xs = torch.randn(n_x, m, H, generator=g, device=device).to(torch.bfloat16).view(torch.int16)
    return wr.contiguous(), bias, xs.contiguous()


class Layer:
    """One decode layer on the device with a bank of n_x input batches.
    Expert e < n_experts is routed, expert n_experts is the shared one."""

    def __init__(self, device, seed: int, fmts, m: int, n_x: int, bias_std: float):
        import torch
        self.device, self.seed, self.m = device, seed, m
        self.fmts = np.asarray(fmts, dtype=np.int32)
        self.E = len(self.fmts) - 1
        self.d, self.pool = build_pool(device, seed, self.fmts, n_experts=self.E)
        wr, bias, xs = router_and_inputs(device, seed, 1, m, n_x, bias_std, n_experts=self.E)
        self.wr, self.bias, self.xs = wr[0].contiguous(), (None if bias is None else bias[0].contiguous()), xs
        self.table = torch.arange(self.E + 1, dtype=torch.int32, device=device)

    def canon(self, slot):
        return canon_slot(self.device, self.seed, slot, int(self.fmts[slot]))

    def expert_bytes(self, e):
        return expert_bytes(int(self.fmts[e]), H, I)


def fp4_layer(device, seed=1, m=1, n_x=64, n_experts=E, fmt=MXFP4):
    """Every expert in one FP4 format (MXFP4, or NVFP4 with fmt=5), zero bias."""
    return Layer(device, seed, [fmt] * (n_experts + 1), m, n_x, 0.0)


def mixed_fmts(seed: int, n: int) -> np.ndarray:
    return assign_formats(np.random.default_rng(seed), n)


def mixed_layer(device, seed=2, m=1, n_x=64, n_experts=E):
    fm = np.concatenate([mixed_fmts(seed, n_experts), [Q2_0]]).astype(np.int32)
    return Layer(device, seed, fm, m, n_x, 0.25)


class Step40:
    """40 chained layers over one slot pool: slots 0..4287 routed (mixed
    formats), slots 4288..4327 the per-layer shared experts (Q2_0)."""

    N_LAYERS, N_SLOTS, PRIVATE = 40, 4288, 107

    def __init__(self, device, seed=3, m=1, n_steps_forced=16, zipf_s=1.0, n_layers=None):
        import torch
        self.device, self.seed, self.m = device, seed, m
        L = self.N_LAYERS if n_layers is None else n_layers
        self.n_layers = L
        routed = mixed_fmts(seed, self.N_SLOTS)
        self.fmts = np.concatenate([routed, np.full(L, Q2_0, np.int32)]).astype(np.int32)
        self.d, self.pool = build_pool(device, seed, self.fmts)
        wr, _, _ = router_and_inputs(device, seed, L, m, 1, 0.0)
        self.wr = wr
        rng = np.random.default_rng(seed + 99)
        tables = np.zeros((L, E + 1), dtype=np.int32)
        self.perm = []
        for l in range(L):
            perm = rng.permutation(E)            # perm[r] = expert of popularity rank r
            self.perm.append(perm)
            for r, e in enumerate(perm):
                tables[l, e] = l * self.PRIVATE + (r % self.PRIVATE)
            tables[l, E] = self.N_SLOTS + l
        self.tables_np = tables
        self.tables = torch.from_numpy(tables).to(device)
        # a bank of forced Zipf routings (one per step, per layer, per row)
        self.forced_np = np.stack([
            np.stack([zipf_forced_idx(rng, m, E, K, zipf_s, self.perm[l]) for l in range(L)])
            for _ in range(n_steps_forced)])  # (steps, L, m, K)
        self.forced = torch.from_numpy(self.forced_np).to(device)
        g = torch.Generator(device=device)
        g.manual_seed(seed * 31 + 5)
        self.x0 = (torch.randn(n_steps_forced, m, H, generator=g, device=device)
                   .to(torch.bfloat16).to(torch.float32).contiguous())

    def canon(self, slot):
        return canon_slot(self.device, self.seed, slot, int(self.fmts[slot]))

    def layer_bytes(self, l, step):
        idx = self.forced_np[step, l]
        slots = {int(self.tables_np[l, e]) for e in idx.reshape(-1)} | {int(self.tables_np[l, E])}
        return sum(expert_bytes(int(self.fmts[s]), H, I) for s in slots)


class LayerSet:
    """n_inst independent decode layers (own router, bias, shared expert and
    routed experts) in one slot pool, so that consecutive calls can rotate
    through layers whose combined weights exceed L2.  Instance i owns slots
    i*(n_experts+1) .. i*(n_experts+1)+n_experts (its shared expert last)."""

    def __init__(self, device, kind: str, n_inst: int, seed: int, m: int, n_x: int, n_experts=E):
        import torch
        self.device, self.seed, self.m, self.E, self.n_inst = device, seed, m, n_experts, n_inst
        per = n_experts + 1
        fm = []
        for i in range(n_inst):
            if kind in ("fp4", "nvfp4"):
                fm.append(np.full(per, MXFP4 if kind == "fp4" else NVFP4, np.int32))
            else:
                fm.append(np.concatenate([mixed_fmts(seed * 101 + i, n_experts), [Q2_0]]).astype(np.int32))
        self.fmts = np.concatenate(fm)
        self.d, self.pool = build_pool(device, seed, self.fmts, n_experts=n_experts)
        wr, bias, xs = router_and_inputs(device, seed, n_inst, m, n_x, 0.0 if kind in ("fp4", "nvfp4") else 0.25,
                                         n_experts=n_experts)
        self.wr = [wr[i].contiguous() for i in range(n_inst)]
        self.bias = None if bias is None else [bias[i].contiguous() for i in range(n_inst)]
        self.xs = xs
        self.tables = [torch.arange(i * per, (i + 1) * per, dtype=torch.int32, device=device) for i in range(n_inst)]

    def slot(self, inst, e):
        return inst * (self.E + 1) + e

    def canon(self, slot):
        return canon_slot(self.device, self.seed, slot, int(self.fmts[slot]))

    def expert_bytes(self, inst, e):
        return expert_bytes(int(self.fmts[self.slot(inst, e)]), H, I)


class Prefill:
    """One mixed-format layer (as mixed_layer) over T token rows: x bf16
    N(0, 1) and a forced Zipf(s) routing, expert perm[r] having rank r (with
    T = 8192, s = 0.8: about 128 rows per expert on average, a few thousand on
    the most popular one).  The selection bias N(0, 0.25) is passed but has no
    effect under forced routing."""

    def __init__(self, device, seed=5, T=8192, zipf_s=0.8, n_experts=E):
        import torch
        lay = mixed_layer(device, seed=seed, m=1, n_x=1, n_experts=n_experts)
        self.layer, self.T, self.E = lay, T, n_experts
        self.d, self.pool, self.wr, self.bias, self.table, self.fmts = (lay.d, lay.pool, lay.wr, lay.bias,
                                                                         lay.table, lay.fmts)
        rng = np.random.default_rng(seed * 13 + 1)
        self.perm = rng.permutation(n_experts)
        self.forced_np = zipf_forced_idx(rng, T, n_experts, K, zipf_s, self.perm)
        self.forced = torch.from_numpy(self.forced_np).to(device)
        g = torch.Generator(device=device)
        g.manual_seed(seed * 7 + 3)
        self.x = torch.randn(T, H, generator=g, device=device).to(torch.bfloat16).view(torch.int16).contiguous()

    def canon(self, slot):
        return self.layer.canon(slot)

    def counts(self):
        return np.bincount(self.forced_np.reshape(-1), minlength=self.E)

    def flops(self):
        """Tensor-core FLOPs of the expert GEMMs: every (token, expert) row of
        the routed experts and the shared expert, 3 matrices of H x I."""
        return 2.0 * 3 * H * I * self.T * (K + 1)

#!/usr/bin/env python
"""Benchmark of the block-quantised MoE expert layer (decode) on GB300.

Metric: MoE layer decode expert-byte GB/s = bytes of the distinct experts a
call streams (each read once) / layer time, router included; also us/layer,
tokens/s and the fraction of measured HBM bandwidth.

Default workload: one DeepSeek-V4.1-Flash-shaped MoE layer, every expert
MXFP4 (hidden 5120, inter 2304, 384 routed + 1 shared, top-6), M = 1 token
row; seeded synthetic weights and activations generated on the device.
Consecutive timed steps rotate over 4 independent layer instances (own
router, shared and routed experts), so every step streams weights that are
not in L2 (inputs larger than L2).  Other workloads: --workload mixed-m1 | mixed-m6 | step40-m1 | step40-m6,
and --workload prefill (one mixed-format layer over 8192 tokens, tcgen05 grouped GEMMs; tokens/s and
tensor TFLOP/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bqe|reference]

Under torchrun (N > 1) every rank runs an independent replica of the layer
(replicas only: the decode layer has no exchange step); the time is the max
over ranks and the value counts the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# DRAM bytes read + written per layer call by k_experts<0> and k_finalize_a on the MXFP4 M=1 layer
# (ncu dram__bytes_read.sum + dram__bytes_write.sum, profiles/k_experts_decode_fp4_m1_E64.md), or None
# while either kernel has changed since that capture.
DECODE_FP4_M1_TRAFFIC = (87.86 + 1.69 + 0.67) * 1e6

METRIC = "MoE layer decode: expert-byte GB/s (% of HBM peak) and us/layer at M=1 and M=6"
HBM_FALLBACK_GBS = 6800.0
WORKLOADS = {
    "fp4-m1": "dsv4flash-moe-layer-mxfp4-decode-M1",
    "mixed-m1": "dsv4flash-moe-layer-mixed-tq1-q2_0-q3_k-decode-M1",
    "mixed-m6": "dsv4flash-moe-layer-mixed-tq1-q2_0-q3_k-decode-M6",
    "step40-m1": "dsv4flash-40-layer-step-4288-slot-pool-M1",
    "step40-m6": "dsv4flash-40-layer-step-4288-slot-pool-M6",
    "prefill": "dsv4flash-moe-layer-mixed-prefill-T8192-zipf0.8",
}
PREFILL_METRIC = "MoE layer prefill: tokens/s and expert-GEMM TFLOP/s at T=8192 (Zipf 0.8 routing)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["bqe", "reference"], default="bqe")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="fp4-m1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--soak-s", type=float, default=2.0, help="untimed load before timing, for clock samples")
    ap.add_argument("--variant", type=int, default=1, help="MXFP4 W1/W3 inner loop: 0 fp32 FMA, 1 f16-input FMA")
    ap.add_argument("--instances", type=int, default=4, help="layer instances rotated so weights exceed L2")
    ap.add_argument("--diag", action="store_true", help="print per-CTA cycle accounting of the expert kernels to stderr")
    ap.add_argument("--experts", type=int, default=384,
                    help="routed experts in the pool (profiling a smaller pool; per-call work is unchanged)")
    ap.add_argument("--tokens", type=int, default=8192, help="prefill: token rows per call")
    ap.add_argument("--panels", default=None, help="decode: max panels per work item, 'A,B' (diagnostic)")
    ap.add_argument("--preload", default=None,
                    help="decode: max shared-expert stages streamed before the wait, 'A,B' (diagnostic)")
    ap.add_argument("--fused", action="store_true", help="decode: the single-kernel layer (bqe_set_fused)")
    ap.add_argument("--cpu-oracle-sample", default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    return HBM_FALLBACK_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the sustained measurement (the GEMM
    kernels run for milliseconds inside a longer step), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        for k in ("bf16_tflops_sustained", "bf16_tflops"):
            if j.get(k):
                return float(j[k]), "measured %s" % k
    return 1700.0, "fallback sustained"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled=True):
        self.p = None
        self.lines = []
        if not enabled:
            return
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]), hw=f[5], hwt=f[6],
                                 swt=f[7], swp=f[8]))
            except ValueError:
                continue
        if not rows:
            return None
        sm = sorted(r["sm"] for r in rows)
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                            ("swp", "sw_power_cap")):
                if r[k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------- distributed
def dist_setup(n):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce_device():
    import torch.distributed as dist
    return "cpu" if dist.get_backend() == "gloo" else "cuda"


def reduce_max(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def replica_throughput(units_local, seconds_local, world):
    """Whole-job throughput of independent replicas: the units every rank
    processed over the slowest rank's time."""
    return reduce_sum(float(units_local), world) / reduce_max(float(seconds_local), world)


# ------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(workload: str, reps: int = 1):
    """Time the oracle (as it stands) on a bounded sample of the workload on the
    host cores.  Returns (expert bytes, seconds, sample description)."""
    import numpy as np
    import synth
    from oracle import moe as O
    rng = np.random.default_rng(12345)
    H, I, E, K = 5120, 2304, 384, 6
    if workload == "prefill":
        # two tokens of the prefill layer: router over both, 2 x (6 routed + shared) expert FFNs
        fm = [synth.TQ1, synth.Q2_0, synth.Q3_K, synth.TQ1, synth.Q2_0, synth.TQ1, synth.Q2_0]
        experts = [synth.random_expert(rng, int(f), H, I) for f in fm]
        router = synth.router_weights(rng, E, H)
        x = synth.x_bf16(rng, 2, H)
        forced = np.array([[0, 1, 2, 3, 4, 5], [5, 4, 3, 2, 1, 0]], dtype=np.int32)
        t0 = time.perf_counter()
        for _ in range(reps):
            O.prefill_rows(x, router, None, experts, np.array(fm, np.int32), H, I, K, 6, forced, [0, 1])
        dt = (time.perf_counter() - t0) / reps
        return 2, dt, ("two prefill tokens of the mixed layer (router over 384 experts, 6 routed + shared expert "
                       "FFN each, experts dequantised once), fp64")
    if workload.startswith("fp4"):
        fm = [synth.MXFP4] * 7
        desc = "one MXFP4 layer call at M=1: router (384 x 5120 fp32) + 6 routed + 1 shared expert FFN, fp64"
    else:
        fm = [synth.TQ1, synth.TQ1, synth.TQ1, synth.Q2_0, synth.Q2_0, synth.Q3_K, synth.Q2_0]
        desc = "one mixed-format layer call at M=1 (3 ternary, 2 Q2_0, 1 Q3_K routed + Q2_0 shared), fp64"
    experts = [synth.random_expert(rng, int(f), H, I) for f in fm]
    router = synth.router_weights(rng, E, H)
    x = synth.x_bf16(rng, 1, H)
    forced = np.arange(6, dtype=np.int32)[None, :]
    nbytes = sum(synth.expert_bytes(int(f), H, I) for f in fm)
    # the router scores all 384 experts; the 7 streamed experts are indices 0..6
    fmts = np.array(fm, dtype=np.int32)
    t0 = time.perf_counter()
    for _ in range(reps):
        O.moe_layer(x, router, None, experts, fmts, H, I, K, 6, forced_idx=forced)
    dt = (time.perf_counter() - t0) / reps
    return nbytes, dt, desc


def run_cpu_baseline(workload: str):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-sample", workload],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "failed: " + r.stderr[-300:]}
    j = json.loads(r.stdout.strip().splitlines()[-1])
    if workload == "prefill":
        return {"value": j["bytes"] / j["seconds"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": j["sample"] + "; %.1f s, single thread" % j["seconds"]}
    return {"value": j["bytes"] / j["seconds"] / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": j["sample"] + "; %.1f s, single thread" % j["seconds"]}


# ----------------------------------------------------------- GPU workloads
def l2_bytes():
    import torch
    return torch.cuda.get_device_properties(0).L2_cache_size


def run_layer(args, rank, world):
    import numpy as np
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    from bit_quantised_expert_gb300 import _abi as A
    from synth import workloads as WL
    import synth

    dev = torch.device("cuda", torch.cuda.current_device())
    A.bqe_set_variant(args.variant)
    if args.panels:
        pa, pb = (int(v) for v in args.panels.split(","))
        A.bqe_set_panels(pa, pb)
    if args.preload is not None:
        pa_, pb_ = (int(v) for v in args.preload.split(","))
        A.bqe_set_preload(pa_, pb_)
    if args.fused:
        A.bqe_set_fused(True)
    M = 6 if args.workload.endswith("m6") else 1
    n_x = 64
    NL = args.instances
    kind = "fp4" if args.workload.startswith("fp4") else "mixed"
    W = WL.LayerSet(dev, kind, NL, seed=1 if kind == "fp4" else 2, m=M, n_x=n_x, n_experts=args.experts)
    d, K_ = W.d, 6
    nb = A.bqe_workspace_bytes(d, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    A.bqe_workspace_init(ws, nb)
    pool = W.pool.cstruct()
    out = torch.zeros(M, 5120, device=dev)
    steps, warm = args.steps, args.warmup
    idx_log = torch.zeros(max(steps, 1), M, K_, dtype=torch.int32, device=dev)
    idx_tmp = torch.zeros(M, K_, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    xbuf = torch.empty_like(W.xs[0])
    xs = [W.xs[i] for i in range(n_x)]

    def fused(inst, ev=None):
        # the production call (the layer entry point), on the current stream
        if ev:
            ev[0].record()
        A.bqe_moe_layer_forward(d, M, xbuf, W.wr[inst], None if W.bias is None else W.bias[inst], pool,
                                W.tables[inst], None, out, 0, idx_tmp, None, ws, nb)
        if ev:
            ev[1].record()

    def layer(inst, ev=None):
        # the same layer as separate kernels: router + top-k, phase A, phase B
        if ev:
            ev[0].record()
        A.bqe_route(d, M, xbuf, W.wr[inst], None if W.bias is None else W.bias[inst], pool, W.tables[inst], None,
                    idx_tmp, None, ws, nb)
        if ev:
            ev[1].record()
        A.bqe_experts_phase(d, M, pool, out, 0, 0, ws, nb)
        if ev:
            ev[2].record()
        A.bqe_experts_phase(d, M, pool, out, 0, 1, ws, nb)
        if ev:
            ev[3].record()

    for i in range(warm):
        xbuf.copy_(xs[i % n_x])
        layer(i % NL)
    torch.cuda.synchronize()
    rc, det = A.bqe_check(ws)
    assert rc == 0, (A.status_name(rc), det)

    # The timed unit is one layer replayed from a CUDA graph (the way a decode
    # loop runs it).  Consecutive steps rotate over NL layer instances whose
    # weights together are several times L2, so every step streams cold
    # weights.  Timing events are nodes inside the graph.
    gev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    fev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    graphs, fgraphs = [], []
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        layer(0)
        fused(0)
    st.wait_stream(side)
    torch.cuda.synchronize()
    for inst in range(NL):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer(inst, gev)
        graphs.append(g)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fused(inst, fev)
        fgraphs.append(g)
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device(), enabled=not args.no_clocks)
    t_end = time.time() + args.soak_s
    i = 0
    while time.time() < t_end:  # untimed load so the clock samples see the GPU busy
        xbuf.copy_(xs[i % n_x])
        fgraphs[i % NL].replay()
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    t_route, t_a, t_b, t_split, t_layer = [], [], [], [], []
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s_ in range(steps):
        xbuf.copy_(xs[s_ % n_x])
        fgraphs[s_ % NL].replay()
        idx_log[s_].copy_(idx_tmp)
        fev[1].synchronize()
        t_layer.append(fev[0].elapsed_time(fev[1]) * 1e-3)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    # the same steps as separate kernels, for the per-kernel breakdown
    for s_ in range(steps):
        xbuf.copy_(xs[s_ % n_x])
        graphs[s_ % NL].replay()
        gev[3].synchronize()
        t_route.append(gev[0].elapsed_time(gev[1]) * 1e-3)
        t_a.append(gev[1].elapsed_time(gev[2]) * 1e-3)
        t_b.append(gev[2].elapsed_time(gev[3]) * 1e-3)
        t_split.append(gev[0].elapsed_time(gev[3]) * 1e-3)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    rc, det = A.bqe_check(ws)
    assert rc == 0, (A.status_name(rc), det)

    idx_np = idx_log.cpu().numpy()
    bytes_e, bytes_a, bytes_b = [], [], []
    for s_ in range(steps):
        inst = s_ % NL
        us = sorted(set(int(e) for e in idx_np[s_].reshape(-1)) | {W.E})
        be = sum(W.expert_bytes(inst, e) for e in us)
        ba = sum(2 * synth.matrix_bytes(int(W.fmts[W.slot(inst, e)]), 2304, 5120) for e in us)  # W1 + W3
        bytes_e.append(be)
        bytes_a.append(ba)
        bytes_b.append(be - ba)
    T = sum(t_layer)
    T_max = reduce_max(T, world)
    total_bytes = reduce_sum(float(sum(bytes_e)), world)
    value = total_bytes / T_max / 1e9
    hbm, hbm_kind = peaks()
    mean = lambda v: sum(v) / len(v)  # noqa: E731
    achieved_a = mean(bytes_a) / mean(t_a) / 1e9
    router_bytes = W.E * 5120 * 4
    achieved_l = (mean(bytes_e) + router_bytes) / mean(t_layer) / 1e9
    l2mb = torch.cuda.get_device_properties(0).L2_cache_size / 2 ** 20
    res = dict(
        metric=METRIC, value=round(value, 2), unit="GB/s", n_gpus=world, steps=steps, warmup=warm,
        ms_per_step=round(T_max / steps * 1e3, 5), higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="fp32-accumulate over %s weights, bf16 activations" % (
            "mxfp4" if kind == "fp4" else "ternary/q2_0/q3_k"),
        data="synthetic (seeded, generated on the device)",
        config=dict(workload=WORKLOADS[args.workload], hidden=5120, inter=2304, n_experts=W.E, top_k=6,
                    n_shared=1, M=M,
                    l2="inputs larger than L2: steps rotate over %d layer instances (%.0f MB of weights streamed "
                       "between reuses vs %.0f MB L2)" % (NL, (NL - 1) * mean(bytes_e) / 1e6, l2mb),
                    parallelism="replicas" if world > 1 else "single-gpu"),
        us_per_layer=round(T_max / steps * 1e6, 3),
        tokens_per_s=round(M * steps * world / T_max, 1),
        frac_of_hbm=round(value / hbm, 4), hbm_peak_gbs=hbm, hbm_peak_kind=hbm_kind,
        expert_bytes_per_step=round(mean(bytes_e)),
        roofline=dict(bound="hbm", achieved=round(achieved_a, 1), peak=hbm, unit="GB/s",
                      frac=round(achieved_a / hbm, 4),
                      traffic=DECODE_FP4_M1_TRAFFIC if (args.workload == "fp4-m1" and not args.fused) else None,
                      kernel="k_experts<0> + finalize (W1/W3 dequant-GEMV + SiLU-GLU)",
                      algorithmic_bytes_per_launch=round(mean(bytes_a)),
                      peak_kind="%s hbm_gbs (burst copy)" % hbm_kind,
                      layer_achieved=round(achieved_l, 1), layer_frac=round(achieved_l / hbm, 4),
                      layer_note="all bytes of the call (experts + router) / layer time"),
        split_kernels=dict(
            note="the same layer as separate kernels (router, W1/W3 + finalize, W2 + finalize)",
            us_per_layer=round(mean(t_split) * 1e6, 3),
            route_us=round(mean(t_route) * 1e6, 3), phase_a_us=round(mean(t_a) * 1e6, 3),
            phase_b_us=round(mean(t_b) * 1e6, 3),
            phase_a_gbs=round(achieved_a, 1), phase_b_gbs=round(mean(bytes_b) / mean(t_b) / 1e9, 1)),
        gpu_launches=5 * steps,  # router, W1/W3 + its finalize, W2 + its finalize
        variant=args.variant,
        timing="CUDA-graph replay per step, events as graph nodes around the layer kernel",
        wall_s_timed_loop=round(wall, 4),
    )
    if clk:
        res["clocks"] = clk

    if args.diag and args.fused:
        # timeline of the single-kernel layer (globaltimer stamps per CTA)
        A.bqe_set_diag(True)
        off = A.bqe_diag_offset(d, M)
        tl = []
        for s_ in range(10):
            A.bqe_workspace_init(ws, nb)
            dv = ws[off:off + 8 * 3 * 1024 * 8].view(torch.int64).view(3, 1024, 8)
            dv[0, 1023, 0] = 2 ** 62
            xbuf.copy_(xs[s_ % n_x])
            fused(s_ % NL)
            torch.cuda.synchronize()
            a = dv[0].cpu().numpy().astype(np.float64)
            t0 = a[1023, 0]
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            rel = (a[:sms, :7] - t0) / 1e3
            tl.append([[float(rel[:, k].min()), float(rel[:, k].mean()), float(rel[:, k].max())] for k in range(7)])
        A.bqe_set_diag(False)
        A.bqe_workspace_init(ws, nb)
        tl = np.array(tl).mean(axis=0)
        names = ["router_done", "logits_seen", "worklist_built", "consumers_done", "epilogue_done",
                 "producer_done", "end"]
        sys.stderr.write("FUSED_TIMELINE_us(min,mean,max) " + json.dumps(
            {n: [round(v, 2) for v in tl[k]] for k, n in enumerate(names)}) + "\n")

    if args.diag:
        # per-CTA cycle accounting (a separate, untimed pass)
        A.bqe_set_diag(True)
        off = A.bqe_diag_offset(d, M)
        nd = 20
        spans = []
        for s_ in range(nd):
            A.bqe_workspace_init(ws, nb) if s_ == 0 else None
            dv = ws[off:off + 8 * 3 * 1024 * 8].view(torch.int64).view(3, 1024, 8)
            dv[:, 1023, 0] = 2 ** 62
            dv[:, 1023, 1] = 0
            dv[:2, 1023, 2] = 2 ** 62  # phases A, B: first and last CTA past the wait
            dv[:2, 1023, 3] = 0
            dv[2, 1023, 4] = 2 ** 62   # finalize kernels: first CTA past the wait, last CTA end
            dv[2, 1023, 5] = 0
            dv[2, 1023, 6] = 2 ** 62
            dv[2, 1023, 7] = 0
            xbuf.copy_(xs[s_ % n_x])
            fused(s_ % NL)  # the layer entry point, eager: kernel parameters carry the diagnostic flag
            torch.cuda.synchronize()
            sp = dv[:, 1023, :].cpu().numpy().astype(np.float64)
            t0 = sp[2, 0]
            spans.append([(sp[k, 1] - sp[k, 0]) / 1e3 for k in (2, 0, 1)] +
                         [(v - t0) / 1e3 for v in (sp[2, 1], sp[0, 0], sp[0, 2], sp[0, 3], sp[0, 1], sp[2, 4],
                                                   sp[2, 5], sp[1, 0], sp[1, 2], sp[1, 3], sp[1, 1], sp[2, 6],
                                                   sp[2, 7])])
        A.bqe_set_diag(False)
        dbg = ws[off:off + 8 * 3 * 1024 * 8].view(torch.int64).view(3, 1024, 8).cpu().numpy()
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        names = ["prod_wait_empty", "prod_issue", "cons_wait_stage", "cons_wait_redbuf", "cons_compute",
                 "epi_wait", "epi_work", "cta_total"]
        rep = {}
        for ph in range(2):
            v = dbg[ph, :sms].astype(np.float64) / nd / 2.07e3  # us per call at 2.07 GHz
            rep["phase_%d" % ph] = {n: [round(float(v[:, k].mean()), 2), round(float(v[:, k].max()), 2)]
                                    for k, n in enumerate(names)}
        ncta = (W.E + 1) // 2
        vr = dbg[2, :ncta].astype(np.float64) / nd / 2.07e3
        rep["router"] = {"cta_gemv_us": [round(float(vr[:, 0].mean()), 2), round(float(vr[:, 0].max()), 2)],
                         "last_cta_total_us": round(float(dbg[2, 1022, 1]) / nd / 2.07e3, 2)}
        rep["router_tail_stamps_us"] = [round(float(v) / nd / 2.07e3, 2) for v in dbg[2, 1021, :8]]
        sp = np.array(spans)
        rep["kernel_span_us(first CTA start -> last CTA end)"] = dict(
            router=round(float(sp[:, 0].mean()), 2), phase_a=round(float(sp[:, 1].mean()), 2),
            phase_b=round(float(sp[:, 2].mean()), 2))
        tl_names = ["router_end", "A_start", "A_first_past_wait", "A_last_past_wait", "A_end", "finA_past_wait",
                    "finA_end", "B_start", "B_first_past_wait", "B_last_past_wait", "B_end", "finB_past_wait",
                    "finB_end"]
        rep["timeline_us(from router start)"] = {n: round(float(sp[:, 3 + k].mean()), 2)
                                                 for k, n in enumerate(tl_names)}
        A.bqe_workspace_init(ws, nb)
        sys.stderr.write("DIAG " + json.dumps(rep) + "\n")

    # ---- end to end through the public call with host buffers --------------
    xh = torch.empty(M, 5120, dtype=torch.int16).pin_memory()
    oh = torch.empty(M, 5120, dtype=torch.float32).pin_memory()
    xd = torch.empty(M, 5120, dtype=torch.int16, device=dev)
    xs_host = [x.cpu() for x in xs]
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for s_ in range(steps):
        inst = s_ % NL
        xh.copy_(xs_host[s_ % n_x])
        e2e_ev[s_][0].record(st)
        xd.copy_(xh, non_blocking=True)
        A.bqe_moe_layer_forward(d, M, xd, W.wr[inst], None if W.bias is None else W.bias[inst], pool,
                                W.tables[inst], None, out, 0, idx_log[s_], None, ws, nb)
        oh.copy_(out, non_blocking=True)
        e2e_ev[s_][1].record(st)
    torch.cuda.synchronize()
    Te = sum(e2e_ev[s_][0].elapsed_time(e2e_ev[s_][1]) * 1e-3 for s_ in range(steps))
    idx_np = idx_log.cpu().numpy()
    be2 = sum(sum(W.expert_bytes(s_ % NL, e) for e in (set(int(v) for v in idx_np[s_].reshape(-1)) | {W.E}))
              for s_ in range(steps))
    Te_max = reduce_max(Te, world)
    res["e2e"] = dict(value=round(reduce_sum(float(be2), world) / Te_max / 1e9, 2), unit="GB/s",
                      h2d_bytes_per_step=M * 5120 * 2, d2h_bytes_per_step=M * 5120 * 4,
                      us_per_layer=round(Te_max / steps * 1e6, 3),
                      note="eager calls through bqe_moe_layer_forward, pinned host x in, host out back")
    return res


def run_step40(args, rank, world):
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    from bit_quantised_expert_gb300 import _abi as A
    from synth import workloads as WL

    dev = torch.device("cuda", torch.cuda.current_device())
    M = 6 if args.workload.endswith("m6") else 1
    S = WL.Step40(dev, m=M)
    d, L = S.d, S.n_layers
    nb = A.bqe_workspace_bytes(d, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    A.bqe_workspace_init(ws, nb)
    pool = S.pool.cstruct()
    resid = torch.zeros(M, 5120, device=dev)
    forced = torch.zeros(L, M, 6, dtype=torch.int32, device=dev)
    nf = S.forced.shape[0]
    st = torch.cuda.current_stream()

    def load(i):
        forced.copy_(S.forced[i % nf])
        resid.copy_(S.x0[i % nf])

    def run():
        # the current stream: inside graph capture this is the capture stream
        A.bqe_moe_step(d, L, M, resid, S.wr, None, pool, S.tables, forced, None, ws, nb)

    for i in range(max(args.warmup, 3)):
        load(i)
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        run()
    st.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        run()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device(), enabled=not args.no_clocks)
    t_end = time.time() + args.soak_s
    i = 0
    while time.time() < t_end:
        load(i)
        g.replay()
        i += 1
    torch.cuda.synchronize()
    steps = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world)
    for s in range(steps):
        load(s)
        evs[s][0].record(st)
        g.replay()
        evs[s][1].record(st)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    rc, det = A.bqe_check(ws)
    assert rc == 0, (A.status_name(rc), det)
    ts = [evs[s][0].elapsed_time(evs[s][1]) * 1e-3 for s in range(steps)]
    by = [sum(S.layer_bytes(l, s % nf) for l in range(L)) for s in range(steps)]
    T = reduce_max(sum(ts), world)
    tot = reduce_sum(float(sum(by)), world)
    hbm, hbm_kind = peaks()
    value = tot / T / 1e9
    res = dict(metric=METRIC, value=round(value, 2), unit="GB/s", n_gpus=world, steps=steps, warmup=args.warmup,
               ms_per_step=round(T / steps * 1e3, 4), higher_is_better=True, scaling="weak", vs_baseline=None,
               dtype="fp32-accumulate over ternary/q2_0/q3_k weights, bf16 activations",
               data="synthetic (seeded, generated on the device)",
               config=dict(workload=WORKLOADS[args.workload], layers=L, slots=4288, M=M,
                           l2="not flushed: each step streams ~3 GB, far above L2",
                           routing="Zipf(1.0) forced selection, scores from the router",
                           parallelism="replicas" if world > 1 else "single-gpu"),
               us_per_layer=round(T / steps / L * 1e6, 3), tokens_per_s=round(M * steps * world / T, 1),
               frac_of_hbm=round(value / hbm, 4), hbm_peak_gbs=hbm, expert_bytes_per_step=round(sum(by) / steps),
               gpu_launches=3 * L * steps, cuda_graph=True)
    if clk:
        res["clocks"] = clk
    return res


def run_prefill(args, rank, world):
    """One mixed-format layer over T = 8192 token rows (Zipf 0.8 forced routing)
    through bqe_moe_prefill, eager calls (8 kernels each, a few ms per call)."""
    import numpy as np
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    from bit_quantised_expert_gb300 import _abi as A
    from synth import workloads as WL

    dev = torch.device("cuda", torch.cuda.current_device())
    W = WL.Prefill(dev, T=args.tokens, n_experts=args.experts)
    T, H = W.T, 5120
    nb = A.bqe_prefill_workspace_bytes(W.d, T)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = torch.empty(T, H, device=dev)
    pool = W.pool.cstruct()
    st = torch.cuda.current_stream()

    def call(x):
        A.bqe_moe_prefill(W.d, T, x, W.wr, W.bias, pool, W.table, W.forced, out, 0, None, None, ws, nb)

    for _ in range(max(args.warmup, 3)):
        call(W.x)
    torch.cuda.synchronize()
    rc, det = A.bqe_check(ws)
    assert rc == 0, (A.status_name(rc), det)
    clocks = ClockSampler(torch.cuda.current_device(), enabled=not args.no_clocks)
    t_end = time.time() + args.soak_s
    while time.time() < t_end:
        call(W.x)
        torch.cuda.synchronize()
    steps = args.steps
    A.bqe_set_diag(True)  # events between the library's kernels, on this stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    per_kernel = []
    barrier(world)
    torch.cuda.synchronize()
    for s_ in range(steps):
        evs[s_][0].record(st)
        call(W.x)
        evs[s_][1].record(st)
        per_kernel.append(A.bqe_prefill_kernel_ms())
    torch.cuda.synchronize()
    barrier(world)
    A.bqe_set_diag(False)
    clk = clocks.stop()
    rc, det = A.bqe_check(ws)
    assert rc == 0, (A.status_name(rc), det)
    ts = [evs[s_][0].elapsed_time(evs[s_][1]) * 1e-3 for s_ in range(steps)]
    Tt = reduce_max(sum(ts), world)
    value = T * steps * world / Tt
    flops = W.flops()
    cnt = W.counts()
    rows = T * 7
    f_w13, f_w2 = 2.0 * 2 * 5120 * 2304 * rows, 2.0 * 5120 * 2304 * rows
    km = {k: sum(p[k] for p in per_kernel) / steps for k in per_kernel[0]}
    bf16_peak, pk_kind = tensor_peak()
    ach = f_w13 / (km["gemm_w13"] * 1e-3) / 1e12
    res = dict(metric=PREFILL_METRIC, value=round(value, 1), unit="tokens/s", n_gpus=world, steps=steps,
               warmup=args.warmup, ms_per_step=round(Tt / steps * 1e3, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None,
               dtype="fp16 tensor-core operands (bf16 for MXFP4 experts), fp32 accumulate; ternary/q2_0/q3_k weights",
               data="synthetic (seeded, generated on the device)",
               config=dict(workload=WORKLOADS["prefill"], hidden=5120, inter=2304, n_experts=W.E, top_k=6,
                           n_shared=1, T=T, routing="Zipf(0.8) forced selection, weights from the router",
                           rows_per_expert=dict(max=int(cnt.max()), median=float(np.median(cnt)),
                                                min=int(cnt.min()), mean=float(cnt.mean())),
                           l2="inputs larger than L2 (x 84 MB, weights ~3.8 GB, grouped operands ~1 GB per call)",
                           parallelism="replicas" if world > 1 else "single-gpu"),
               tflops=round(flops * steps * world / Tt / 1e12, 2),
               expert_gemm_flops_per_step=flops,
               kernel_ms=km,
               roofline=dict(bound="tensor", achieved=round(ach, 1), peak=bf16_peak, unit="TFLOP/s",
                             frac=round(ach / bf16_peak, 4), traffic=None,
                             kernel="k_pf_gemm<0> (W1/W3 grouped GEMM: in-smem dequant + tcgen05 MMA + SiLU-GLU)",
                             algorithmic_flops_per_launch=f_w13,
                             peak_kind="%s bf16 dense (fp16 runs at the same rate)" % pk_kind,
                             w2_achieved=round(f_w2 / (km["gemm_w2"] * 1e-3) / 1e12, 1)),
               gpu_launches=8 * steps,
               timing="eager calls; CUDA events on the calling stream around each call and between its kernels")
    if clk:
        res["clocks"] = clk
    if args.diag:
        # per-role cycle accounting of the two GEMM kernels of one more call
        A.bqe_set_diag(True)
        call(W.x)
        torch.cuda.synchronize()
        A.bqe_set_diag(False)
        off = A.bqe_prefill_diag_offset(W.d, T)
        dv = ws[off:off + 8 * 2 * 256 * 12].view(torch.int64).view(2, 256, 12).cpu().numpy().astype(np.float64)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        names = ["load_wait", "dq_wait_raw", "dq_wait_stage", "dq_work", "mma_wait_a", "mma_issue",
                 "mma_wait_acc", "epi_wait", "epi_work", "cta_total", "items", "mma_wait_b"]
        rep = {}
        for gi, gname in enumerate(("gemm_w13", "gemm_w2")):
            v = dv[gi, :sms]
            rep[gname] = {n: [round(float(v[:, k].mean()) / 2.07e3, 1), round(float(v[:, k].max()) / 2.07e3, 1)]
                          for k, n in enumerate(names) if n != "items"}
            rep[gname]["items_per_cta"] = [float(v[:, 10].mean()), float(v[:, 10].max())]
        sys.stderr.write("PREFILL_DIAG_us(mean,max over CTAs) " + json.dumps(rep) + "\n")
    # end to end: pinned host x in, host out back, every step
    xh = W.x.cpu().pin_memory()
    oh = torch.empty(T, H, dtype=torch.float32).pin_memory()
    xd = torch.empty_like(W.x)
    e2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(min(steps, 10))]
    for s_ in range(len(e2)):
        e2[s_][0].record(st)
        xd.copy_(xh, non_blocking=True)
        call(xd)
        oh.copy_(out, non_blocking=True)
        e2[s_][1].record(st)
    torch.cuda.synchronize()
    Te = reduce_max(sum(a.elapsed_time(b) * 1e-3 for a, b in e2), world)
    res["e2e"] = dict(value=round(T * len(e2) * world / Te, 1), unit="tokens/s", h2d_bytes_per_step=T * H * 2,
                      d2h_bytes_per_step=T * H * 4, ms_per_step=round(Te / len(e2) * 1e3, 3),
                      note="eager bqe_moe_prefill with pinned host x in and host out back")
    return res


def run_reference(args, rank, world):
    """The oracle (fp64, as it stands) on the host cores, one bounded sample per step."""
    if rank != 0:
        return None
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(k, "1")  # before numpy loads its BLAS: report the threads really used
    import numpy as np
    import synth
    from oracle import formats as F
    from oracle import moe as O
    rng = np.random.default_rng(777)
    fmt = synth.MXFP4 if args.workload.startswith("fp4") else synth.Q2_0
    H, I = 5120, 2304
    ex = synth.random_expert(rng, fmt, H, I)
    x = synth.x_bf16(rng, 1, H)
    nbytes = synth.expert_bytes(fmt, H, I)

    def step():
        w1, w3, w2 = F.dequant_expert(fmt, ex, H, I)
        O.expert_ffn(O.bf16_bits_to_f64(x), w1, w3, w2)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    T = time.perf_counter() - t0
    value = nbytes * args.steps / T / 1e9
    sample = "one expert FFN (%s, %d bytes) per step at M=1 in fp64 numpy" % (synth.FMT_NAMES[fmt], nbytes)
    return dict(metric=METRIC, value=round(value, 4), unit="GB/s", n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(T / args.steps * 1e3, 3), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic (seeded)", impl="reference",
                config=dict(workload=WORKLOADS[args.workload], M=1),
                cpu_baseline=dict(value=round(value, 4), unit="GB/s", cores=_threads_used(), kind="oracle",
                                  sample=sample),
                e2e=dict(value=round(value, 4), unit="GB/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def _threads_used():
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count() or 1


def main():
    args = parse()
    if args.cpu_oracle_sample:
        nbytes, dt, desc = cpu_oracle_sample(args.cpu_oracle_sample)
        print(json.dumps(dict(bytes=nbytes, seconds=dt, sample=desc)))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    rank, world, local = dist_setup(args.gpus)
    if args.workload.startswith("step40"):
        res = run_step40(args, rank, world)
    elif args.workload == "prefill":
        res = run_prefill(args, rank, world)
    else:
        res = run_layer(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = run_cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the block-quantised MoE expert layer (decode) on GB300.

Metric: MoE layer decode expert-byte GB/s = bytes of the distinct experts a
call streams (each read once) / layer time, router included; also us/layer,
tokens/s and the fraction of measured HBM bandwidth.

Headline (`value`): one DeepSeek-V4.1-Flash-shaped MoE layer with every
expert MXFP4 (hidden 5120, inter 2304, 384 routed + 1 shared, top-6) at M = 1
token row, seeded synthetic weights and activations generated on the device.
Consecutive timed steps rotate over 4 independent layer instances (own router,
shared and routed experts) and a bank of 64 inputs, so every step streams
weights that are not in L2 (inputs larger than L2).

The default run adds sub-records, timed in interleaved rounds under the same
clock record, each with us/layer as median and p10/p90 over its steps:
  mixed_m1   mixed-format layers (ternary / Q2_0 / Q3_K experts in the weight
             shares 42.8 / 39.2 / 18.0 %, Q2_0 shared, bias N(0, 0.25)), M = 1
  mixed_m6   the same layers at M = 6 independent rows (a batched verify of
             one token and five drafted ones)
  step40_m1  40 chained layers over a 4288-slot pool with Zipf(1.0) routing,
             one CUDA graph per step
--workload picks one of them as the only (headline) record instead;
--workload prefill times one mixed layer over 8192 tokens (tcgen05 grouped
GEMMs: tokens/s and tensor TFLOP/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bqe|reference]

Under torchrun (N > 1) every rank runs an independent replica of the layer
(replicas only: the decode layer has no exchange step); the time is the max
over ranks and the value counts the bytes of all ranks.  --impl reference
times the fp64 oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

H, I, E, K = 5120, 2304, 384, 6
METRIC = "MoE layer decode: expert-byte GB/s (% of HBM peak) and us/layer at M=1 and M=6"
HBM_FALLBACK_GBS = 6800.0
WORKLOADS = {
    "fp4-m1": "dsv4flash-moe-layer-mxfp4-decode-M1",
    "nvfp4-m1": "dsv4flash-moe-layer-nvfp4-decode-M1",
    "mixed-m1": "dsv4flash-moe-layer-mixed-tq1-q2_0-q3_k-decode-M1",
    "mixed-m6": "dsv4flash-moe-layer-mixed-tq1-q2_0-q3_k-decode-M6",
    "step40-m1": "dsv4flash-40-layer-step-4288-slot-pool-M1",
    "step40-m6": "dsv4flash-40-layer-step-4288-slot-pool-M6",
    "prefill": "dsv4flash-moe-layer-mixed-prefill-T8192-zipf0.8",
}
SUB_RECORDS = ("mixed-m1", "mixed-m6", "step40-m1", "nvfp4-m1")
PREFILL_METRIC = "MoE layer prefill: tokens/s and expert-GEMM TFLOP/s at T=8192 (Zipf 0.8 routing)"

# DRAM traffic of one decode-layer launch (k_moe) on the MXFP4 M=1 layer:
# ncu dram__bytes_read.sum + dram__bytes_write.sum of the kernel on a
# 64-expert pool, plus the router rows of the 320 experts that pool lacks
# (5120 x 4 bytes each; what a launch streams besides the router does not
# depend on the pool size).  The figure holds only for the kernel sources
# whose digest is recorded with it; after any change to them the bench
# reports null until a new capture is taken.
KERNEL_SOURCES = ("bit_quantised_expert_gb300/csrc/bqe_moe.cu", "bit_quantised_expert_gb300/csrc/bqe_gemv.cuh",
                  "bit_quantised_expert_gb300/csrc/bqe_internal.cuh")
TRAFFIC_FP4_M1 = dict(sha256="3d7a8eeea843a82e15916b7f3ec2dd861c4a2d10e8bda497b0e79dfb949ff2bc", bytes=142606592)


def kernel_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["bqe", "reference"], default="bqe")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=None,
                    help="time only this workload as the headline (default: fp4-m1 plus the sub-records)")
    ap.add_argument("--sub-steps", type=int, default=60, help="steps per sub-record, split over --rounds")
    ap.add_argument("--rounds", type=int, default=3, help="interleaved rounds of the sub-records")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--soak-s", type=float, default=2.0, help="untimed load before timing, for clock samples")
    ap.add_argument("--instances", type=int, default=4, help="layer instances rotated so weights exceed L2")
    ap.add_argument("--diag", action="store_true", help="print a per-CTA timeline of one decode call to stderr")
    ap.add_argument("--experts", type=int, default=384,
                    help="routed experts in the pool (profiling a smaller pool; per-call work is unchanged)")
    ap.add_argument("--tokens", type=int, default=8192, help="prefill: token rows per call")
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


def pct(v, q):
    """q-th percentile (0..100) of v, linear between order statistics."""
    v = sorted(v)
    if not v:
        return None
    r = (len(v) - 1) * q / 100.0
    lo = int(r)
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (r - lo)


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
# The oracle (fp64 numpy, as it stands) timed on the host cores: P worker
# processes (spawned, never forked) each run one full call of the layer on
# their own seeded inputs; the value counts the expert bytes of all P calls
# over the wall time of the slowest.
def _oracle_worker_init(workload: str, seed: int):
    import numpy as np
    import synth
    global _ORACLE_CASE
    rng = np.random.default_rng(12345 + seed)
    if workload == "prefill":
        # two tokens of the prefill layer: router over both, 6 routed + shared expert FFNs each
        fm = [synth.TQ1, synth.Q2_0, synth.Q3_K, synth.TQ1, synth.Q2_0, synth.TQ1, synth.Q2_0]
        experts = [synth.random_expert(rng, int(f), H, I) for f in fm]
        router = synth.router_weights(rng, E, H)
        x = synth.x_bf16(rng, 2, H)
        forced = np.array([[0, 1, 2, 3, 4, 5], [5, 4, 3, 2, 1, 0]], dtype=np.int32)
        _ORACLE_CASE = ("prefill", x, router, experts, np.array(fm, np.int32), forced, 6)
        return
    if workload.startswith("fp4") or workload.startswith("nvfp4"):
        fm = [synth.NVFP4 if workload.startswith("nv") else synth.MXFP4] * 7
    else:
        fm = [synth.TQ1, synth.TQ1, synth.TQ1, synth.Q2_0, synth.Q2_0, synth.Q3_K, synth.Q2_0]
    M = 6 if workload.endswith("m6") else 1
    if M > 1:
        # six independent rows touch up to 36 distinct routed experts; the
        # sample keeps 12 of them (two per rank), each row choosing 6
        fm = [fm[e % 6] for e in range(12)] + [synth.Q2_0]
    nexp = len(fm) - 1
    experts = [synth.random_expert(rng, int(f), H, I) for f in fm]
    router = synth.router_weights(rng, E, H)
    x = synth.x_bf16(rng, M, H)
    forced = np.stack([(np.arange(K) + 2 * m) % nexp for m in range(M)]).astype(np.int32)
    _ORACLE_CASE = ("decode", x, router, experts, np.array(fm, np.int32), forced, nexp)


def _oracle_worker_run(_):
    from oracle import moe as O
    kind, x, router, experts, fmts, forced, nexp = _ORACLE_CASE
    t0 = time.perf_counter()
    if kind == "prefill":
        O.prefill_rows(x, router, None, experts, fmts, H, I, K, nexp, forced, [0, 1])
    else:
        O.moe_layer(x, router, None, experts, fmts, H, I, K, nexp, forced_idx=forced)
    return time.perf_counter() - t0


def _oracle_bytes(workload: str) -> int:
    import synth
    if workload.startswith("fp4") or workload.startswith("nvfp4"):
        fm = [synth.NVFP4 if workload.startswith("nv") else synth.MXFP4] * 7
    else:
        fm = [synth.TQ1, synth.TQ1, synth.TQ1, synth.Q2_0, synth.Q2_0, synth.Q3_K, synth.Q2_0]
    if workload.endswith("m6"):
        fm = [fm[e % 6] for e in range(12)] + [synth.Q2_0]
    return sum(synth.expert_bytes(int(f), H, I) for f in fm)


def _oracle_sample_desc(workload: str) -> str:
    if workload == "prefill":
        return ("two prefill tokens of the mixed layer (router over 384 experts, 6 routed + shared expert FFN "
                "each), fp64")
    if workload.startswith("fp4") or workload.startswith("nvfp4"):
        return ("one %s layer call at M=1 (router 384 x 5120 fp32, 6 routed + 1 shared expert FFN), fp64"
                % ("NVFP4" if workload.startswith("nv") else "MXFP4"))
    if workload.endswith("m6"):
        return ("one mixed-format layer call at M=6 (router 384 x 5120 fp32, 6 routed experts per row among 12 "
                "distinct ternary/Q2_0/Q3_K ones + Q2_0 shared), fp64")
    return "one mixed-format layer call at M=1 (3 ternary, 2 Q2_0, 1 Q3_K routed + Q2_0 shared), fp64"


def oracle_workers() -> int:
    """Host cores to use, bounded so that every worker's fp64 expert copies
    (about 3 GB for a layer call) fit in the available memory."""
    n = os.cpu_count() or 1
    try:
        with open("/proc/meminfo") as fh:
            for line in fh:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
                    n = min(n, max(1, int(avail // 3.5e9)))
                    break
    except OSError:
        pass
    return n


class OraclePool:
    """P spawned workers, each holding one seeded layer-call sample."""

    def __init__(self, workload: str, n: int):
        import multiprocessing as mp
        self.n = n
        self.ctx = mp.get_context("spawn")
        self.pools = [self.ctx.Pool(1, initializer=_oracle_worker_init, initargs=(workload, i)) for i in range(n)]

    def step(self):
        """Every worker runs its call once; returns (wall seconds, per-call seconds)."""
        t0 = time.perf_counter()
        rs = [p.apply_async(_oracle_worker_run, (0,)) for p in self.pools]
        per = [r.get() for r in rs]
        return time.perf_counter() - t0, per

    def close(self):
        for p in self.pools:
            p.close()
        for p in self.pools:
            p.join()


def run_cpu_baseline(workload: str):
    """The oracle on all usable host cores: two rounds of one layer call per
    worker, after one untimed round (imports, first-touch of the weights)."""
    # single-threaded BLAS inside each worker: the cores are used by the workers
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    n = oracle_workers()
    pool = OraclePool(workload, n)
    try:
        pool.step()
        walls = [pool.step()[0] for _ in range(2)]
    finally:
        pool.close()
    T = sum(walls)
    sample = "%s; %d worker processes (one per core, 1 BLAS thread each) x %d rounds, %.1f s" % (
        _oracle_sample_desc(workload), n, len(walls), T)
    if workload == "prefill":
        return {"value": round(n * len(walls) * 2 / T, 4), "unit": "tokens/s", "cores": n, "kind": "oracle",
                "sample": sample}
    return {"value": round(n * len(walls) * _oracle_bytes(workload) / T / 1e9, 5), "unit": "GB/s", "cores": n,
            "kind": "oracle", "sample": sample}


# ----------------------------------------------------------- GPU workloads
class LayerCase:
    """One decode workload resident on the device: layer instances, a bank of
    inputs, a workspace and one CUDA graph per instance (events as graph
    nodes around the layer call)."""

    def __init__(self, A, dev, W, M, xs, name):
        import torch
        self.A, self.dev, self.W, self.M, self.name = A, dev, W, M, name
        self.xs = xs                      # (n_x, M, H) int16 (bf16 bits)
        self.n_x, self.NL = xs.shape[0], W.n_inst
        self.nb = A.bqe_workspace_bytes(W.d, M)
        self.ws = torch.empty(self.nb, dtype=torch.uint8, device=dev)
        A.bqe_workspace_init(self.ws, self.nb)
        self.pool = W.pool.cstruct()
        self.out = torch.zeros(M, H, device=dev)
        self.idx = torch.zeros(M, K, dtype=torch.int32, device=dev)
        self.xbuf = torch.empty_like(xs[0])
        self.ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        self.times, self.bytes = [], []
        self.launches = 0

    def call(self, inst, ev=None, x=None, idx=None):
        if ev:
            ev[0].record()
        W = self.W
        self.A.bqe_moe_layer_forward(W.d, self.M, self.xbuf if x is None else x, W.wr[inst],
                                     None if W.bias is None else W.bias[inst], self.pool, W.tables[inst], None,
                                     self.out, 0, self.idx if idx is None else idx, None, self.ws, self.nb)
        if ev:
            ev[1].record()

    def prepare(self, warm):
        import torch
        for i in range(warm):
            self.xbuf.copy_(self.xs[i % self.n_x])
            self.call(i % self.NL)
        torch.cuda.synchronize()
        self.check()
        st = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(st)
        with torch.cuda.stream(side):
            self.call(0)
        st.wait_stream(side)
        torch.cuda.synchronize()
        self.graphs = []
        for inst in range(self.NL):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.call(inst, self.ev)
            self.graphs.append(g)
        torch.cuda.synchronize()
        self.step_no = 0

    def check(self):
        rc, det = self.A.bqe_check(self.ws)
        assert rc == 0, (self.name, self.A.status_name(rc), det)

    def soak(self, i):
        self.xbuf.copy_(self.xs[i % self.n_x])
        self.graphs[i % self.NL].replay()

    def run(self, n):
        """n timed steps; per step the layer time (graph events) and the expert
        bytes of the distinct experts its routing chose."""
        for _ in range(n):
            s = self.step_no
            inst = s % self.NL
            self.xbuf.copy_(self.xs[s % self.n_x])
            self.graphs[inst].replay()
            self.ev[1].synchronize()
            self.times.append(self.ev[0].elapsed_time(self.ev[1]) * 1e-3)
            idx = self.idx.cpu().numpy()
            us = set(int(e) for e in idx.reshape(-1)) | {self.W.E}
            self.bytes.append(sum(self.W.expert_bytes(inst, e) for e in us))
            self.launches += 1
            self.step_no += 1


class Step40Case:
    """40 chained decode layers (bqe_moe_step) captured in one CUDA graph."""

    def __init__(self, A, dev, M, name):
        import torch
        from synth import workloads as WL
        self.A, self.dev, self.M, self.name = A, dev, M, name
        self.S = S = WL.Step40(dev, m=M)
        self.nb = A.bqe_workspace_bytes(S.d, M)
        self.ws = torch.empty(self.nb, dtype=torch.uint8, device=dev)
        A.bqe_workspace_init(self.ws, self.nb)
        self.pool = S.pool.cstruct()
        self.resid = torch.zeros(M, H, device=dev)
        self.forced = torch.zeros(S.n_layers, M, K, dtype=torch.int32, device=dev)
        self.nf = S.forced.shape[0]
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        self.times, self.bytes = [], []
        self.launches = 0

    def load(self, i):
        self.forced.copy_(self.S.forced[i % self.nf])
        self.resid.copy_(self.S.x0[i % self.nf])

    def call(self):
        S = self.S
        self.A.bqe_moe_step(S.d, S.n_layers, self.M, self.resid, S.wr, None, self.pool, S.tables, self.forced, None,
                            self.ws, self.nb)

    def prepare(self, warm):
        import torch
        for i in range(max(warm, 1)):
            self.load(i)
            self.call()
        torch.cuda.synchronize()
        self.check()
        st = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(st)
        with torch.cuda.stream(side):
            self.call()
        st.wait_stream(side)
        torch.cuda.synchronize()
        self.g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g):
            self.call()
        torch.cuda.synchronize()
        self.step_no = 0

    def check(self):
        rc, det = self.A.bqe_check(self.ws)
        assert rc == 0, (self.name, self.A.status_name(rc), det)

    def soak(self, i):
        self.load(i)
        self.g.replay()

    def run(self, n):
        import torch
        st = torch.cuda.current_stream()
        L = self.S.n_layers
        for _ in range(n):
            s = self.step_no
            self.load(s)
            self.ev[0].record(st)
            self.g.replay()
            self.ev[1].record(st)
            self.ev[1].synchronize()
            self.times.append(self.ev[0].elapsed_time(self.ev[1]) * 1e-3 / L)  # per layer
            self.bytes.append(sum(self.S.layer_bytes(l, s % self.nf) for l in range(L)) / L)
            self.launches += L
            self.step_no += 1


def make_case(A, dev, workload, args, banks):
    """The device workload of `workload`; `banks` shares layer sets between
    the M = 1 and M = 6 mixed records (M = 1 takes each bank entry's first row)."""
    from synth import workloads as WL
    M = 6 if workload.endswith("m6") else 1
    if workload.startswith("step40"):
        return Step40Case(A, dev, M, workload)
    kind = "fp4" if workload.startswith("fp4") else "nvfp4" if workload.startswith("nvfp4") else "mixed"
    if kind not in banks:
        m = 6 if kind == "mixed" else 1
        banks[kind] = WL.LayerSet(dev, kind, args.instances, seed={"fp4": 1, "mixed": 2, "nvfp4": 3}[kind], m=m,
                                  n_x=64, n_experts=args.experts)
    W = banks[kind]
    xs = W.xs if W.m == M else W.xs[:, :M].contiguous()
    return LayerCase(A, dev, W, M, xs, workload)


def summary(case, hbm):
    """us/layer as median and p10/p90 over the steps, expert-byte GB/s over
    their sum, and the fraction of HBM."""
    T, B = sum(case.times), sum(case.bytes)
    gbs = B / T / 1e9
    us = [t * 1e6 for t in case.times]
    return dict(workload=WORKLOADS[case.name], M=case.M, steps=len(us),
                us_per_layer_median=round(pct(us, 50), 3), us_per_layer_p10=round(pct(us, 10), 3),
                us_per_layer_p90=round(pct(us, 90), 3), us_per_layer_mean=round(sum(us) / len(us), 3),
                expert_gbs=round(gbs, 2), frac_of_hbm=round(gbs / hbm, 4),
                expert_bytes_per_layer=round(B / len(us)), tokens_per_s=round(case.M * len(us) / T, 1))


def soak(cases, seconds):
    """Untimed load before timing, so the clock samples see the GPU busy."""
    import torch
    t_end = time.time() + seconds
    i = 0
    while time.time() < t_end:
        for c in cases:
            c.soak(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def diag_timeline(A, case):
    """Per-CTA timeline of one eager decode call (globaltimer stamps), to stderr."""
    import numpy as np
    import torch
    W, M = case.W, case.M
    off = A.bqe_diag_offset(W.d, M)
    dbg = case.ws[off:off + 8 * 3 * 1024 * 8].view(torch.int64).view(3, 1024, 8)
    rows = []
    for s_ in range(10):
        dbg.zero_()
        for k in (0, 2, 3, 5):
            dbg[k >> 3, 1023, k & 7] = 2 ** 62
        case.xbuf.copy_(case.xs[s_ % case.n_x])
        A.bqe_set_diag(True)
        try:
            case.call(s_ % case.NL)
        finally:
            A.bqe_set_diag(False)
        torch.cuda.synchronize()
        d = dbg.cpu().numpy().astype(np.float64)
        t0 = d[0, 1023, 0]
        rows.append([(d[k >> 3, 1023, k & 7] - t0) / 1e3 for k in (1, 2, 10, 3, 4, 9, 6)])
    case.check()
    names = ["logits_published_max", "routing_known_min", "routing_known_max", "first_item_landed",
             "last_w13_item_done", "last_compute_done", "end"]
    tl = np.array(rows).mean(axis=0)
    sys.stderr.write("DECODE_TIMELINE_us(from first CTA start) %s %s\n" % (case.name, json.dumps(
        {n: round(float(v), 2) for n, v in zip(names, tl)})))


def run_decode(args, rank, world):
    import torch
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    from bit_quantised_expert_gb300 import _abi as A

    dev = torch.device("cuda", torch.cuda.current_device())
    head_name = args.workload or "fp4-m1"
    subs = [] if args.workload else list(SUB_RECORDS)
    banks = {}
    head = make_case(A, dev, head_name, args, banks)
    subcases = [make_case(A, dev, w, args, banks) for w in subs]
    warm = max(args.warmup, 3)
    for c in [head] + subcases:
        c.prepare(warm)
    hbm, hbm_kind = peaks()

    clocks = ClockSampler(torch.cuda.current_device(), enabled=not args.no_clocks)
    soak([head] + subcases, args.soak_s)
    # headline: exactly K timed steps, bracketed by barrier + synchronize
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    head.run(args.steps)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    # sub-records: interleaved rounds, each workload a block of steps per round
    R = max(1, args.rounds)
    per = [args.sub_steps // R + (1 if r < args.sub_steps % R else 0) for r in range(R)]
    for r in range(R):
        for c in subcases:
            torch.cuda.synchronize()
            c.run(per[r])
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    for c in [head] + subcases:
        c.check()

    T_max = reduce_max(sum(head.times), world)
    total_bytes = reduce_sum(float(sum(head.bytes)), world)
    value = total_bytes / T_max / 1e9
    steps = args.steps
    M = head.M
    mean = lambda v: sum(v) / len(v)  # noqa: E731
    l2mb = torch.cuda.get_device_properties(0).L2_cache_size / 2 ** 20
    if isinstance(head, LayerCase):
        router_bytes = head.W.E * H * 4
        cfg = dict(workload=WORKLOADS[head_name], hidden=H, inter=I, n_experts=head.W.E, top_k=K, n_shared=1, M=M,
                   l2="inputs larger than L2: steps rotate over %d layer instances and 64 inputs (%.0f MB of "
                      "weights streamed between reuses vs %.0f MB L2)" % (
                          head.NL, (head.NL - 1) * mean(head.bytes) / 1e6, l2mb),
                   parallelism="replicas" if world > 1 else "single-gpu")
        kind = ("mxfp4" if head_name.startswith("fp4") else "nvfp4" if head_name.startswith("nvfp4")
                else "ternary/q2_0/q3_k")
    else:
        router_bytes = E * H * 4
        cfg = dict(workload=WORKLOADS[head_name], layers=head.S.n_layers, slots=4288, M=M,
                   l2="inputs larger than L2: each step streams ~3 GB",
                   routing="Zipf(1.0) forced selection, weights from the router",
                   parallelism="replicas" if world > 1 else "single-gpu")
        kind = "ternary/q2_0/q3_k"
    # roofline of the one kernel of the layer: all bytes it must read (the
    # distinct experts and the fp32 router) over its CUDA-event duration
    alg = mean(head.bytes) + router_bytes
    achieved = alg / mean(head.times) / 1e9
    traffic = None
    if (head_name == "fp4-m1" and args.experts == E and TRAFFIC_FP4_M1["bytes"]
            and TRAFFIC_FP4_M1["sha256"] == kernel_digest()):
        traffic = TRAFFIC_FP4_M1["bytes"]
    us = [t * 1e6 for t in head.times]
    res = dict(
        metric=METRIC, value=round(value, 2), unit="GB/s", n_gpus=world, steps=steps, warmup=args.warmup,
        ms_per_step=round(T_max / steps * 1e3, 5), higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="fp32-accumulate over %s weights, bf16 activations" % kind,
        data="synthetic (seeded, generated on the device)", config=cfg,
        us_per_layer=round(T_max / steps * 1e6 / (head.S.n_layers if not isinstance(head, LayerCase) else 1), 3),
        us_per_layer_median=round(pct(us, 50), 3), us_per_layer_p10=round(pct(us, 10), 3),
        us_per_layer_p90=round(pct(us, 90), 3),
        tokens_per_s=round(M * steps * world / T_max, 1),
        frac_of_hbm=round(value / hbm, 4), hbm_peak_gbs=hbm, hbm_peak_kind=hbm_kind,
        expert_bytes_per_step=round(mean(head.bytes)),
        roofline=dict(bound="hbm", achieved=round(achieved, 1), peak=hbm, unit="GB/s",
                      frac=round(achieved / hbm, 4), traffic=traffic,
                      kernel="k_moe (the whole decode layer: router, top-k, W1/W3, SiLU-GLU, W2, combine)",
                      algorithmic_bytes_per_launch=round(alg),
                      peak_kind="%s hbm_gbs (burst copy; the kernel is timed alone)" % hbm_kind),
        gpu_launches=head.launches,
        timing="CUDA-graph replay per step, CUDA events around the layer kernel on its stream",
        wall_s_timed_loop=round(wall, 4),
    )
    if not isinstance(head, LayerCase):
        res["ms_per_step"] = round(T_max / steps * head.S.n_layers * 1e3, 4)
        res["cuda_graph"] = True
    if subcases:
        res["sub_records"] = {c.name.replace("-", "_"): summary(c, hbm) for c in subcases}
        res["sub_records_timing"] = ("%d interleaved rounds after the headline steps, CUDA-graph replay, "
                                     "events around each layer (step40: around the 40-layer graph, per layer)" % R)
        res["sub_records_gpu_launches"] = sum(c.launches for c in subcases)
        sr = res["sub_records"]
        if "mixed_m1" in sr and "mixed_m6" in sr:
            # a verify pass of 5 drafts is one M = 6 call per layer: it pays when
            # it emits more tokens than t(M = 6) / t(M = 1); the field report
            # (section 3B) logs 3.39 tokens per pass
            t1, t6 = sr["mixed_m1"]["us_per_layer_median"], sr["mixed_m6"]["us_per_layer_median"]
            res["verify_m6"] = dict(break_even_tokens_per_pass=round(t6 / t1, 3),
                                    speedup_at_3_39_tokens_per_pass=round(3.39 * t1 / t6, 3),
                                    note="derived from the mixed_m1 / mixed_m6 sub-records")
    if clk:
        res["clocks"] = clk
    if args.diag and isinstance(head, LayerCase):
        diag_timeline(A, head)
        for c in subcases:
            if isinstance(c, LayerCase):
                diag_timeline(A, c)

    # ---- end to end through the public call with host buffers --------------
    if isinstance(head, LayerCase):
        res["e2e"] = e2e_layer(A, dev, head, steps, world)
    return res


def e2e_layer(A, dev, case, steps, world):
    """Eager calls of bqe_moe_layer_forward: every step copies its input from
    pinned host memory and reads the output back into pinned host memory,
    inside the timed region."""
    import torch
    M = case.M
    st = torch.cuda.current_stream()
    xh = torch.empty(M, H, dtype=torch.int16).pin_memory()
    oh = torch.empty(M, H, dtype=torch.float32).pin_memory()
    xd = torch.empty(M, H, dtype=torch.int16, device=dev)
    xs_host = [x.cpu() for x in case.xs]
    idx_log = torch.zeros(steps, M, K, dtype=torch.int32, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for s_ in range(3):
        xd.copy_(xs_host[s_ % case.n_x].to(dev))
        case.call(s_ % case.NL, x=xd)
    torch.cuda.synchronize()
    for s_ in range(steps):
        xh.copy_(xs_host[s_ % case.n_x])
        ev[s_][0].record(st)
        xd.copy_(xh, non_blocking=True)
        case.call(s_ % case.NL, x=xd, idx=idx_log[s_])
        oh.copy_(case.out, non_blocking=True)
        ev[s_][1].record(st)
    torch.cuda.synchronize()
    case.check()
    Te = sum(ev[s_][0].elapsed_time(ev[s_][1]) * 1e-3 for s_ in range(steps))
    idx_np = idx_log.cpu().numpy()
    be = sum(sum(case.W.expert_bytes(s_ % case.NL, e) for e in (set(int(v) for v in idx_np[s_].reshape(-1)) |
                                                                 {case.W.E})) for s_ in range(steps))
    Te_max = reduce_max(Te, world)
    return dict(value=round(reduce_sum(float(be), world) / Te_max / 1e9, 2), unit="GB/s",
                h2d_bytes_per_step=M * H * 2, d2h_bytes_per_step=M * H * 4,
                us_per_layer=round(Te_max / steps * 1e6, 3),
                note="eager calls through bqe_moe_layer_forward, pinned host x in, host out back")


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
    """The oracle (fp64, as it stands) on the host cores: each step, every
    worker process runs one full call of the headline layer on its own seeded
    inputs (rank 0 only)."""
    if rank != 0:
        return None
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    workload = args.workload or "fp4-m1"
    if workload.startswith("step40"):
        workload = "mixed-m1"  # one layer of the step: the sample unit of the per-layer metric
    n = oracle_workers()
    pool = OraclePool(workload, n)
    try:
        for _ in range(args.warmup):
            pool.step()
        walls = [pool.step()[0] for _ in range(args.steps)]
    finally:
        pool.close()
    T = sum(walls)
    sample = "%s; %d worker processes (one per core, 1 BLAS thread each) per step" % (
        _oracle_sample_desc(workload), n)
    if workload == "prefill":
        value = n * 2 * args.steps / T
        return dict(metric=PREFILL_METRIC, value=round(value, 4), unit="tokens/s", n_gpus=world,
                    steps=args.steps, warmup=args.warmup, ms_per_step=round(T / args.steps * 1e3, 3),
                    higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic (seeded)",
                    impl="reference", config=dict(workload=WORKLOADS[workload], hidden=H, inter=I, n_experts=E,
                                                  top_k=K, n_shared=1, T=2),
                    cpu_baseline=dict(value=round(value, 4), unit="tokens/s", cores=n, kind="oracle", sample=sample),
                    e2e=dict(value=round(value, 4), unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    value = n * _oracle_bytes(workload) * args.steps / T / 1e9
    return dict(metric=METRIC, value=round(value, 5), unit="GB/s", n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(T / args.steps * 1e3, 3), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic (seeded)", impl="reference",
                config=dict(workload=WORKLOADS[workload], hidden=H, inter=I, n_experts=E, top_k=K, n_shared=1,
                            M=6 if workload.endswith("m6") else 1),
                cpu_baseline=dict(value=round(value, 5), unit="GB/s", cores=n, kind="oracle", sample=sample),
                e2e=dict(value=round(value, 5), unit="GB/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    rank, world, local = dist_setup(args.gpus)
    if args.workload == "prefill":
        res = run_prefill(args, rank, world)
    else:
        res = run_decode(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = run_cpu_baseline("prefill" if args.workload == "prefill" else (args.workload or "fp4-m1"))
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

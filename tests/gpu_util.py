"""Shared set-up for the GPU tests: device layers built from seeded synthetic
inputs, calls through the C ABI, and comparisons with the fp64 oracle."""
from __future__ import annotations

import numpy as np

import synth
from oracle import formats as F
from oracle import moe as O

REL_L2 = 1e-4       # fp32 decode outputs: relative L2 error bound
MAX_ABS = 1e-3      # ... and max-abs error bound, relative to max |reference|
TIE = 1e-6          # selections whose k-th and (k+1)-th keys are closer are ties


def torch_dev():
    import torch
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


class DeviceLayer:
    """One layer's router, bias, slot pool and slot table on the device."""

    def __init__(self, L, dev, fmts=None, canon_on_device=None):
        import torch
        from bit_quantised_expert_gb300 import _abi as A
        from bit_quantised_expert_gb300.pool import SlotPool
        self.A, self.L, self.dev = A, L, dev
        H, I, E, K = L["hidden"], L["inter"], L["n_experts"], L["top_k"]
        self.H, self.I, self.E, self.K = H, I, E, K
        self.d = A.desc(H, I, E, K)
        fm = L["fmts"] if fmts is None else fmts
        self.pool = SlotPool(self.d, fm, dev)
        for s in range(E + 1):
            self.pool.upload(s, L["experts"][s] if canon_on_device is None else canon_on_device(s))
        self.table = torch.arange(E + 1, dtype=torch.int32, device=dev)
        self.wr = torch.from_numpy(L["router"]).to(dev)
        self.bias = torch.from_numpy(L["bias"]).to(dev) if L.get("bias") is not None else None
        self.ws_M = None

    def workspace(self, M):
        import torch
        A = self.A
        if self.ws_M != M:
            self.ws_bytes = A.bqe_workspace_bytes(self.d, M)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.dev)
            A.bqe_workspace_init(self.ws, self.ws_bytes)
            self.ws_M = M
        return self.ws, self.ws_bytes

    def route(self, x_bits, use_bias=True):
        """The routing-only entry point: (idx, w)."""
        import torch
        A = self.A
        M = x_bits.shape[0]
        ws, nb = self.workspace(M)
        x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(self.dev)
        idx = torch.zeros(M, self.K, dtype=torch.int32, device=self.dev)
        w = torch.zeros(M, self.K, dtype=torch.float32, device=self.dev)
        A.bqe_route(self.d, M, x, self.wr, self.bias if use_bias else None, self.pool.cstruct(), self.table, None,
                    idx, w, ws, nb)
        rc, det = A.bqe_check(ws)
        assert rc == A.BQE_OK, (A.status_name(rc), det)
        return idx.cpu().numpy(), w.cpu().numpy()

    def forward(self, x_bits, forced=None, use_bias=True, accumulate_into=None):
        import torch
        A = self.A
        M = x_bits.shape[0]
        ws, nb = self.workspace(M)
        x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(self.dev)
        out = accumulate_into if accumulate_into is not None else torch.zeros(M, self.H, device=self.dev)
        idx = torch.zeros(M, self.K, dtype=torch.int32, device=self.dev)
        w = torch.zeros(M, self.K, dtype=torch.float32, device=self.dev)
        fi = None if forced is None else torch.from_numpy(np.ascontiguousarray(forced, dtype=np.int32)).to(self.dev)
        b = self.bias if use_bias else None
        A.bqe_moe_layer_forward(self.d, M, x, self.wr, b, self.pool.cstruct(), self.table, fi, out,
                                accumulate_into is not None, idx, w, ws, nb)
        rc, det = A.bqe_check(ws)
        assert rc == A.BQE_OK, (A.status_name(rc), det)
        return out.double().cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check_routing(ref, got_idx, got_w, forced=None):
    """Indices exact except rows whose selection is a near-tie; weights close."""
    M = got_idx.shape[0]
    checked = 0
    for m in range(M):
        if forced is None and ref["gap"][m] < TIE:
            continue
        assert got_idx[m].tolist() == ref["idx"][m].tolist(), (m, got_idx[m], ref["idx"][m])
        checked += 1
    return checked


def check_out(got, ref, rel=REL_L2, mabs=MAX_ABS, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(got - ref))
    lim = mabs * np.max(np.abs(ref))
    assert err <= rel, "%s rel-L2 %.3e > %.1e" % (what, err, rel)
    assert mx <= lim, "%s max-abs %.3e > %.3e" % (what, mx, lim)
    return err, mx / max(np.max(np.abs(ref)), 1e-300)


def oracle_layer_sampled(L_fmts, get_canon, x_bits, router, bias, idx, H, I, E, K, cols, shared=None):
    """Oracle outputs out[m, n] for n in `cols` (None: every column) with the
    selection idx (M, K): full fp64 W1/W3 of every used expert and the
    requested rows of W2."""
    if cols is None:
        cols = np.arange(H)
    shared = E if shared is None else shared
    x = O.bf16_bits_to_f64(x_bits).reshape(-1, H)
    r = O.route(x, router, bias, K, idx)
    M = x.shape[0]
    used = sorted(set(int(e) for e in np.asarray(idx).reshape(-1)) | {shared})
    out = np.zeros((M, len(cols)))
    for e in used:
        fmt = int(L_fmts[e])
        p1, p3, p2 = F.split_expert(fmt, get_canon(e), H, I)
        w1 = F.dequant_matrix(fmt, p1, I, H)
        w3 = F.dequant_matrix(fmt, p3, I, H)
        bw, bb = F.BLOCK[fmt]
        rowb = (I // bw) * bb
        if len(cols) == H and np.array_equal(cols, np.arange(H)):
            w2 = F.dequant_matrix(fmt, p2, H, I)
        else:
            w2 = np.stack([F.dequant_matrix(fmt, p2[n * rowb:(n + 1) * rowb], 1, I)[0] for n in cols])
        rows = [m for m in range(M) if e == shared or e in set(np.asarray(idx)[m].tolist())]
        h = O.silu(x[rows] @ w1.T) * (x[rows] @ w3.T)
        y = h @ w2.T
        for ri, m in enumerate(rows):
            if e == shared:
                out[m] += y[ri]
            else:
                js = np.where(np.asarray(idx)[m] == e)[0]
                out[m] += r["w"][m, js].sum() * y[ri]
    return out, r

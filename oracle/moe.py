"""Oracle for the MoE expert layer (fp64).  TEST INFRASTRUCTURE ONLY.

What the layer computes (DeepSeek-V4.1-Flash 4xL20 field report, sections 1
and 2: hidden 5120, moe_intermediate 2304, 384 routed experts + 1 shared,
6 experts per token; "single expert = 3 x 5120 x 2304 parameters"):

  z[m, e]   = sum_h x[m, h] Wr[e, h]                 router logits
  s         = sigmoid(z)                             scores
  key       = s + b                                  b only steers selection
  idx[m]    = the k experts of largest key (ties -> lower expert id)
  w[m, j]   = s[m, idx[m, j]] / sum_j' s[m, idx[m, j']]
  y_e(x)    = W2_e (silu(W1_e x) * (W3_e x)),  silu(t) = t / (1 + e^-t)
  out[m]    = sum_j w[m, j] y_idx[m,j](x[m]) + y_shared(x[m])

The selection-only bias follows the Strata 4090 post, section 5.3: the bias
changes which experts a token computes, while the mixing weights stay exact
(they are the unbiased scores).  The score function (sigmoid, normalised over
the selected experts) and the absence of a routed scaling factor are this
library's reading where the pages are silent.
"""
from __future__ import annotations

import numpy as np

from . import formats


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the top half of an IEEE binary32; widen exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), returning uint16
    bits.  Written out: first to binary32 (numpy cast, round to nearest even),
    then drop 16 fraction bits with round-to-nearest-even on the dropped half.
    (Double rounding through binary32 can differ from a direct fp64->bf16
    rounding only when the binary32 value is an exact tie; the oracle uses it
    only for reporting the chained step, never as a parity gate.)"""
    u = np.asarray(v, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> 16
    rest = u & 0xFFFF
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & 1) == 1))
    return (keep + up).astype(np.uint16)


def sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def silu(t: np.ndarray) -> np.ndarray:
    return t / (1.0 + np.exp(-t))


def route(x: np.ndarray, router_w: np.ndarray, sel_bias, top_k: int, forced_idx=None):
    """Router GEMV, scores, biased top-k and mixing weights for rows x (M, H) fp64.

    Returns dict: z (M, E), s (M, E), key (M, E), idx (M, k) int, w (M, k),
    gap (M,) = key of the k-th selected minus key of the best unselected expert
    (a small gap marks a near-tie whose selection may legitimately differ
    under another rounding of z), order (M, E) the full key order.
    With forced_idx (M, k) the selection is given and only w is computed from s.
    """
    x = np.asarray(x, dtype=np.float64)
    wr = np.asarray(router_w, dtype=np.float64)
    z = x @ wr.T
    s = sigmoid(z)
    b = np.zeros(wr.shape[0]) if sel_bias is None else np.asarray(sel_bias, dtype=np.float64)
    key = s + b[None, :]
    M, E = key.shape
    order = np.empty((M, E), dtype=np.int64)
    for m in range(M):
        # primary: key descending; secondary: expert id ascending
        order[m] = np.lexsort((np.arange(E), -key[m]))
    if forced_idx is None:
        idx = order[:, :top_k].copy()
    else:
        idx = np.asarray(forced_idx, dtype=np.int64).reshape(M, top_k)
    gap = np.array([key[m, order[m, top_k - 1]] - key[m, order[m, top_k]] if E > top_k else np.inf
                    for m in range(M)])
    ss = np.take_along_axis(s, idx, axis=1)
    w = ss / ss.sum(axis=1, keepdims=True)
    return dict(z=z, s=s, key=key, idx=idx, w=w, gap=gap, order=order)


def expert_ffn(x: np.ndarray, w1: np.ndarray, w3: np.ndarray, w2: np.ndarray):
    """y = W2 (silu(W1 x) * (W3 x)) for rows x (R, H); returns (y, h)."""
    g = x @ w1.T
    u = x @ w3.T
    h = silu(g) * u
    return h @ w2.T, h


class ExpertCache:
    """Dequantises canonical expert bytes on first use (fp64, exact)."""

    def __init__(self, experts, fmts, hidden: int, inter: int):
        self.experts, self.fmts, self.H, self.I = experts, fmts, hidden, inter
        self._c = {}

    def __call__(self, e: int):
        if e not in self._c:
            self._c[e] = formats.dequant_expert(int(self.fmts[e]), self.experts[e], self.H, self.I)
        return self._c[e]


def moe_layer(x_bits, router_w, sel_bias, experts, fmts, hidden, inter, top_k,
              shared: int, forced_idx=None, cache=None):
    """One MoE layer for bf16 rows x_bits (M, H).

    experts[e] / fmts[e]: canonical bytes and format of expert e; expert
    `shared` is the shared expert (weight 1, every row).  Returns dict with
    out (M, H) fp64 and the routing of route().
    """
    x = bf16_bits_to_f64(x_bits).reshape(-1, hidden)
    r = route(x, router_w, sel_bias, top_k, forced_idx)
    cache = cache or ExpertCache(experts, fmts, hidden, inter)
    M = x.shape[0]
    out = np.zeros((M, hidden))
    for m in range(M):
        w1, w3, w2 = cache(shared)
        out[m] += expert_ffn(x[m:m + 1], w1, w3, w2)[0][0]
        for j in range(top_k):
            w1, w3, w2 = cache(int(r["idx"][m, j]))
            out[m] += r["w"][m, j] * expert_ffn(x[m:m + 1], w1, w3, w2)[0][0]
    r["out"] = out
    return r


RMS_EPS = 1e-6


def rmsnorm_to_bf16(resid: np.ndarray) -> np.ndarray:
    """t = bf16(r / sqrt(mean(r^2) + eps)) per row, unit gain.  The pages chain
    40 MoE layers through a residual stream; the normalisation in front of each
    layer (pre-norm, unit gain, eps 1e-6) is this library's reading."""
    r = np.asarray(resid, dtype=np.float64)
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + RMS_EPS)
    return round_to_bf16(r / rms)


def moe_chain(x_bits, layers, hidden, inter, top_k, t_forced=None):
    """Residual chain r_0 = x, t_l = rmsnorm_to_bf16(r_l), r_{l+1} = r_l + MoE_l(t_l).

    layers[l]: dict(router, bias, experts, fmts, shared, forced_idx).
    With t_forced (L, M, H) bf16 bits the chain is teacher-forced: layer l
    consumes t_forced[l] instead of its own t_l, and out_l is returned per layer.
    """
    r = bf16_bits_to_f64(x_bits).reshape(-1, hidden).copy()
    outs, ts = [], []
    for l, L in enumerate(layers):
        t = rmsnorm_to_bf16(r) if t_forced is None else np.asarray(t_forced[l])
        ts.append(t)
        res = moe_layer(t, L["router"], L["bias"], L["experts"], L["fmts"], hidden, inter,
                        top_k, L["shared"], L.get("forced_idx"), L.get("cache"))
        outs.append(res["out"])
        r = r + res["out"]
    return dict(resid=r, outs=outs, ts=ts)


def prefill_permutation(idx: np.ndarray, n_experts: int):
    """Group the (token, slot) pairs of a routing idx (T, k) by expert, tokens
    ascending within an expert.  Returns (counts (E,), offsets (E+1,),
    pairs (T*k, 2) of (token, slot))."""
    T, k = idx.shape
    counts = np.bincount(idx.reshape(-1), minlength=n_experts)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    pairs = np.empty((T * k, 2), dtype=np.int64)
    fill = offsets[:-1].copy()
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            pairs[fill[e]] = (t, j)
            fill[e] += 1
    return counts, offsets, pairs


def prefill_rows(x_bits, router_w, sel_bias, experts, fmts, hidden, inter, top_k, shared,
                 forced_idx, rows, cache=None):
    """The prefill layer evaluated on a subset of token rows: the per-token
    result equals the decode layer's (prefill only regroups tokens by expert;
    the Strata 4090 post, section 5.3, requires prefill accelerations to leave
    results unchanged).  Routing is computed for every token; outputs for rows."""
    x = bf16_bits_to_f64(x_bits).reshape(-1, hidden)
    full = route(x, router_w, sel_bias, top_k, forced_idx)
    cache = cache or ExpertCache(experts, fmts, hidden, inter)
    out = np.zeros((len(rows), hidden))
    for i, m in enumerate(rows):
        w1, w3, w2 = cache(shared)
        out[i] += expert_ffn(x[m:m + 1], w1, w3, w2)[0][0]
        for j in range(top_k):
            w1, w3, w2 = cache(int(full["idx"][m, j]))
            out[i] += full["w"][m, j] * expert_ffn(x[m:m + 1], w1, w3, w2)[0][0]
    full["out_rows"] = out
    return full


def expert_bytes_streamed(idx: np.ndarray, fmts, hidden: int, inter: int, shared: int, slot_of=None):
    """Algorithmic expert bytes of one decode call: every distinct expert (or
    distinct slot, when experts alias slots) among the selected ones plus the
    shared expert is read exactly once.  Bytes per expert = 3 matrices of
    hidden x inter weights at the format's bytes per weight (field report,
    section 2: the decode cost is set by bytes per token)."""
    chosen = set(int(e) for e in np.asarray(idx).reshape(-1)) | {shared}
    keys = {slot_of[e] if slot_of is not None else e: e for e in chosen}
    total = 0
    for key, e in keys.items():
        bw, bb = formats.BLOCK[int(fmts[e])]
        total += 3 * hidden * inter // bw * bb
    return total

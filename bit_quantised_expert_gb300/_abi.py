"""ctypes binding of libbqe.so (include/bqe.h), same names as the C ABI.

Argument marshalling only: tensors become device pointers, host structs become
ctypes structures, status codes become exceptions.  Every computation runs in
the library's CUDA kernels; there is no fallback.  Importing this module when
the library has not been built raises immediately.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libbqe.so")

BQE_OK, BQE_EINVAL, BQE_ENOSPC, BQE_ECUDA, BQE_EDEVICE, BQE_ETIMEOUT, BQE_EUNSUPPORTED = range(7)
BQE_FMT_TQ1, BQE_FMT_Q2_0, BQE_FMT_Q3_K, BQE_FMT_MXFP4, BQE_FMT_NVFP4 = 1, 2, 3, 4, 5


class BqeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_name(status), status))


class bqe_layer_desc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32)]


class bqe_pool(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("base_bytes", ctypes.c_uint64), ("slot_off", ctypes.c_void_p),
                ("slot_fmt", ctypes.c_void_p), ("n_slots", ctypes.c_int32), ("fmt_mask", ctypes.c_int32)]


class bqe_stats(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("experts_streamed", ctypes.c_int32), ("per_format", ctypes.c_int32 * 6),
                ("row_uses", ctypes.c_int32), ("expert_bytes", ctypes.c_uint64), ("router_bytes", ctypes.c_uint64)]


class bqe_cache_stats(ctypes.Structure):
    _fields_ = [("requests", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("bytes_uploaded", ctypes.c_uint64)]


VERIFY_MAX_DRAFT = 15


class bqe_verify_stats(ctypes.Structure):
    _fields_ = [("passes", ctypes.c_uint64), ("tokens", ctypes.c_uint64),
                ("hist", ctypes.c_uint64 * (VERIFY_MAX_DRAFT + 1))]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libbqe.so is not built (%s); run bit_quantised_expert_gb300.buildlib.build() "
                          "or __graft_entry__.build() first" % LIB_PATH)
    return ctypes.CDLL(LIB_PATH)


lib = _load()

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_U64 = ctypes.c_uint64
_DESC = ctypes.POINTER(bqe_layer_desc)
_POOL = ctypes.POINTER(bqe_pool)

# (name, restype, argtypes) for every symbol of include/bqe.h
SIGNATURES = {
    "bqe_block_weights": (_I32, [_I32]),
    "bqe_block_bytes": (_I32, [_I32]),
    "bqe_packed_bytes": (_U64, [_I32, _I32, _I32]),
    "bqe_expert_bytes": (_U64, [_DESC, _I32]),
    "bqe_scale_bytes": (_I32, [_I32]),
    "bqe_pack": (ctypes.c_int, [_I32, _I32, _I32, _P, _P, _P]),
    "bqe_pool_pack_slot": (ctypes.c_int, [_DESC, _I32, _P, _P, _P]),
    "bqe_pool_bytes": (_U64, [_DESC, _I32, _P]),
    "bqe_pool_init": (ctypes.c_int, [_POOL, _DESC, _I32, _P, _P, _U64, _P]),
    "bqe_pool_upload": (ctypes.c_int, [_POOL, _DESC, _I32, _P, _P]),
    "bqe_unpack_host": (ctypes.c_int, [_I32, _I32, _I32, _P, _P, _P]),
    "bqe_layer_stats": (ctypes.c_int, [_DESC, _I32, _P, _P, ctypes.POINTER(bqe_stats)]),
    "bqe_dequant": (ctypes.c_int, [_I32, _I32, _I32, _P, _P, _P]),
    "bqe_workspace_bytes": (_U64, [_DESC, _I32]),
    "bqe_workspace_init": (ctypes.c_int, [_P, _U64, _P]),
    "bqe_moe_layer_forward": (ctypes.c_int, [_DESC, _I32, _P, _P, _P, _POOL, _P, _P, _P, _I32, _P, _P, _P, _U64, _P]),
    "bqe_route": (ctypes.c_int, [_DESC, _I32, _P, _P, _P, _POOL, _P, _P, _P, _P, _P, _U64, _P]),
    "bqe_moe_layer_forward_noalloc": (ctypes.c_int, [_DESC, _I32, _P, _P, _P, _POOL, _P, _P, _P, _I32, _P, _P, _P,
                                                     _P]),
    "bqe_prefill_workspace_bytes": (_U64, [_DESC, _I32]),
    "bqe_moe_prefill": (ctypes.c_int, [_DESC, _I32, _P, _P, _P, _POOL, _P, _P, _P, _I32, _P, _P, _P, _U64, _P]),
    "bqe_moe_step": (ctypes.c_int, [_DESC, _I32, _I32, _P, _P, _P, _POOL, _P, _P, _P, _P, _U64, _P]),
    "bqe_check": (ctypes.c_int, [_P, _P, ctypes.POINTER(_I32)]),
    "bqe_check_noalloc": (ctypes.c_int, [_P, ctypes.POINTER(_I32)]),
    "bqe_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "bqe_set_wait_limit_ns": (None, [_U64]),
    "bqe_set_test_drop_item": (None, [_I32]),
    "bqe_set_prefill_f16": (None, [_I32]),
    "bqe_prefill_kernel_ms": (ctypes.c_int, [_P]),
    "bqe_prefill_diag_offset": (_U64, [_DESC, _I32]),
    "bqe_set_diag": (None, [_I32]),
    "bqe_diag_offset": (_U64, [_DESC, _I32]),
    "bqe_assign_formats": (ctypes.c_int, [_I32, _I32, _P, _P, _P, _P, _I32, ctypes.c_double, _P, _U64, _P, _P, _P,
                                          _P]),
    "bqe_cache_create": (ctypes.c_int, [_DESC, _I32, _P, _POOL, _P, _I32, _I32, _P, ctypes.POINTER(_P)]),
    "bqe_cache_destroy": (None, [_P]),
    "bqe_cache_plan": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _P]),
    "bqe_cache_fetch": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _U64, _P, _P, _P, _P]),
    "bqe_cache_done": (ctypes.c_int, [_P, ctypes.c_int64, _P]),
    "bqe_cache_ready": (ctypes.c_int, [_P, ctypes.c_int64, _P]),
    "bqe_verify_pass": (ctypes.c_int, [_I32, _P, _P, _P, ctypes.POINTER(_I32), _P, ctypes.POINTER(bqe_verify_stats)]),
    "bqe_cache_stats_get": (ctypes.c_int, [_P, ctypes.POINTER(bqe_cache_stats)]),
}

for _name, (_res, _args) in SIGNATURES.items():
    if hasattr(lib, _name):
        _f = getattr(lib, _name)
        _f.restype = _res
        _f.argtypes = _args


def status_name(s: int) -> str:
    return lib.bqe_status_str(int(s)).decode()


def ptr(t) -> int | None:
    """Device (or host) address of a tensor / array / raw int; None -> NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError("cannot take the address of %r" % type(t))


def stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ok(rc: int, what: str):
    if rc != BQE_OK:
        raise BqeError(rc, what)


def desc(hidden, inter, n_experts, top_k, n_shared=1) -> bqe_layer_desc:
    return bqe_layer_desc(hidden, inter, n_experts, top_k, n_shared)


# --------------------------------------------------------------- formats
def bqe_block_weights(fmt: int) -> int:
    return lib.bqe_block_weights(fmt)


def bqe_block_bytes(fmt: int) -> int:
    return lib.bqe_block_bytes(fmt)


def bqe_packed_bytes(fmt: int, rows: int, cols: int) -> int:
    return lib.bqe_packed_bytes(fmt, rows, cols)


def bqe_expert_bytes(d: bqe_layer_desc, fmt: int) -> int:
    return lib.bqe_expert_bytes(ctypes.byref(d), fmt)


def bqe_scale_bytes(fmt: int) -> int:
    return lib.bqe_scale_bytes(fmt)


def bqe_pack(fmt: int, rows: int, cols: int, codes, scales, out) -> None:
    """Host packing: codes/scales/out are C-contiguous uint8 numpy arrays."""
    _ok(lib.bqe_pack(fmt, rows, cols, ptr(codes), ptr(scales), ptr(out)), "bqe_pack")


# ------------------------------------------------------------------ pool
def bqe_pool_pack_slot(d, fmt, canon_src, slot_dst, stream=None) -> None:
    _ok(lib.bqe_pool_pack_slot(ctypes.byref(d), fmt, ptr(canon_src), ptr(slot_dst), stream_ptr(stream)),
        "bqe_pool_pack_slot")


def bqe_pool_bytes(d, slot_fmts) -> int:
    import numpy as np
    f = np.ascontiguousarray(slot_fmts, dtype=np.int32)
    return lib.bqe_pool_bytes(ctypes.byref(d), int(f.size), f.ctypes.data)


def bqe_pool_init(d, slot_fmts, dev_mem, dev_bytes, stream=None) -> bqe_pool:
    import numpy as np
    f = np.ascontiguousarray(slot_fmts, dtype=np.int32)
    p = bqe_pool()
    _ok(lib.bqe_pool_init(ctypes.byref(p), ctypes.byref(d), int(f.size), f.ctypes.data, ptr(dev_mem), int(dev_bytes),
                          stream_ptr(stream)), "bqe_pool_init")
    return p


def bqe_pool_upload(pool: bqe_pool, d, slot: int, canon_dev, stream=None) -> None:
    _ok(lib.bqe_pool_upload(ctypes.byref(pool), ctypes.byref(d), int(slot), ptr(canon_dev), stream_ptr(stream)),
        "bqe_pool_upload")


def bqe_unpack_host(fmt: int, rows: int, cols: int, packed, codes, scales) -> None:
    """Host unpacking (inverse of bqe_pack): C-contiguous uint8 numpy arrays."""
    _ok(lib.bqe_unpack_host(fmt, rows, cols, ptr(packed), ptr(codes), ptr(scales)), "bqe_unpack_host")


def bqe_layer_stats(d, M: int, ws, stream=None) -> dict:
    st = bqe_stats()
    _ok(lib.bqe_layer_stats(ctypes.byref(d), M, ptr(ws), stream_ptr(stream), ctypes.byref(st)), "bqe_layer_stats")
    return dict(rows=st.rows, experts_streamed=st.experts_streamed, per_format=list(st.per_format),
                row_uses=st.row_uses, expert_bytes=st.expert_bytes, router_bytes=st.router_bytes)


def bqe_dequant(fmt, rows, cols, src, out, stream=None) -> None:
    _ok(lib.bqe_dequant(fmt, rows, cols, ptr(src), ptr(out), stream_ptr(stream)), "bqe_dequant")


# ---------------------------------------------------------------- decode
def bqe_workspace_bytes(d, M: int) -> int:
    return lib.bqe_workspace_bytes(ctypes.byref(d), M)


def bqe_workspace_init(ws, nbytes: int, stream=None) -> None:
    _ok(lib.bqe_workspace_init(ptr(ws), nbytes, stream_ptr(stream)), "bqe_workspace_init")


def bqe_moe_layer_forward(d, M, x, router_w, sel_bias, pool: bqe_pool, slot_table, forced_idx, out,
                          accumulate, topk_idx, topk_w, ws, ws_bytes, stream=None) -> None:
    _ok(lib.bqe_moe_layer_forward(ctypes.byref(d), M, ptr(x), ptr(router_w), ptr(sel_bias), ctypes.byref(pool),
                                  ptr(slot_table), ptr(forced_idx), ptr(out), int(accumulate), ptr(topk_idx),
                                  ptr(topk_w), ptr(ws), ws_bytes, stream_ptr(stream)), "bqe_moe_layer_forward")


def bqe_moe_layer_forward_noalloc(d, M, x, router_w, sel_bias, pool: bqe_pool, slot_table, forced_idx, out,
                                  accumulate, topk_idx, topk_w, status_out, stream=None) -> None:
    """The layer with the library's fixed scratch array as workspace (no allocation)."""
    _ok(lib.bqe_moe_layer_forward_noalloc(ctypes.byref(d), M, ptr(x), ptr(router_w), ptr(sel_bias),
                                          ctypes.byref(pool), ptr(slot_table), ptr(forced_idx), ptr(out),
                                          int(accumulate), ptr(topk_idx), ptr(topk_w), ptr(status_out),
                                          stream_ptr(stream)), "bqe_moe_layer_forward_noalloc")


# ---------------------------------------------------------------- prefill
def bqe_prefill_workspace_bytes(d, T: int) -> int:
    return lib.bqe_prefill_workspace_bytes(ctypes.byref(d), T)


def bqe_moe_prefill(d, T, x, router_w, sel_bias, pool: bqe_pool, slot_table, forced_idx, out, accumulate,
                    topk_idx, topk_w, ws, ws_bytes, stream=None) -> None:
    _ok(lib.bqe_moe_prefill(ctypes.byref(d), T, ptr(x), ptr(router_w), ptr(sel_bias), ctypes.byref(pool),
                            ptr(slot_table), ptr(forced_idx), ptr(out), int(accumulate), ptr(topk_idx),
                            ptr(topk_w), ptr(ws), ws_bytes, stream_ptr(stream)), "bqe_moe_prefill")


def bqe_route(d, M, x, router_w, sel_bias, pool, slot_table, forced_idx, topk_idx, topk_w, ws, ws_bytes,
              stream=None) -> None:
    _ok(lib.bqe_route(ctypes.byref(d), M, ptr(x), ptr(router_w), ptr(sel_bias), ctypes.byref(pool),
                      ptr(slot_table), ptr(forced_idx), ptr(topk_idx), ptr(topk_w), ptr(ws), ws_bytes,
                      stream_ptr(stream)), "bqe_route")


def bqe_moe_step(d, n_layers, M, resid, router_w, sel_bias, pool, slot_tables, forced_idx, t_out, ws, ws_bytes,
                 stream=None) -> None:
    _ok(lib.bqe_moe_step(ctypes.byref(d), n_layers, M, ptr(resid), ptr(router_w), ptr(sel_bias), ctypes.byref(pool),
                         ptr(slot_tables), ptr(forced_idx), ptr(t_out), ptr(ws), ws_bytes, stream_ptr(stream)),
        "bqe_moe_step")


def bqe_assign_formats(err, energy, layer_weight, heldout_tokens, min_tokens: int, tq1_cap_frac: float,
                       fmt_bytes, budget: int):
    """Host call; err (L, E, 3) float64, energy / layer_weight (L,) float64,
    heldout_tokens (L, E) int32 or None, fmt_bytes (3,) uint64.  Returns
    (formats (L, E) int32, lambda, bytes, cost); raises BqeError on a bad
    argument or a budget below what the guard rails allow."""
    import numpy as np
    err = np.ascontiguousarray(err, dtype=np.float64)
    L, E = int(err.shape[0]), int(err.shape[1])
    energy = np.ascontiguousarray(energy, dtype=np.float64)
    layer_weight = np.ascontiguousarray(layer_weight, dtype=np.float64)
    tok = None if heldout_tokens is None else np.ascontiguousarray(heldout_tokens, dtype=np.int32)
    fb = np.ascontiguousarray(fmt_bytes, dtype=np.uint64)
    out = np.zeros((L, E), dtype=np.int32)
    lam = ctypes.c_double()
    nbytes = ctypes.c_uint64()
    cost = ctypes.c_double()
    _ok(lib.bqe_assign_formats(L, E, ptr(err), ptr(energy), ptr(layer_weight), ptr(tok), int(min_tokens),
                               float(tq1_cap_frac), ptr(fb), int(budget), ptr(out), ctypes.byref(lam),
                               ctypes.byref(nbytes), ctypes.byref(cost)), "bqe_assign_formats")
    return out, lam.value, nbytes.value, cost.value


def bqe_cache_create(d, n_layers: int, expert_fmt, pool: bqe_pool, pool_slot_fmt, first_slot: int, n_slots: int,
                     slot_tables):
    """expert_fmt (L, E) and pool_slot_fmt (pool slots,) host int32; slot_tables
    a device tensor of L x (E + 1) int32.  Returns the cache handle (int)."""
    import numpy as np
    ef = np.ascontiguousarray(expert_fmt, dtype=np.int32)
    pf = np.ascontiguousarray(pool_slot_fmt, dtype=np.int32)
    h = _P()
    _ok(lib.bqe_cache_create(ctypes.byref(d), int(n_layers), ptr(ef), ctypes.byref(pool), ptr(pf), int(first_slot),
                             int(n_slots), ptr(slot_tables), ctypes.byref(h)), "bqe_cache_create")
    return h.value


def bqe_cache_destroy(h) -> None:
    lib.bqe_cache_destroy(h)


def bqe_cache_plan(h, layer: int, experts):
    import numpy as np
    ex = np.ascontiguousarray(experts, dtype=np.int32)
    n = int(ex.size)
    slots, miss, ev = (np.zeros(max(n, 1), np.int32) for _ in range(3))
    _ok(lib.bqe_cache_plan(h, int(layer), n, ptr(ex), ptr(slots), ptr(miss), ptr(ev)), "bqe_cache_plan")
    return slots[:n], miss[:n], ev[:n]


def bqe_cache_fetch(h, layer: int, experts, host_src, staging, upload_stream, compute_stream):
    """host_src: a ctypes array of L x E host pointers (pinned canonical expert
    bytes); staging a device tensor.  Returns (plan number, misses)."""
    import numpy as np
    ex = np.ascontiguousarray(experts, dtype=np.int32)
    nm = _I32()
    pl = ctypes.c_int64()
    _ok(lib.bqe_cache_fetch(h, int(layer), int(ex.size), ptr(ex), ctypes.cast(host_src, _P), ptr(staging),
                            staging.numel() * staging.element_size(), stream_ptr(upload_stream),
                            stream_ptr(compute_stream), ctypes.byref(pl), ctypes.byref(nm)), "bqe_cache_fetch")
    return pl.value, nm.value


def bqe_cache_ready(h, plan: int, compute_stream=None) -> None:
    _ok(lib.bqe_cache_ready(h, int(plan), stream_ptr(compute_stream)), "bqe_cache_ready")


def bqe_cache_done(h, plan: int, compute_stream=None) -> None:
    _ok(lib.bqe_cache_done(h, int(plan), stream_ptr(compute_stream)), "bqe_cache_done")


def bqe_cache_stats_get(h) -> dict:
    st = bqe_cache_stats()
    _ok(lib.bqe_cache_stats_get(h, ctypes.byref(st)), "bqe_cache_stats_get")
    return {k: getattr(st, k) for k, _ in st._fields_}


def bqe_verify_pass(draft, target, stats: "bqe_verify_stats | None" = None):
    """Host call.  Returns (emitted tokens, commit mask) of one verify pass."""
    import numpy as np
    d = np.ascontiguousarray(draft, dtype=np.int32)
    t = np.ascontiguousarray(target, dtype=np.int32)
    n = int(d.size)
    em = np.zeros(n + 1, np.int32)
    mask = np.zeros(n + 1, np.int32)
    ne = _I32()
    _ok(lib.bqe_verify_pass(n, ptr(d) if n else None, ptr(t), ptr(em), ctypes.byref(ne), ptr(mask),
                            ctypes.byref(stats) if stats is not None else None), "bqe_verify_pass")
    return em[:ne.value], mask


def bqe_check(ws, stream=None) -> tuple[int, int]:
    """Returns (status, detail) without raising."""
    det = _I32(0)
    rc = lib.bqe_check(ptr(ws), stream_ptr(stream), ctypes.byref(det))
    return rc, det.value


def bqe_check_noalloc(stream=None) -> tuple[int, int]:
    """The no-allocation entry point's error word: (status, detail) without raising."""
    det = _I32(0)
    rc = lib.bqe_check_noalloc(stream_ptr(stream), ctypes.byref(det))
    return rc, det.value


def bqe_set_wait_limit_ns(ns: int) -> None:
    lib.bqe_set_wait_limit_ns(int(ns))


def bqe_set_test_drop_item(item: int) -> None:
    lib.bqe_set_test_drop_item(int(item))


def bqe_set_diag(on: bool) -> None:
    lib.bqe_set_diag(1 if on else 0)


def bqe_diag_offset(d, M: int) -> int:
    return lib.bqe_diag_offset(ctypes.byref(d), M)


def bqe_set_prefill_f16(on: bool) -> None:
    lib.bqe_set_prefill_f16(1 if on else 0)


def bqe_prefill_diag_offset(d, T: int) -> int:
    return lib.bqe_prefill_diag_offset(ctypes.byref(d), T)


PREFILL_KERNELS = ("logits", "select", "plan", "fill", "gather", "gemm_w13", "gemm_w2", "combine")


def bqe_prefill_kernel_ms() -> dict:
    """Per-kernel milliseconds of the last bqe_moe_prefill call made in diagnostic mode."""
    buf = (ctypes.c_float * len(PREFILL_KERNELS))()
    _ok(lib.bqe_prefill_kernel_ms(ctypes.addressof(buf)), "bqe_prefill_kernel_ms")
    return dict(zip(PREFILL_KERNELS, list(buf)))

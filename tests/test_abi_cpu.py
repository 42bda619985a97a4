"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point of include/bqe.h, the format sizes agree with the
pages' bits per weight, and the host packer writes blocks that the oracle
decodes to the intended values."""
import os
import re

import numpy as np
import pytest

import synth
from oracle import formats as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def A():
    from bit_quantised_expert_gb300 import buildlib
    buildlib.build()
    from bit_quantised_expert_gb300 import _abi
    return _abi


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(bqe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(A):
    names = declared_functions()
    assert len(names) >= 15, names
    missing = [n for n in names if not hasattr(A.lib, n)]
    assert not missing, missing
    # and the binding marshals every one of them
    assert set(names) <= set(A.SIGNATURES), set(names) - set(A.SIGNATURES)


def test_block_sizes(A):
    for fmt, (bw, bb) in F.BLOCK.items():
        assert A.bqe_block_weights(fmt) == bw
        assert A.bqe_block_bytes(fmt) == bb
    assert A.bqe_block_bytes(0) == 0 and A.bqe_block_bytes(6) == 0
    assert A.bqe_packed_bytes(A.BQE_FMT_MXFP4, 2304, 5120) == 2304 * 160 * 17
    assert A.bqe_packed_bytes(A.BQE_FMT_TQ1, 32, 100) == 0  # not a whole block
    d = A.desc(5120, 2304, 384, 6)
    assert A.bqe_expert_bytes(d, A.BQE_FMT_MXFP4) == 18_800_640
    assert A.bqe_expert_bytes(d, A.BQE_FMT_NVFP4) == 3 * 5120 * 2304 * 9 // 16 == 19_906_560  # 4.5 bpw
    for fmt in (1, 2, 3, 4, 5):
        assert A.bqe_expert_bytes(d, fmt) == synth.expert_bytes(fmt, 5120, 2304)


def test_workspace_bytes(A):
    d = A.desc(5120, 2304, 384, 6)
    w1 = A.bqe_workspace_bytes(d, 1)
    w8 = A.bqe_workspace_bytes(d, 8)
    assert 0 < w1 < w8
    assert A.bqe_workspace_bytes(d, 0) == 0
    assert A.bqe_workspace_bytes(d, 9) == 0
    assert A.bqe_workspace_bytes(A.desc(5000, 2304, 384, 6), 1) == 0
    assert A.bqe_workspace_bytes(A.desc(5120, 2304, 384, 6, 2), 1) == 0


def _intended(fmt, codes, scales):
    """Weights a packer input stands for, from the format definitions."""
    bw = F.BLOCK[fmt][0]
    c = codes.reshape(-1, bw).astype(np.float64)
    if fmt in (F.MXFP4, F.NVFP4):
        mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6.0])
        ci = codes.reshape(-1, bw).astype(np.int64)
        v = np.where(ci & 8, -mag[ci & 7], mag[ci & 7])
        if fmt == F.MXFP4:
            return v * np.exp2(scales.reshape(-1, 1).astype(np.float64) - 127)
        import torch  # E4M3 scale through PyTorch's own float8 conversion
        sc = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        return v * sc.reshape(-1, 1)
    d = scales.reshape(-1, A_SB[fmt])[:, -2:].copy().view(np.float16).astype(np.float64)
    if fmt == F.Q2_0:
        return d * (2 * c - 3)
    if fmt == F.TQ1:
        return d * (c - 1)
    s = scales.reshape(-1, 18)[:, :16].astype(np.float64)
    return d * np.repeat(s, 16, axis=1) * (c - 4)


A_SB = {F.TQ1: 2, F.Q2_0: 2, F.Q3_K: 18, F.MXFP4: 1, F.NVFP4: 1}


@pytest.mark.parametrize("fmt", [F.TQ1, F.Q2_0, F.Q3_K, F.MXFP4, F.NVFP4])
def test_pack_matches_oracle_decode(A, fmt):
    rng = np.random.default_rng(fmt)
    rows, cols = 4, 512
    bw, bb = F.BLOCK[fmt]
    nblk = rows * cols // bw
    hi = {F.TQ1: 3, F.Q2_0: 4, F.Q3_K: 8, F.MXFP4: 16, F.NVFP4: 16}[fmt]
    codes = rng.integers(0, hi, size=rows * cols, dtype=np.uint8)
    if fmt == F.MXFP4:
        scales = rng.integers(100, 140, size=nblk, dtype=np.uint8)
    elif fmt == F.NVFP4:
        scales = rng.integers(0, 256, size=nblk, dtype=np.uint8)
        scales[(scales & 0x7F) == 0x7F] = 0x38  # no NaN scale
    else:
        d = np.abs(rng.normal(0, 0.05, size=nblk)).astype(np.float16).view(np.uint8).reshape(nblk, 2)
        if fmt == F.Q3_K:
            s = rng.integers(0, 64, size=(nblk, 16), dtype=np.uint8)
            scales = np.concatenate([s, d], axis=1).reshape(-1)
        else:
            scales = d.reshape(-1)
    out = np.zeros(A.bqe_packed_bytes(fmt, rows, cols), dtype=np.uint8)
    A.bqe_pack(fmt, rows, cols, codes, np.ascontiguousarray(scales), out)
    got = F.dequant_matrix(fmt, out, rows, cols).reshape(-1, bw)
    want = _intended(fmt, codes, np.ascontiguousarray(scales))
    assert np.array_equal(got, want)


def test_pack_rejects_out_of_domain(A):
    codes = np.full(64, 4, dtype=np.uint8)  # q = 4 is not a 2-bit code
    scales = np.zeros(2, dtype=np.uint8)
    out = np.zeros(18, dtype=np.uint8)
    with pytest.raises(A.BqeError) as e:
        A.bqe_pack(A.BQE_FMT_Q2_0, 1, 64, codes, scales, out)
    assert e.value.status == A.BQE_EINVAL
    with pytest.raises(A.BqeError):
        A.bqe_pack(A.BQE_FMT_MXFP4, 1, 32, np.zeros(32, np.uint8), np.array([255], np.uint8),
                   np.zeros(17, np.uint8))
    for nan in (0x7F, 0xFF):
        with pytest.raises(A.BqeError):
            A.bqe_pack(A.BQE_FMT_NVFP4, 1, 16, np.zeros(16, np.uint8), np.array([nan], np.uint8),
                       np.zeros(9, np.uint8))


def test_status_strings(A):
    for s in range(7):
        assert A.status_name(s)
    assert "unknown" in A.status_name(99)


def test_argument_checks_before_any_device_work(A):
    """The entry points reject bad arguments synchronously, before touching a
    pointer or the device (fake, aligned addresses; nothing is dereferenced)."""
    import ctypes
    lib = A.lib
    d = A.desc(5120, 2304, 384, 6)
    fake = ctypes.c_void_p(1 << 20)  # 256-byte aligned, never dereferenced
    pool = A.bqe_pool(base=1 << 20, base_bytes=1 << 30, slot_off=1 << 21, slot_fmt=1 << 22, n_slots=385)
    bad_pool = A.bqe_pool(base=None, base_bytes=0, slot_off=None, slot_fmt=None, n_slots=0)
    need = A.bqe_workspace_bytes(d, 1)
    args = lambda M, x, ws, nb, p=pool: (ctypes.byref(d), M, x, fake, None, ctypes.byref(p), fake, None, fake, 0,  # noqa: E731
                                         None, None, ws, nb, None)
    assert lib.bqe_moe_layer_forward(*args(0, fake, fake, need)) == A.BQE_EINVAL      # no rows
    assert lib.bqe_moe_layer_forward(*args(9, fake, fake, need)) == A.BQE_EINVAL      # more than 8 rows
    assert lib.bqe_moe_layer_forward(*args(1, None, fake, need)) == A.BQE_EINVAL      # no input
    assert lib.bqe_moe_layer_forward(*args(1, fake, None, need)) == A.BQE_EINVAL      # no workspace
    assert lib.bqe_moe_layer_forward(*args(1, fake, ctypes.c_void_p((1 << 20) + 16), need)) == A.BQE_EINVAL  # misaligned
    assert lib.bqe_moe_layer_forward(*args(1, fake, fake, need, bad_pool)) == A.BQE_EINVAL  # empty pool
    assert lib.bqe_moe_layer_forward(*args(1, fake, fake, need - 256)) == A.BQE_ENOSPC     # workspace too small
    for bad in (A.desc(5120, 2304, 384, 6, n_shared=2), A.desc(5120, 2304, 384, 0), A.desc(5000, 2304, 384, 6),
                A.desc(5120, 2304, 513, 6), A.desc(5120, 2304, 384, 17)):
        assert A.bqe_workspace_bytes(bad, 1) == 0
        assert lib.bqe_moe_layer_forward(ctypes.byref(bad), 1, fake, fake, None, ctypes.byref(pool), fake, None,
                                         fake, 0, None, None, fake, need, None) == A.BQE_EINVAL
    # prefill: token count bounds and the workspace size
    assert A.bqe_prefill_workspace_bytes(d, 0) == 0
    pneed = A.bqe_prefill_workspace_bytes(d, 64)
    assert pneed > 0 and A.bqe_prefill_workspace_bytes(d, 128) > pneed
    assert lib.bqe_moe_prefill(ctypes.byref(d), 0, fake, fake, None, ctypes.byref(pool), fake, None, fake, 0, None,
                               None, fake, pneed, None) == A.BQE_EINVAL
    assert lib.bqe_moe_prefill(ctypes.byref(d), 64, fake, fake, None, ctypes.byref(pool), fake, None, fake, 0, None,
                               None, fake, pneed - 256, None) == A.BQE_ENOSPC
    assert lib.bqe_workspace_init(None, 16, None) == A.BQE_EINVAL


@pytest.mark.parametrize("fmt", [F.TQ1, F.Q2_0, F.Q3_K, F.MXFP4, F.NVFP4])
def test_unpack_host_inverts_pack(A, fmt):
    """bqe_unpack_host returns the codes and scale bytes bqe_pack was given,
    for every code of the format's domain."""
    rng = np.random.default_rng(40 + fmt)
    rows, cols = 3, 1024
    bw, _ = F.BLOCK[fmt]
    nblk = rows * cols // bw
    hi = {F.TQ1: 3, F.Q2_0: 4, F.Q3_K: 8, F.MXFP4: 16, F.NVFP4: 16}[fmt]
    codes = rng.integers(0, hi, size=rows * cols, dtype=np.uint8)
    sb = A_SB[fmt]
    if fmt == F.MXFP4:
        scales = rng.integers(0, 255, size=nblk, dtype=np.uint8)  # 255 (NaN) is not an encodable scale
    elif fmt == F.NVFP4:
        scales = rng.integers(0, 256, size=nblk, dtype=np.uint8)
        scales[(scales & 0x7F) == 0x7F] = 0  # 0x7F / 0xFF (NaN) are not encodable scales
    elif fmt == F.Q3_K:
        d = rng.integers(0, 256, size=(nblk, 2), dtype=np.uint8)
        scales = np.concatenate([rng.integers(0, 64, size=(nblk, 16), dtype=np.uint8), d], axis=1).reshape(-1)
    else:
        scales = rng.integers(0, 256, size=nblk * 2, dtype=np.uint8)
    packed = np.zeros(A.bqe_packed_bytes(fmt, rows, cols), dtype=np.uint8)
    A.bqe_pack(fmt, rows, cols, codes, np.ascontiguousarray(scales), packed)
    c2 = np.zeros_like(codes)
    s2 = np.zeros(nblk * sb, dtype=np.uint8)
    A.bqe_unpack_host(fmt, rows, cols, packed, c2, s2)
    assert np.array_equal(c2, codes)
    assert np.array_equal(s2, scales)


def test_unpack_host_rejects_bad_ternary_byte(A):
    blk = np.zeros(56, dtype=np.uint8)
    blk[7] = 243  # five trits span 0..242
    with pytest.raises(A.BqeError) as e:
        A.bqe_unpack_host(A.BQE_FMT_TQ1, 1, 256, blk, np.zeros(256, np.uint8), np.zeros(2, np.uint8))
    assert e.value.status == A.BQE_EINVAL


def test_pool_bytes_layout(A):
    """Pool size = the two tables (uint64 offsets, int32 formats, each rounded
    up to 256 bytes) + every slot's expert bytes rounded up to 256."""
    d = A.desc(5120, 2304, 384, 6)
    fm = np.array([F.TQ1, F.Q2_0, F.Q3_K, F.MXFP4, F.Q2_0, F.NVFP4], dtype=np.int32)
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    want = up(8 * 6) + up(4 * 6) + sum(up(synth.expert_bytes(int(f), 5120, 2304)) for f in fm)
    assert A.bqe_pool_bytes(d, fm) == want
    assert A.bqe_pool_bytes(d, np.array([1, 6], np.int32)) == 0  # unknown format
    assert A.bqe_pool_bytes(A.desc(5000, 2304, 384, 6), fm) == 0


def test_pool_init_argument_checks(A):
    """bqe_pool_init rejects bad arguments before any copy: no GPU is needed
    to see the status (the fake device address is never dereferenced)."""
    import ctypes
    d = A.desc(5120, 2304, 384, 6)
    fm = np.array([F.MXFP4, F.Q2_0], dtype=np.int32)
    need = A.bqe_pool_bytes(d, fm)
    p = A.bqe_pool()
    fp = fm.ctypes.data
    lib = A.lib
    assert lib.bqe_pool_init(None, ctypes.byref(d), 2, fp, 1 << 20, need, None) == A.BQE_EINVAL
    assert lib.bqe_pool_init(ctypes.byref(p), ctypes.byref(d), 0, fp, 1 << 20, need, None) == A.BQE_EINVAL
    assert lib.bqe_pool_init(ctypes.byref(p), ctypes.byref(d), 2, fp, None, need, None) == A.BQE_EINVAL
    assert lib.bqe_pool_init(ctypes.byref(p), ctypes.byref(d), 2, fp, (1 << 20) + 64, need, None) == A.BQE_EINVAL
    assert lib.bqe_pool_init(ctypes.byref(p), ctypes.byref(d), 2, fp, 1 << 20, need - 1, None) == A.BQE_ENOSPC
    bad = np.array([F.MXFP4, 7], dtype=np.int32)
    assert lib.bqe_pool_init(ctypes.byref(p), ctypes.byref(d), 2, bad.ctypes.data, 1 << 20, need, None) == A.BQE_EINVAL
    # upload: slot out of range or an empty pool struct
    assert lib.bqe_pool_upload(ctypes.byref(p), ctypes.byref(d), 0, 1 << 20, None) == A.BQE_EINVAL


def test_noalloc_argument_checks_before_any_device_work(A):
    """The allocation-free entry point checks its arguments before it touches
    its fixed device array: without a GPU, a bad call still gets its own
    status (a call that reached the device would report BQE_ECUDA)."""
    import ctypes
    lib = A.lib
    d = A.desc(1024, 768, 24, 3)
    fake = ctypes.c_void_p(1 << 20)
    pool = A.bqe_pool(base=1 << 20, base_bytes=1 << 30, slot_off=1 << 21, slot_fmt=1 << 22, n_slots=25)
    bad_pool = A.bqe_pool(base=None, base_bytes=0, slot_off=None, slot_fmt=None, n_slots=0)
    call = lambda dd, M, x, p, out: lib.bqe_moe_layer_forward_noalloc(  # noqa: E731
        ctypes.byref(dd), M, x, fake, None, ctypes.byref(p), fake, None, out, 0, None, None, None, None)
    assert call(d, 0, fake, pool, fake) == A.BQE_EINVAL       # no rows
    assert call(d, 9, fake, pool, fake) == A.BQE_EINVAL       # more than 8 rows
    assert call(d, 1, None, pool, fake) == A.BQE_EINVAL       # no input
    assert call(d, 1, fake, pool, None) == A.BQE_EINVAL       # no output
    assert call(d, 1, fake, bad_pool, fake) == A.BQE_EINVAL   # empty pool
    assert call(A.desc(1000, 768, 24, 3), 1, fake, pool, fake) == A.BQE_EINVAL  # hidden not a multiple of 512
    big = A.desc(7168, 2304, 384, 6)
    assert A.bqe_workspace_bytes(big, 8) > 8 << 20
    assert call(big, 8, fake, pool, fake) == A.BQE_ENOSPC     # workspace beyond the fixed array

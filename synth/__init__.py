"""Seeded synthetic inputs for the block-quantised MoE expert layer.

This module is shared by the tests, the benchmark and the oracle's callers.
It holds no arithmetic of the method: it only draws random bytes that are
valid in each packed block layout, router weights, selection biases,
activations (rounded to bf16 as inputs) and Zipf-skewed forced routings.
Which byte of a block is a code and which is a scale is layout knowledge,
not decoding; no block is ever decoded here.

Two backends draw the same kinds of inputs:
  * numpy (``np.random.default_rng(seed)``): small cases, reproducible on
    any host; these are what the oracle consumes in parity tests;
  * torch on a CUDA device (``torch.Generator(device)``): multi-GB pools for
    the benchmark and the full-size parity cases, generated where they live.

Block layouts (canonical, array-of-blocks, blocks run along a row's input
dimension):
  PTQ1_0 ternary  256 weights, 56 B: 51 bytes of 5 base-3 digits, 1 byte with
                  the 256th digit, fp16 d, 2 zero pad bytes
  Q2_0             64 weights, 18 B: 16 bytes of 2-bit codes, fp16 d
  Q3_K            256 weights, 110 B: 64 B low-2-bit plane, 32 B high-bit
                  plane, 12 B of sixteen 6-bit sub-scales, fp16 d
  MXFP4            32 weights, 17 B: 16 B of E2M1 nibbles, 1 B UE8M0 exponent
  NVFP4            16 weights, 9 B: 8 B of E2M1 nibbles, 1 B FP8 E4M3 scale
"""
from __future__ import annotations

import numpy as np

TQ1, Q2_0, Q3_K, MXFP4, NVFP4 = 1, 2, 3, 4, 5
FMT_NAMES = {TQ1: "tq1", Q2_0: "q2_0", Q3_K: "q3_k", MXFP4: "mxfp4", NVFP4: "nvfp4"}
# format -> (weights per block, bytes per block)
BLOCK = {TQ1: (256, 56), Q2_0: (64, 18), Q3_K: (256, 110), MXFP4: (32, 17), NVFP4: (16, 9)}


def block_weights(fmt: int) -> int:
    return BLOCK[fmt][0]


def block_bytes(fmt: int) -> int:
    return BLOCK[fmt][1]


def matrix_bytes(fmt: int, rows: int, cols: int) -> int:
    bw, bb = BLOCK[fmt]
    assert cols % bw == 0
    return rows * (cols // bw) * bb


def expert_bytes(fmt: int, hidden: int, inter: int) -> int:
    """W1 (inter x hidden) | W3 (inter x hidden) | W2 (hidden x inter)."""
    return 2 * matrix_bytes(fmt, inter, hidden) + matrix_bytes(fmt, hidden, inter)


# ----------------------------------------------------------------------------
# numpy backend
# ----------------------------------------------------------------------------

def fp16_bits_abs_normal(rng, n: int, std: float) -> np.ndarray:
    """fp16 bit patterns of |N(0, std)| (numpy's float16 cast rounds to nearest even)."""
    return np.abs(rng.normal(0.0, std, size=n)).astype(np.float16).view(np.uint16)


def random_blocks(rng, fmt: int, nblocks: int) -> np.ndarray:
    """nblocks valid canonical blocks of one format, shape (nblocks, block_bytes)."""
    bw, bb = BLOCK[fmt]
    out = np.zeros((nblocks, bb), dtype=np.uint8)
    if fmt == MXFP4:
        out[:, :16] = rng.integers(0, 256, size=(nblocks, 16), dtype=np.uint8)
        # UE8M0 exponent byte uniform in 119..123, i.e. 2^-8 .. 2^-4
        out[:, 16] = rng.integers(119, 124, size=nblocks, dtype=np.uint8)
    elif fmt == NVFP4:
        out[:, :8] = rng.integers(0, 256, size=(nblocks, 8), dtype=np.uint8)
        # positive E4M3 scale bytes 0..39: exponent field 0..4, i.e. up to
        # 1.875 x 2^-3, subnormals and zero included (0x7F / 0xFF, NaN, never)
        out[:, 8] = rng.integers(0, 40, size=nblocks, dtype=np.uint8)
    elif fmt == Q2_0:
        out[:, :16] = rng.integers(0, 256, size=(nblocks, 16), dtype=np.uint8)
        d = fp16_bits_abs_normal(rng, nblocks, 0.02)
        out[:, 16] = d & 0xFF
        out[:, 17] = d >> 8
    elif fmt == TQ1:
        # each of the first 51 bytes packs 5 digits in 0..2 (byte value 0..242);
        # byte 51 holds one digit (0..2); bytes 54..55 are zero padding
        out[:, :51] = rng.integers(0, 243, size=(nblocks, 51), dtype=np.uint8)
        out[:, 51] = rng.integers(0, 3, size=nblocks, dtype=np.uint8)
        d = fp16_bits_abs_normal(rng, nblocks, 0.02)
        out[:, 52] = d & 0xFF
        out[:, 53] = d >> 8
    elif fmt == Q3_K:
        # any bit pattern is a valid code plane / sub-scale stream
        out[:, :108] = rng.integers(0, 256, size=(nblocks, 108), dtype=np.uint8)
        d = fp16_bits_abs_normal(rng, nblocks, 0.02 / 32.0)
        out[:, 108] = d & 0xFF
        out[:, 109] = d >> 8
    else:
        raise ValueError(fmt)
    return out


def random_matrix(rng, fmt: int, rows: int, cols: int) -> np.ndarray:
    bw, bb = BLOCK[fmt]
    return random_blocks(rng, fmt, rows * (cols // bw)).reshape(-1)


def random_expert(rng, fmt: int, hidden: int, inter: int) -> np.ndarray:
    """Canonical bytes of one expert: W1 | W3 | W2, each row-major in blocks."""
    return np.concatenate([
        random_matrix(rng, fmt, inter, hidden),
        random_matrix(rng, fmt, inter, hidden),
        random_matrix(rng, fmt, hidden, inter),
    ])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.
    Input preparation only: activations are bf16 by definition of the workload."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def x_bf16(rng, m: int, hidden: int, std: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits(rng.normal(0.0, std, size=(m, hidden)).astype(np.float32))


def router_weights(rng, n_experts: int, hidden: int) -> np.ndarray:
    return rng.normal(0.0, 1.0 / np.sqrt(hidden), size=(n_experts, hidden)).astype(np.float32)


def selection_bias(rng, n_experts: int, std: float) -> np.ndarray:
    if std == 0.0:
        return np.zeros(n_experts, dtype=np.float32)
    return rng.normal(0.0, std, size=n_experts).astype(np.float32)


def largest_remainder_counts(n: int, shares) -> list[int]:
    raw = [n * s for s in shares]
    base = [int(np.floor(r)) for r in raw]
    rem = n - sum(base)
    order = sorted(range(len(shares)), key=lambda i: -(raw[i] - base[i]))
    for i in order[:rem]:
        base[i] += 1
    return base


# Byte shares of the per-expert mix: ternary / Q2_0 / Q3_K weight shares
# (Strata 4090 post, section 5.1 table: 42.8% / 39.2% / 18.0%).
MIX_SHARES = ((TQ1, 0.428), (Q2_0, 0.392), (Q3_K, 0.180))


def assign_formats(rng, n: int, shares=MIX_SHARES) -> np.ndarray:
    counts = largest_remainder_counts(n, [s for _, s in shares])
    fm = np.concatenate([np.full(c, f, dtype=np.int32) for (f, _), c in zip(shares, counts)])
    rng.shuffle(fm)
    return fm


def format_error_proxy(rng, n_layers: int, n_experts: int):
    """Synthetic inputs of the per-expert format assignment (the real ones
    are held-out errors of quantised experts on calibration data, which is
    not here).  Returns err (L, E, 3) for ternary / Q2_0 / Q3_K, the routed
    output energy of each layer (L,) and held-out token counts (L, E):
      energy_l     ~ lognormal(0, 0.5);
      sensitivity  ~ lognormal(0, 0.7) per expert, x4 for every expert of one
                     layer (three quarters of the way down: one layer much
                     more sensitive than the rest, as the Strata 4090 post
                     reports for one layer);
      err[l,e,f]   = energy_l * sensitivity * 4^-bpw_f * lognormal(0, 0.15),
                     bpw = 1.75 / 2.25 / 3.4375 (a round-to-nearest error
                     that falls 4x per bit, with per-format scatter);
      tokens       ~ Poisson(lognormal(3, 1)) (a few rarely routed experts)."""
    energy = rng.lognormal(0.0, 0.5, size=n_layers)
    sens = rng.lognormal(0.0, 0.7, size=(n_layers, n_experts))
    sens[(3 * n_layers) // 4] *= 4.0
    bpw = np.array([1.75, 2.25, 3.4375])
    jitter = rng.lognormal(0.0, 0.15, size=(n_layers, n_experts, 3))
    err = energy[:, None, None] * sens[:, :, None] * (4.0 ** -bpw)[None, None, :] * jitter
    tokens = rng.poisson(rng.lognormal(3.0, 1.0, size=(n_layers, n_experts))).astype(np.int32)
    return err, energy, tokens


def zipf_probs(n: int, s: float) -> np.ndarray:
    p = 1.0 / np.arange(1, n + 1, dtype=np.float64) ** s
    return p / p.sum()


def zipf_forced_idx(rng, m: int, n_experts: int, k: int, s: float, perm: np.ndarray) -> np.ndarray:
    """Rows of k distinct experts drawn without replacement, expert perm[r]
    having Zipf(s) popularity of rank r."""
    p = zipf_probs(n_experts, s)
    out = np.empty((m, k), dtype=np.int32)
    for i in range(m):
        ranks = rng.choice(n_experts, size=k, replace=False, p=p)
        out[i] = perm[ranks]
    return out


# ----------------------------------------------------------------------------
# Workload presets (sizes of a DeepSeek-V4.1-Flash MoE layer and a tiny one)
# ----------------------------------------------------------------------------

TINY = dict(name="tiny-q2_0", hidden=512, inter=256, n_experts=16, top_k=2)
DSV4 = dict(name="dsv4flash", hidden=5120, inter=2304, n_experts=384, top_k=6)


def tiny_layer(seed: int = 0, m: int = 1):
    """Tiny layer: 16 routed + 1 shared expert, all Q2_0, zero bias, top-2."""
    rng = np.random.default_rng(seed)
    H, I, E, k = TINY["hidden"], TINY["inter"], TINY["n_experts"], TINY["top_k"]
    router = router_weights(rng, E, H)
    experts = [random_expert(rng, Q2_0, H, I) for _ in range(E + 1)]
    fmts = np.full(E + 1, Q2_0, dtype=np.int32)
    x = x_bf16(rng, m, H)
    return dict(hidden=H, inter=I, n_experts=E, top_k=k, router=router,
                bias=np.zeros(E, np.float32), experts=experts, fmts=fmts, x=x)


def small_layer(seed: int, fmt_list, hidden: int, inter: int, n_experts: int, top_k: int,
                m: int, bias_std: float = 0.0):
    """A layer of arbitrary small shape; expert e has format fmt_list[e] (last = shared)."""
    rng = np.random.default_rng(seed)
    router = router_weights(rng, n_experts, hidden)
    experts = [random_expert(rng, int(f), hidden, inter) for f in fmt_list]
    bias = selection_bias(rng, n_experts, bias_std)
    x = x_bf16(rng, m, hidden)
    return dict(hidden=hidden, inter=inter, n_experts=n_experts, top_k=top_k, router=router,
                bias=bias, experts=experts, fmts=np.asarray(fmt_list, np.int32), x=x)


# ----------------------------------------------------------------------------
# torch backend (device-side generation of large pools)
# ----------------------------------------------------------------------------

def torch_random_blocks(gen, fmt: int, nblocks: int, device):
    """Same kinds of blocks as random_blocks(), drawn on `device` with a seeded
    torch.Generator.  Returns a uint8 tensor of shape (nblocks, block_bytes)."""
    import torch
    bw, bb = BLOCK[fmt]
    out = torch.zeros((nblocks, bb), dtype=torch.uint8, device=device)

    def ri(lo, hi, shape):
        return torch.randint(lo, hi, shape, generator=gen, device=device, dtype=torch.int32).to(torch.uint8)

    def d_bits(std):
        d = torch.randn(nblocks, generator=gen, device=device, dtype=torch.float32).abs_() * std
        b = d.to(torch.float16).view(torch.int16).to(torch.int32) & 0xFFFF
        return (b & 0xFF).to(torch.uint8), (b >> 8).to(torch.uint8)

    if fmt == MXFP4:
        out[:, :16] = ri(0, 256, (nblocks, 16))
        out[:, 16] = ri(119, 124, (nblocks,))
    elif fmt == NVFP4:
        out[:, :8] = ri(0, 256, (nblocks, 8))
        out[:, 8] = ri(0, 40, (nblocks,))
    elif fmt == Q2_0:
        out[:, :16] = ri(0, 256, (nblocks, 16))
        lo, hi = d_bits(0.02)
        out[:, 16], out[:, 17] = lo, hi
    elif fmt == TQ1:
        out[:, :51] = ri(0, 243, (nblocks, 51))
        out[:, 51] = ri(0, 3, (nblocks,))
        lo, hi = d_bits(0.02)
        out[:, 52], out[:, 53] = lo, hi
    elif fmt == Q3_K:
        out[:, :108] = ri(0, 256, (nblocks, 108))
        lo, hi = d_bits(0.02 / 32.0)
        out[:, 108], out[:, 109] = lo, hi
    else:
        raise ValueError(fmt)
    return out


def torch_random_expert(gen, fmt: int, hidden: int, inter: int, device):
    import torch
    bw, _ = BLOCK[fmt]
    n1 = inter * (hidden // bw)
    n2 = hidden * (inter // bw)
    return torch.cat([
        torch_random_blocks(gen, fmt, n1, device).reshape(-1),
        torch_random_blocks(gen, fmt, n1, device).reshape(-1),
        torch_random_blocks(gen, fmt, n2, device).reshape(-1),
    ])

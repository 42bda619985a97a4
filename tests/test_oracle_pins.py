"""Pins for the oracle: each check ties it to something other than itself.

  * golden blocks written by hand from the layout definitions (tests/golden);
  * exhaustive enumeration (all 243 ternary bytes, all fp16 bit patterns,
    every E2M1 code x several exponents, every Q3_K (q, s) pair) against
    independent constructions;
  * the pages' closed forms and bits-per-weight identities;
  * brute-force loops on tiny shapes for the router, top-k, expert FFN and
    layer combine, and special cases with closed forms;
  * planted mistakes in the oracle that these pins must catch.
"""
import itertools
import math
import os

import numpy as np
import pytest

from oracle import formats as F
from oracle import moe as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    cases = []
    blk = None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("block:"):
            blk = np.array([int(t, 16) for t in line.split()[1:]], dtype=np.uint8)
        elif line.startswith("values:"):
            vals, group = [], []
            for t in line.split()[1:]:
                if t.startswith("*"):
                    vals += group * int(t[1:])
                    group = []
                else:
                    group.append(float(t))
            vals += group
            cases.append((blk, np.array(vals)))
            blk = None
    return cases


def same_bits(a, b):
    """Exact equality including the sign of zero."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return a.shape == b.shape and np.array_equal(a.view(np.uint64), b.view(np.uint64))


# ---------------------------------------------------------------- golden blocks

@pytest.mark.parametrize("name,fn,nw", [
    ("mxfp4.txt", F.dequant_mxfp4, 32),
    ("q2_0.txt", F.dequant_q2_0, 64),
    ("tq1.txt", F.dequant_tq1, 256),
    ("nvfp4.txt", F.dequant_nvfp4, 16),
])
def test_golden_blocks(name, fn, nw):
    cases = read_golden(name)
    assert cases
    for blk, vals in cases:
        assert vals.size == nw
        got = fn(blk[None, :])[0]
        assert same_bits(got, vals), (name, got, vals)


# --------------------------------------------------------- exhaustive decodes

def test_fp16_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    got = F.fp16_to_f64((bits & 0xFF).astype(np.uint8), (bits >> 8).astype(np.uint8))
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert same_bits(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_e2m1_every_code_and_exponent():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for E in (0, 1, 119, 120, 121, 122, 123, 127, 200, 254):
        blk = np.zeros((16, 17), dtype=np.uint8)
        for c in range(16):
            blk[c, :16] = c | (c << 4)
            blk[c, 16] = E
        got = F.dequant_mxfp4(blk)
        for c in range(16):
            m = mags[c & 7] * math.ldexp(1.0, E - 127)
            want = -m if c & 8 else m
            assert same_bits(got[c], np.full(32, want)), (E, c)


def test_e4m3_every_byte_against_torch():
    """All 256 E4M3 scale bytes against PyTorch's float8_e4m3fn conversion."""
    import torch
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_to_f64(b)
    fin = np.isfinite(ref)
    assert same_bits(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and int(np.isnan(got).sum()) == 2


def test_nvfp4_every_code_and_scale():
    """Each code times each finite scale: the product of the two definitions."""
    e2m1 = F.e2m1_to_f64(np.arange(16))
    for sb in range(256):
        if sb in (0x7F, 0xFF):
            continue
        blk = np.zeros((2, 9), dtype=np.uint8)
        blk[0, :8] = [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]
        blk[1, :8] = [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]
        blk[:, 8] = sb
        got = F.dequant_nvfp4(blk)
        sc = F.e4m3_to_f64(np.array([sb], np.uint8))[0]
        assert same_bits(got[0], e2m1 * sc), sb


def test_ternary_all_243_bytes():
    # independent enumeration: digit tuples in lexicographic order with the
    # first digit least significant
    for value, digits in enumerate((tuple(reversed(p)) for p in itertools.product(range(3), repeat=5))):
        assert F.tq1_digits(np.array([value]))[0].tolist() == list(digits)
    blk = np.zeros((243, 56), dtype=np.uint8)
    for v in range(243):
        blk[v, :51] = v
        blk[v, 51] = v % 3
        blk[v, 52:54] = (0x00, 0x3C)
    got = F.dequant_tq1(blk)
    for v in range(243):
        ds = [(v // 3 ** r) % 3 for r in range(5)]
        want = [d - 1.0 for d in ds] * 51 + [float(v % 3) - 1.0]
        assert same_bits(got[v], want)


def _bits_le(fields):
    """Pack (value, width) fields LSB-first into bytes (independent bit writer)."""
    acc, pos = 0, 0
    for v, w in fields:
        assert 0 <= v < (1 << w)
        acc |= v << pos
        pos += w
    return list(acc.to_bytes((pos + 7) // 8, "little"))


def build_q3k(q, s, d_bits):
    """Hand-assembled Q3_K block from 256 codes q (0..7), 16 sub-scales s (0..63)
    and the fp16 bit pattern of d, following the layout text field by field."""
    lo = _bits_le([(qj & 3, 2) for qj in q])          # 64 bytes
    hi = _bits_le([(qj >> 2, 1) for qj in q])         # 32 bytes
    sc = _bits_le([(sj, 6) for sj in s])              # 12 bytes
    return np.array(lo + hi + sc + [d_bits & 0xFF, d_bits >> 8], dtype=np.uint8)


def test_q3k_every_code_and_subscale():
    # every q in 0..7 appears at every position modulo 8, every s in 0..63
    for base in range(0, 64, 16):
        s = [base + j for j in range(16)]
        q = [(j * 3 + base) % 8 for j in range(256)]
        blk = build_q3k(q, s, 0x3C00)
        assert blk.size == 110
        got = F.dequant_q3k(blk[None])[0]
        want = [s[j // 16] * (q[j] - 4.0) for j in range(256)]
        assert same_bits(got, want)
    # d = 0.5, s = 63, q alternating 0 / 7
    q = [0 if j % 2 == 0 else 7 for j in range(256)]
    blk = build_q3k(q, [63] * 16, 0x3800)
    got = F.dequant_q3k(blk[None])[0]
    assert same_bits(got, [0.5 * 63 * (qq - 4.0) for qq in q])


def test_q2_0_every_code_position():
    for j in range(64):
        for qv in range(4):
            blk = np.zeros(18, dtype=np.uint8)
            blk[:16] = _bits_le([(qv if i == j else 0, 2) for i in range(64)])
            blk[16:] = (0x00, 0x3C)
            got = F.dequant_q2_0(blk[None])[0]
            want = np.full(64, -3.0)
            want[j] = 2 * qv - 3.0
            assert same_bits(got, want)


def test_mxfp4_nibble_positions():
    for j in range(32):
        blk = np.zeros(17, dtype=np.uint8)
        blk[:16] = _bits_le([(5 if i == j else 0, 4) for i in range(32)])  # code 5 = 3.0
        blk[16] = 127
        got = F.dequant_mxfp4(blk[None])[0]
        want = np.zeros(32)
        want[j] = 3.0
        assert same_bits(got, want)


# ----------------------------------------------------- closed forms from pages

def test_field_report_closed_forms():
    """DeepSeek-V4.1-Flash 4xL20 field report, section 2."""
    H, I, E, L, k = 5120, 2304, 384, 40, 6
    fp4_codes = 3 * H * I // 2                       # 0.5 B per weight
    assert fp4_codes == 17_694_720                   # "17.7 MB"
    assert round(fp4_codes / 1e6, 1) == 17.7
    assert round(k * L * fp4_codes / 1e9, 2) == 4.25  # "4.25 GB" per token
    assert round(L * E * fp4_codes / 1e9) == 272      # "272 GB", 15360 experts
    assert L * E == 15360
    # with one UE8M0 byte per 32 weights (4.25 bpw)
    assert synth.expert_bytes(synth.MXFP4, H, I) == 18_800_640
    # bandwidth upper bounds quoted in the same section
    assert round(4.25 / 25.2 * 1e3) == 169            # ms/token over PCIe
    assert round(4.25 / 864 * 1e3, 1) == 4.9          # ms/token from VRAM


def test_bits_per_weight_identities():
    """Strata 4090 post, section 5.1 table: 1.75 / 2.25 / 3.44 bpw, mix 2.250;
    section 3 check: 543.6 B expert weights x 2.25 bit / 8 = 152.9 GB."""
    bpw = {f: 8.0 * bb / bw for f, (bw, bb) in F.BLOCK.items()}
    assert bpw[F.TQ1] == 1.75
    assert bpw[F.Q2_0] == 2.25
    assert round(bpw[F.Q3_K], 2) == 3.44
    assert bpw[F.MXFP4] == 4.25
    mix = 0.428 * bpw[F.TQ1] + 0.392 * bpw[F.Q2_0] + 0.180 * bpw[F.Q3_K]
    assert round(mix, 3) == 2.250  # shares are weight-count shares
    assert round(543.6e9 * 2.25 / 8 / 1e9, 1) == 152.9
    # slot pool of 4288 slots (field report, section 3B) at the mixed shares
    n = synth.largest_remainder_counts(4288, [0.428, 0.392, 0.180])
    assert n == [1835, 1681, 772]
    per = {f: synth.expert_bytes(f, 5120, 2304) for f in (F.TQ1, F.Q2_0, F.Q3_K)}
    pool = n[0] * per[F.TQ1] + n[1] * per[F.Q2_0] + n[2] * per[F.Q3_K]
    assert 42.5e9 < pool < 42.8e9


def test_dequant_matrix_row_order():
    rng = np.random.default_rng(3)
    for fmt in (F.TQ1, F.Q2_0, F.Q3_K, F.MXFP4):
        bw, bb = F.BLOCK[fmt]
        rows, cols = 3, 2 * 256
        packed = synth.random_matrix(rng, fmt, rows, cols)
        W = F.dequant_matrix(fmt, packed, rows, cols)
        blocks = packed.reshape(rows, cols // bw, bb)
        for r in range(rows):
            for b in range(cols // bw):
                assert same_bits(W[r, b * bw:(b + 1) * bw], F.DECODERS[fmt](blocks[r, b][None])[0])


# ---------------------------------------------------------- router / top-k

def test_sigmoid_and_silu_closed_forms():
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert abs(O.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(O.sigmoid(np.array([math.log(3.0)]))[0] - 0.75) < 1e-15


def test_topk_brute_force():
    rng = np.random.default_rng(1)
    for trial in range(50):
        M, E, H, k = 3, 9, 7, 3
        x = rng.normal(size=(M, H))
        wr = rng.normal(size=(E, H))
        b = rng.normal(size=E) * (trial % 2)
        r = O.route(x, wr, b, k)
        for m in range(M):
            key = []
            for e in range(E):
                z = sum(x[m, h] * wr[e, h] for h in range(H))
                s = 1.0 / (1.0 + math.exp(-z))
                key.append((-(s + b[e]), e, s))
            best = sorted(key)[:k]
            assert [e for _, e, _ in best] == r["idx"][m].tolist()
            tot = sum(s for _, _, s in best)
            assert np.allclose(r["w"][m], [s / tot for _, _, s in best], rtol=1e-13, atol=0)


def test_topk_ties_go_to_lower_index():
    x = np.zeros((1, 4))
    wr = np.zeros((6, 4))
    r = O.route(x, wr, None, 3)  # all scores 0.5
    assert r["idx"][0].tolist() == [0, 1, 2]
    assert np.allclose(r["w"][0], 1 / 3)
    assert r["gap"][0] == 0.0


def test_bias_steers_selection_only():
    """Strata 4090 post, section 5.3: the bias changes which experts are
    computed, the mixing weights stay the exact (unbiased) scores."""
    rng = np.random.default_rng(2)
    x = rng.normal(size=(2, 16))
    wr = rng.normal(size=(10, 16))
    r0 = O.route(x, wr, np.zeros(10), 2)
    loser = int(r0["order"][0, -1])
    b = np.zeros(10)
    b[loser] = 2.0  # larger than any score difference
    r1 = O.route(x, wr, b, 2)
    assert r1["idx"][0, 0] == loser
    s = r1["s"][0]
    sel = r1["idx"][0]
    assert np.allclose(r1["w"][0], s[sel] / s[sel].sum(), rtol=1e-14)
    assert np.array_equal(r1["s"], r0["s"])
    # forced selection keeps unbiased weights too
    r2 = O.route(x, wr, b, 2, forced_idx=np.array([[3, 7], [1, 2]]))
    assert r2["idx"].tolist() == [[3, 7], [1, 2]]
    assert np.allclose(r2["w"][1], r2["s"][1, [1, 2]] / r2["s"][1, [1, 2]].sum())


# ------------------------------------------------------- expert FFN / layer

def test_expert_ffn_brute_force():
    rng = np.random.default_rng(4)
    H, I, R = 6, 4, 2
    x = rng.normal(size=(R, H))
    w1, w3, w2 = rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I))
    y, _ = O.expert_ffn(x, w1, w3, w2)
    for r in range(R):
        h = []
        for i in range(I):
            g = sum(w1[i, j] * x[r, j] for j in range(H))
            u = sum(w3[i, j] * x[r, j] for j in range(H))
            h.append(g / (1 + math.exp(-g)) * u)
        for n in range(H):
            assert abs(y[r, n] - sum(w2[n, i] * h[i] for i in range(I))) < 1e-12


def test_single_nonzero_weight_closed_form():
    H, I = 64, 64
    # build dense matrices with a single nonzero entry and check the layer maths
    x = np.zeros((1, H))
    x[0, 5], x[0, 9] = 1.5, -2.0
    w1 = np.zeros((I, H)); w1[3, 5] = 0.75
    w3 = np.zeros((I, H)); w3[3, 9] = 0.5
    w2 = np.zeros((H, I)); w2[7, 3] = -1.25
    y, h = O.expert_ffn(x, w1, w3, w2)
    g = 0.75 * 1.5
    u = 0.5 * -2.0
    want = -1.25 * (g / (1 + math.exp(-g))) * u
    assert abs(y[0, 7] - want) < 1e-15
    y[0, 7] = 0.0
    assert not y.any()


def _layer(seed, fmts, m=2, k=2, bias_std=0.0, H=256, I=256):
    E = len(fmts) - 1
    return synth.small_layer(seed, fmts, H, I, E, k, m, bias_std)


def test_zero_experts_give_shared_only():
    L = _layer(5, [synth.Q2_0] * 5)
    # zero out every routed expert: d = 0 in every block
    for e in range(4):
        blk = L["experts"][e].reshape(-1, 18).copy()
        blk[:, 16:] = 0
        L["experts"][e] = blk.reshape(-1)
    r = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 256, 256, 2, 4)
    x = O.bf16_bits_to_f64(L["x"])
    w1, w3, w2 = F.dequant_expert(synth.Q2_0, L["experts"][4], 256, 256)
    ys, _ = O.expert_ffn(x, w1, w3, w2)
    assert np.allclose(r["out"], ys, rtol=1e-13, atol=1e-15)


def test_k1_equals_single_expert_plus_shared():
    L = _layer(6, [synth.MXFP4, synth.TQ1, synth.Q3_K, synth.Q2_0], m=3, k=1)
    r = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 256, 256, 1, 3)
    x = O.bf16_bits_to_f64(L["x"])
    assert np.allclose(r["w"], 1.0)
    for m in range(3):
        e = int(r["idx"][m, 0])
        ye, _ = O.expert_ffn(x[m:m + 1], *F.dequant_expert(int(L["fmts"][e]), L["experts"][e], 256, 256))
        ys, _ = O.expert_ffn(x[m:m + 1], *F.dequant_expert(int(L["fmts"][3]), L["experts"][3], 256, 256))
        assert np.allclose(r["out"][m], ye[0] + ys[0], rtol=1e-14, atol=1e-14)


def test_layer_rows_independent():
    L = _layer(7, [synth.Q2_0, synth.TQ1, synth.Q3_K, synth.MXFP4, synth.Q2_0], m=4, k=2, bias_std=0.25)
    full = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 256, 256, 2, 4)
    for m in range(4):
        one = O.moe_layer(L["x"][m:m + 1], L["router"], L["bias"], L["experts"], L["fmts"], 256, 256, 2, 4)
        assert np.array_equal(one["idx"][0], full["idx"][m])
        assert np.allclose(one["out"][0], full["out"][m], rtol=1e-13, atol=1e-13)


def test_rmsnorm_constant_vector():
    r = np.full((2, 64), 3.0)
    r[1] = -0.25
    t = O.rmsnorm_to_bf16(r)
    assert np.all(t[0] == t[0, 0]) and np.all(t[1] == t[1, 0])
    v0 = O.bf16_bits_to_f64(t[0, :1])[0]
    v1 = O.bf16_bits_to_f64(t[1, :1])[0]
    assert abs(v0 - 3.0 / math.sqrt(9.0 + 1e-6)) <= 2 ** -8
    assert abs(v1 + 0.25 / math.sqrt(0.0625 + 1e-6)) <= 2 ** -8
    assert v0 <= 1.0 and v1 >= -1.0


def test_round_to_bf16_exhaustive_neighbourhood():
    # every bf16 value in a range and the midpoints between neighbours
    bits = np.arange(0x3F00, 0x4100, dtype=np.uint32)
    vals = (bits << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(O.round_to_bf16(vals), bits.astype(np.uint16))
    mids = (vals[:-1] + vals[1:]) / 2
    got = O.round_to_bf16(mids)
    even = np.where(bits[:-1] % 2 == 0, bits[:-1], bits[1:])
    assert np.array_equal(got, even.astype(np.uint16))
    assert np.array_equal(O.round_to_bf16(-vals), (bits | 0x8000).astype(np.uint16))


def test_prefill_permutation_is_bijection():
    rng = np.random.default_rng(8)
    idx = np.stack([rng.choice(12, 3, replace=False) for _ in range(40)])
    counts, offsets, pairs = O.prefill_permutation(idx, 12)
    assert counts.sum() == 120 and offsets[-1] == 120
    seen = set(map(tuple, pairs.tolist()))
    assert len(seen) == 120
    for e in range(12):
        toks = pairs[offsets[e]:offsets[e + 1], 0]
        assert np.all(np.diff(toks) > 0)
        for t, j in pairs[offsets[e]:offsets[e + 1]]:
            assert idx[t, j] == e


def test_prefill_rows_equal_decode():
    L = _layer(9, [synth.Q2_0, synth.TQ1, synth.Q3_K, synth.MXFP4, synth.Q2_0], m=6, k=2)
    rows = [0, 3, 5]
    p = O.prefill_rows(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 256, 256, 2, 4, None, rows)
    d = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 256, 256, 2, 4)
    assert np.allclose(p["out_rows"], d["out"][rows], rtol=1e-13, atol=1e-15)


def test_expert_bytes_streamed():
    fm = np.array([synth.MXFP4] * 7)
    idx = np.array([[0, 1, 2, 3, 4, 5]])
    assert O.expert_bytes_streamed(idx, fm, 5120, 2304, 6) == 7 * 18_800_640
    idx2 = np.array([[0, 1], [1, 2]])
    assert O.expert_bytes_streamed(idx2, np.array([synth.TQ1, synth.Q2_0, synth.Q3_K, synth.Q2_0]),
                                   5120, 2304, 3) == 7_741_440 + 2 * 9_953_280 + 15_206_400


# ------------------------------------------------ planted mistakes are caught

def test_planted_nibble_swap_is_caught(monkeypatch):
    def swapped(blocks):
        b = blocks.astype(np.int64)
        c = b[..., :16]
        nib = np.stack([(c >> 4) & 0xF, c & 0xF], axis=-1).reshape(*b.shape[:-1], 32)
        return F.e2m1_to_f64(nib) * F.ue8m0_to_f64(b[..., 16])[..., None]
    blk, vals = read_golden("mxfp4.txt")[0]
    assert not same_bits(swapped(blk[None])[0], vals)


def test_planted_q2_offset_is_caught():
    blk, vals = read_golden("q2_0.txt")[0]
    b = blk.astype(np.int64)
    j = np.arange(64)
    q = (b[j // 4] >> (2 * (j % 4))) & 3
    wrong = 1.0 * (2 * q - 2)  # dropped term: -2 instead of -3
    assert not same_bits(wrong, vals)


def test_planted_digit_order_is_caught():
    blk, vals = read_golden("tq1.txt")[0]
    v = blk[:51].astype(np.int64)
    msd_first = np.stack([(v // 3 ** (4 - r)) % 3 for r in range(5)], axis=-1).reshape(-1) - 1.0
    assert not same_bits(np.concatenate([msd_first, [1.0]]), vals)


def test_planted_bias_in_weights_is_caught():
    rng = np.random.default_rng(10)
    x = rng.normal(size=(1, 8))
    wr = rng.normal(size=(6, 8))
    b = rng.normal(size=6)
    r = O.route(x, wr, b, 2)
    key = r["key"][0, r["idx"][0]]
    assert not np.allclose(r["w"][0], key / key.sum())


# ------------------------------------------- layer combine and chain, brute force
#
# These pins restate the layer with plain Python loops over scalars (no call
# into oracle.moe): the weighted combine with k >= 2 and a non-zero bias, the
# RMS normalisation on a vector whose mean |r| differs from its RMS, and a
# two-layer residual chain.  bf16 rounding here goes through torch's own
# conversion (binary64 -> binary32 -> bfloat16, round to nearest even), not
# the oracle's integer rounding.  The planted-mistake tests below run
# mutated oracle functions (monkeypatched into oracle.moe) through these same
# pins and require each one to fail.

import struct

import torch


def _bf16_to_float(b):
    return struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]


def _float_to_bf16_bits(v):
    t = torch.tensor([float(np.float32(v))], dtype=torch.float32).to(torch.bfloat16)
    return int(t.view(torch.int16).item()) & 0xFFFF


def _brute_layer(x_bits, router, bias, experts, fmts, H, I, k, shared):
    """out[m] = y_shared(x_m) + sum_j s_j / (sum s) y_j(x_m), scalar loops."""
    E = router.shape[0]
    dense = {}

    def weights(e):
        if e not in dense:
            dense[e] = [m.tolist() for m in F.dequant_expert(int(fmts[e]), experts[e], H, I)]
        return dense[e]

    def ffn(e, xv):
        w1, w3, w2 = weights(e)
        h = []
        for i in range(I):
            g = 0.0
            u = 0.0
            for j in range(H):
                g += w1[i][j] * xv[j]
                u += w3[i][j] * xv[j]
            h.append(g / (1.0 + math.exp(-g)) * u)
        return [sum(w2[n][i] * h[i] for i in range(I)) for n in range(H)]

    outs = []
    for row in x_bits:
        xv = [_bf16_to_float(b) for b in row]
        s = []
        for e in range(E):
            z = 0.0
            for j in range(H):
                z += float(router[e][j]) * xv[j]
            s.append(1.0 / (1.0 + math.exp(-z)))
        key = [s[e] + float(bias[e]) for e in range(E)]
        chosen = sorted(range(E), key=lambda e: (-key[e], e))[:k]
        tot = sum(s[e] for e in chosen)
        out = ffn(shared, xv)
        for e in chosen:
            y = ffn(e, xv)
            for n in range(H):
                out[n] += s[e] / tot * y[n]
        outs.append(out)
    return np.array(outs)


def _combine_case(k):
    # 5 routed experts + shared, H = I = 64 (Q2_0 and MXFP4 blocks divide 64)
    fmts = [synth.Q2_0, synth.MXFP4, synth.Q2_0, synth.MXFP4, synth.Q2_0, synth.MXFP4]
    return synth.small_layer(20 + k, fmts, 64, 64, 5, k, 2, bias_std=0.25)


def pin_combine(k):
    L = _combine_case(k)
    got = O.moe_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 64, 64, k, 5)["out"]
    want = _brute_layer(L["x"], L["router"], L["bias"], L["experts"], L["fmts"], 64, 64, k, 5)
    assert np.allclose(got, want, rtol=1e-11, atol=1e-12), np.abs(got - want).max()


def pin_rmsnorm_nonconstant():
    # r = (3, 4, 0, 0): mean r^2 = 6.25, rms = sqrt(6.25 + 1e-6); mean |r| = 1.75
    r = np.array([[3.0, 4.0, 0.0, 0.0], [-6.0, 0.0, 8.0, 0.0]])
    t = O.rmsnorm_to_bf16(r)
    rms = [math.sqrt(6.25 + 1e-6), math.sqrt(25.0 + 1e-6)]
    for m in range(2):
        for j in range(4):
            assert t[m, j] == _float_to_bf16_bits(r[m, j] / rms[m]), (m, j, t[m, j])
    # closed form of the first row: 3 / 2.5 -> bf16 1.203125, 4 / 2.5 -> bf16 1.6015625
    assert _bf16_to_float(t[0, 0]) == 1.203125 and _bf16_to_float(t[0, 1]) == 1.6015625


def pin_chain():
    H = I = 64
    fmts = [synth.MXFP4, synth.Q2_0, synth.MXFP4, synth.Q2_0, synth.Q2_0]
    layers = []
    for l in range(2):
        L = synth.small_layer(40 + l, fmts, H, I, 4, 2, 2, bias_std=0.25)
        layers.append(dict(router=L["router"], bias=L["bias"], experts=L["experts"], fmts=L["fmts"],
                           shared=4))
    x_bits = synth.small_layer(50, fmts, H, I, 4, 2, 2)["x"]
    got = O.moe_chain(x_bits, layers, H, I, 2)
    r = [[_bf16_to_float(b) for b in row] for row in x_bits]
    for l, L in enumerate(layers):
        t = []
        for row in r:
            rms = math.sqrt(sum(v * v for v in row) / H + 1e-6)
            t.append([_float_to_bf16_bits(v / rms) for v in row])
        t = np.array(t, dtype=np.uint16)
        assert np.array_equal(t, got["ts"][l]), l
        out = _brute_layer(t, L["router"], L["bias"], L["experts"], L["fmts"], H, I, 2, 4)
        assert np.allclose(out, got["outs"][l], rtol=1e-11, atol=1e-12), l
        r = [[r[m][n] + out[m][n] for n in range(H)] for m in range(len(r))]
    assert np.allclose(np.array(r), got["resid"], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("k", [2, 3])
def test_weighted_combine_brute_force(k):
    pin_combine(k)


def test_rmsnorm_nonconstant_closed_form():
    pin_rmsnorm_nonconstant()


def test_two_layer_chain_brute_force():
    pin_chain()


# planted mistakes, each run through the oracle and caught by a named pin

def _route_with(w_of):
    real = O.route

    def mutated(x, router_w, sel_bias, top_k, forced_idx=None):
        r = real(x, router_w, sel_bias, top_k, forced_idx)
        r["w"] = w_of(r)
        return r
    return mutated


def test_planted_dropped_mixing_weight_fails_combine_pin(monkeypatch):
    monkeypatch.setattr(O, "route", _route_with(lambda r: np.ones_like(r["w"])))
    with pytest.raises(AssertionError):
        pin_combine(2)


def test_planted_biased_key_weights_fail_combine_pin(monkeypatch):
    def biased(r):
        kk = np.take_along_axis(r["key"], r["idx"], axis=1)
        return kk / kk.sum(axis=1, keepdims=True)
    monkeypatch.setattr(O, "route", _route_with(biased))
    with pytest.raises(AssertionError):
        pin_combine(3)


def test_planted_mean_abs_norm_fails_norm_and_chain_pins(monkeypatch):
    def mean_abs(resid):
        rr = np.asarray(resid, dtype=np.float64)
        return O.round_to_bf16(rr / (np.mean(np.abs(rr), axis=-1, keepdims=True) + O.RMS_EPS))
    monkeypatch.setattr(O, "rmsnorm_to_bf16", mean_abs)
    with pytest.raises(AssertionError):
        pin_rmsnorm_nonconstant()
    with pytest.raises(AssertionError):
        pin_chain()


def test_planted_transposed_w2_fails_combine_pin(monkeypatch):
    def transposed(x, w1, w3, w2):
        g = x @ w1.T
        u = x @ w3.T
        h = O.silu(g) * u
        return h @ w2, h  # W2 applied transposed (square at H = I)
    monkeypatch.setattr(O, "expert_ffn", transposed)
    with pytest.raises(AssertionError):
        pin_combine(2)


def test_planted_silu_sign_fails_combine_pin(monkeypatch):
    monkeypatch.setattr(O, "silu", lambda t: t / (1.0 + np.exp(t)))
    with pytest.raises(AssertionError):
        pin_combine(2)

"""Pins for the oracle's block decoder and encoder.

Decoder: hand-built blocks whose weights are known in closed form (literal bytes for the 32- and 64-weight
types; blocks assembled field by field for the K-quants), plus random valid fields packed by the tests' own
field writer (tests/spec_fields.py, written from the specification's layout tables, independently of the
oracle's C) and compared exactly as rationals.

Encoder: round-trip bound of the specification's section 4 on several weight distributions, read back with
the tests' own field reader; codes and sub-scales in range; literal blocks whose scale and codes follow from
the section's rules by hand.
"""
import zlib
from fractions import Fraction

import numpy as np
import pytest

import spec_fields as sf

QTYPES = ["Q4_0", "Q4_1", "Q5_0", "Q5_1", "Q8_0", "Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K", "A4G64"]


def _decode(orc, qtype, blk):
    qk = sf.QK[qtype]
    return orc.dequant_f64(qtype, np.frombuffer(blk, dtype=np.uint8).copy(), 1, qk)[0]


# ---------------------------------------------------------------- literal hand-built blocks

def test_q4_0_literal(orc):
    # d = 1.0 (0x3C00); byte j holds element j (low nibble) = j and element j+16 (high) = 15 - j
    blk = bytes.fromhex("003c" + "f0e1d2c3b4a5968778695a4b3c2d1e0f")
    want = [j - 8 for j in range(16)] + [7 - j for j in range(16)]
    assert list(_decode(orc, "Q4_0", blk)) == want


def test_q4_0_negative_scale(orc):
    # d = -0.5 (0xB800); all codes 9 -> each weight -0.5
    blk = bytes.fromhex("00b8" + "99" * 16)
    assert list(_decode(orc, "Q4_0", blk)) == [-0.5] * 32


def test_q8_0_literal(orc):
    # d = 0.25 (0x3400); int8 codes 0, 1, -1, 127, -128, then zeros
    blk = bytes.fromhex("0034" + "00" + "01" + "ff" + "7f" + "80" + "00" * 27)
    want = [0, 0.25, -0.25, 31.75, -32.0] + [0] * 27
    assert list(_decode(orc, "Q8_0", blk)) == want


def test_q4_1_literal(orc):
    # d = 0.5 (0x3800), m = -2 (0xC000); element j = j, element j+16 = 15-j
    blk = bytes.fromhex("0038" + "00c0" + "f0e1d2c3b4a5968778695a4b3c2d1e0f")
    want = [0.5 * j - 2 for j in range(16)] + [0.5 * (15 - j) - 2 for j in range(16)]
    assert list(_decode(orc, "Q4_1", blk)) == want


def test_q5_0_literal(orc):
    # d = 1.0; qh = 0xAAAAAAAA (high bit on odd elements); nibbles as in the Q4_0 case
    blk = bytes.fromhex("003c" + "aaaaaaaa" + "f0e1d2c3b4a5968778695a4b3c2d1e0f")
    low = list(range(16)) + [15 - j for j in range(16)]
    want = [low[i] + 16 * (i % 2) - 16 for i in range(32)]
    assert list(_decode(orc, "Q5_0", blk)) == want


def test_q5_1_literal(orc):
    # d = 2.0 (0x4000), m = 1.0 (0x3C00); qh = 0x0000FFFF: high bit on elements 0..15
    blk = bytes.fromhex("0040" + "003c" + "ffff0000" + "f0e1d2c3b4a5968778695a4b3c2d1e0f")
    low = list(range(16)) + [15 - j for j in range(16)]
    want = [2.0 * (low[i] + (16 if i < 16 else 0)) + 1.0 for i in range(32)]
    assert list(_decode(orc, "Q5_1", blk)) == want


def test_a4g64_literal(orc):
    # s = 0.5 (bf16 0x3F00), b = -1.0 (bf16 0xBF80); byte j: low = j % 16, high = 15 - j % 16
    qs = bytes(((j % 16) | ((15 - j % 16) << 4)) for j in range(32))
    blk = bytes.fromhex("003f" + "80bf") + qs
    want = [0.5 * (i % 16) - 1.0 for i in range(32)] + [0.5 * (15 - (i - 32) % 16) - 1.0 for i in range(32, 64)]
    assert list(_decode(orc, "A4G64", blk)) == want


# ---------------------------------------------------------------- K-quant blocks assembled field by field

def _code(i, levels):
    """A code pattern with no period that divides the layouts' strides (32, 64, 128), so that a swapped
    nibble, bit plane or half-block changes the decoded weights."""
    return ((i * 7) // 3 + i // 11 + (i // 64) * 5) % levels


def test_q2_k_closed_form(orc):
    # d = 1, dmin = 0.5, sc_s = s, mn_s = 15 - s
    q = [_code(i, 4) for i in range(256)]
    f = {"d": sf.h16(1.0), "dmin": sf.h16(0.5), "sc": list(range(16)), "mn": [15 - s for s in range(16)], "q": q}
    want = [1.0 * (i // 16) * q[i] - 0.5 * (15 - i // 16) for i in range(256)]
    assert list(_decode(orc, "Q2_K", sf.pack("Q2_K", f))) == want


def test_q3_k_closed_form(orc):
    # d = 0.25; stored sub-scale 32 + s - 8 (signed s - 8)
    q = [_code(i, 8) for i in range(256)]
    f = {"d": sf.h16(0.25), "sc": [32 + s - 8 for s in range(16)], "q": q}
    want = [0.25 * ((i // 16) - 8) * (q[i] - 4) for i in range(256)]
    assert list(_decode(orc, "Q3_K", sf.pack("Q3_K", f))) == want


@pytest.mark.parametrize("qtype", ["Q4_K", "Q5_K"])
def test_q45_k_closed_form(orc, qtype):
    # d = 0.125, dmin = 2; sc_s = 7 * s + 1, mn_s = 63 - 5 * s
    lv = 16 if qtype == "Q4_K" else 32
    q = [_code(i, lv) for i in range(256)]
    f = {"d": sf.h16(0.125), "dmin": sf.h16(2.0), "sc": [7 * s + 1 for s in range(8)],
         "mn": [63 - 5 * s for s in range(8)], "q": q}
    want = [0.125 * (7 * (i // 32) + 1) * q[i] - 2.0 * (63 - 5 * (i // 32)) for i in range(256)]
    assert list(_decode(orc, qtype, sf.pack(qtype, f))) == want


def test_q6_k_closed_form(orc):
    # d = 1/64; signed sub-scale 17 * s - 128
    q = [_code(i, 64) for i in range(256)]
    f = {"d": sf.h16(1 / 64), "sc": [17 * s - 128 for s in range(16)], "q": q}
    want = [(1 / 64) * (17 * (i // 16) - 128) * (q[i] - 32) for i in range(256)]
    assert list(_decode(orc, "Q6_K", sf.pack("Q6_K", f))) == want


# ---------------------------------------------------------------- random fields, exact comparison

@pytest.mark.parametrize("qtype", QTYPES)
def test_decode_random_fields_exact(orc, qtype):
    g = np.random.default_rng(sf.QK[qtype] + len(qtype))
    blocks, want = [], []
    for _ in range(24):
        f = sf.random_fields(qtype, g)
        blocks.append(sf.pack(qtype, f))
        want.append(sf.values(qtype, f))
    nb = len(blocks)
    wq = np.frombuffer(b"".join(blocks), dtype=np.uint8).copy()
    K = sf.QK[qtype] * nb
    got = orc.dequant_f64(qtype, wq, 1, K)[0]
    flat = [v for blk in want for v in blk]
    assert all(Fraction(float(a)) == b for a, b in zip(got, flat))
    # the binary32 rule: one rounding of the exact value
    got32 = orc.dequant_f32(qtype, wq, 1, K)[0]
    assert np.array_equal(got32, np.array([np.float32(float(v)) for v in flat], dtype=np.float32))


@pytest.mark.parametrize("qtype", ["F32", "F16", "BF16"])
def test_plain_types_roundtrip(orc, qtype):
    g = np.random.default_rng(5)
    w = (g.standard_normal((3, 40)) * 0.02).astype(np.float32)
    wq = orc.quantize(qtype, w)
    back = orc.dequant_f64(qtype, wq, 3, 40)
    if qtype == "F32":
        want = w.astype(np.float64)
    elif qtype == "F16":
        want = w.astype(np.float16).astype(np.float64)
    else:
        import torch
        want = torch.from_numpy(w).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(back, want)


# ---------------------------------------------------------------- encoder: round-trip bound

def _dist(kind, g, n):
    if kind == "normal":
        return (0.02 * g.standard_normal(n)).astype(np.float32)
    if kind == "uniform":
        return g.uniform(-1, 1, n).astype(np.float32)
    if kind == "positive":
        return g.uniform(0.1, 2.0, n).astype(np.float32)
    if kind == "negative":
        return g.uniform(-3.0, -0.5, n).astype(np.float32)
    if kind == "outliers":
        w = (0.01 * g.standard_normal(n)).astype(np.float32)
        w[g.integers(0, n, n // 50)] *= 40
        return w
    if kind == "sparse":
        w = (0.05 * g.standard_normal(n)).astype(np.float32)
        w[g.random(n) < 0.7] = 0
        return w
    raise ValueError(kind)


def _group_bound(qtype, f, w_grp):
    """Per-element bound |w - w_hat| <= S/2 + |l - L| + T|r - S| of the specification's section 4 (times a
    1 + 2^-20 factor for the binary32 division that picks each code), for one encoded block."""
    w = [Fraction(float(v)) for v in w_grp]
    n = len(w)
    out = []
    if qtype in ("Q4_0", "Q5_0", "Q8_0"):
        T = {"Q4_0": 7, "Q5_0": 15, "Q8_0": 127}[qtype]
        r = max(abs(v) for v in w) / T
        S = sf.val16(f["d"])
        out = [S / 2 + T * abs(r - S)] * n
    elif qtype in ("Q4_1", "Q5_1", "A4G64"):
        T = 31 if qtype == "Q5_1" else 15
        lo, hi = min(w), max(w)
        r = (hi - lo) / T
        if qtype == "A4G64":
            S, L = sf.valb16(f["s"]), sf.valb16(f["b"])
        else:
            S, L = sf.val16(f["d"]), sf.val16(f["m"])
        out = [S / 2 + abs(lo - L) + T * abs(r - S)] * n
    else:
        sub = sf.SUB[qtype]
        for s in range(256 // sub):
            grp = w[s * sub:(s + 1) * sub]
            if qtype in ("Q2_K", "Q4_K", "Q5_K"):
                T = {"Q2_K": 3, "Q4_K": 15, "Q5_K": 31}[qtype]
                l = min(Fraction(0), min(grp))
                r = (max(grp) - l) / T
                S = sf.val16(f["d"]) * f["sc"][s]
                L = -sf.val16(f["dmin"]) * f["mn"][s]
                b = S / 2 + abs(l - L) + T * abs(r - S)
            else:
                T = 3 if qtype == "Q3_K" else 31
                r = max(abs(v) for v in grp) / T
                sc = f["sc"][s] - 32 if qtype == "Q3_K" else f["sc"][s]
                S = sf.val16(f["d"]) * sc
                b = S / 2 + T * abs(r - S)
            out += [b] * sub
    return out


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("kind", ["normal", "uniform", "positive", "negative", "outliers", "sparse"])
def test_encoder_roundtrip_bound(orc, qtype, kind):
    g = np.random.default_rng(zlib.crc32((qtype + kind).encode()))
    qk, nbytes = sf.QK[qtype], sf.BYTES[qtype]
    nblk = max(4, 1024 // qk)
    w = _dist(kind, g, qk * nblk).reshape(1, -1)
    wq = orc.quantize(qtype, w)[0]
    back = orc.dequant_f64(qtype, wq, 1, w.shape[1])[0]
    slack = Fraction(1) + Fraction(1, 2 ** 20)
    for bi in range(nblk):
        blk = wq[bi * nbytes:(bi + 1) * nbytes]
        f = sf.unpack(qtype, blk)
        # codes and sub-scales in their stated ranges
        if qtype == "Q3_K":
            assert all(32 <= s <= 63 for s in f["sc"])
        if qtype == "Q6_K":
            assert all(0 <= s <= 127 for s in f["sc"])
        grp = w[0, bi * qk:(bi + 1) * qk]
        bnd = _group_bound(qtype, f, grp)
        for i in range(qk):
            err = abs(Fraction(float(back[bi * qk + i])) - Fraction(float(grp[i])))
            assert err <= bnd[i] * slack + Fraction(1, 2 ** 60), (qtype, kind, bi, i, float(err), float(bnd[i]))


@pytest.mark.parametrize("qtype", QTYPES)
def test_encoder_zero_block(orc, qtype):
    qk = sf.QK[qtype]
    w = np.zeros((1, qk), dtype=np.float32)
    back = orc.dequant_f64(qtype, orc.quantize(qtype, w), 1, qk)
    assert np.all(back == 0)


@pytest.mark.parametrize("qtype", QTYPES)
def test_encoder_error_scale(orc, qtype):
    """On N(0, 0.02) weights the mean error falls with the code width, as the bits per weight say."""
    g = np.random.default_rng(11)
    w = (0.02 * g.standard_normal((8, 2048))).astype(np.float32)
    back = orc.dequant_f64(qtype, orc.quantize(qtype, w), 8, 2048)
    rel = np.sqrt(np.mean((back - w) ** 2)) / 0.02
    limit = {"Q8_0": 0.01, "Q6_K": 0.02, "Q5_0": 0.06, "Q5_1": 0.05, "Q5_K": 0.06, "Q4_0": 0.12,
             "Q4_1": 0.10, "Q4_K": 0.12, "A4G64": 0.12, "Q3_K": 0.30, "Q2_K": 0.60}[qtype]
    assert rel < limit, rel


# ---------------------------------------------------------------- encoder: literal decisions
# Blocks whose scale and codes follow from the specification's section 4 by hand (every quotient below is
# exact, and the ties go to even), so that a different scale rule (say amax / 8 for Q4_0) or a tie rounded
# away from zero changes the bytes.

def test_encoder_q4_0_literal(orc):
    # amax = 7 -> d = f16(7 / 7) = 1.0 (0x3C00); q = rne(w) + 8 (3.5 -> 4, 2.5 -> 2, -2.5 -> -2, -0.5 -> 0)
    w = np.zeros(32, dtype=np.float32)
    w[:8] = [7.0, -7.0, 3.5, 2.5, 1.5, 0.5, -0.5, -1.5]
    w[16:20] = [-7.0, 6.0, -2.5, 0.25]
    codes = [15, 1, 12, 10, 10, 8, 8, 6] + [8] * 8 + [1, 14, 6, 8] + [8] * 12
    want = bytes([0x00, 0x3C]) + bytes(codes[j] | (codes[j + 16] << 4) for j in range(16))
    assert orc.quantize("Q4_0", w.reshape(1, 32)).tobytes() == want


def test_encoder_q8_0_literal(orc):
    # amax = 127 -> d = f16(127 / 127) = 1.0; q = rne(w): 63.5 -> 64, 62.5 -> 62, -0.5 -> 0
    w = np.zeros(32, dtype=np.float32)
    w[:6] = [127.0, -127.0, 63.5, 62.5, -0.5, 1.25]
    codes = [127, -127, 64, 62, 0, 1] + [0] * 26
    want = bytes([0x00, 0x3C]) + bytes(c & 0xFF for c in codes)
    assert orc.quantize("Q8_0", w.reshape(1, 32)).tobytes() == want


def test_encoder_q4_1_literal(orc):
    # lo = -2, hi = 13 -> d = f16(15 / 15) = 1.0, m = f16(-2) (0xC000); q = rne(w + 2): 0.5 -> 2.5 -> 2,
    # 1.5 -> 3.5 -> 4, -2 -> 0, 13 -> 15
    w = np.full(32, 3.0, dtype=np.float32)
    w[:4] = [-2.0, 13.0, 0.5, 1.5]
    codes = [0, 15, 2, 4] + [5] * 28
    want = bytes([0x00, 0x3C, 0x00, 0xC0]) + bytes(codes[j] | (codes[j + 16] << 4) for j in range(16))
    assert orc.quantize("Q4_1", w.reshape(1, 32)).tobytes() == want

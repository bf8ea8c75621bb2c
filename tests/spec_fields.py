"""Field-level packing and unpacking of the block formats, written in the tests straight from the block
format specification's layout tables (section 2), independently of the oracle's C decoder.

It builds blocks from chosen field values (scales, sub-scales, codes) so that the tests can state the
expected weights in closed form, and reads fields back so that encoder outputs can be checked against
their round-trip bound. Nothing here multiplies weights by activations.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

QK = {"F32": 1, "F16": 1, "BF16": 1, "Q4_0": 32, "Q4_1": 32, "Q5_0": 32, "Q5_1": 32, "Q8_0": 32,
      "Q2_K": 256, "Q3_K": 256, "Q4_K": 256, "Q5_K": 256, "Q6_K": 256, "A4G64": 64}
BYTES = {"F32": 4, "F16": 2, "BF16": 2, "Q4_0": 18, "Q4_1": 20, "Q5_0": 22, "Q5_1": 24, "Q8_0": 34,
         "Q2_K": 84, "Q3_K": 110, "Q4_K": 144, "Q5_K": 176, "Q6_K": 210, "A4G64": 36}
SUB = {"Q2_K": 16, "Q3_K": 16, "Q4_K": 32, "Q5_K": 32, "Q6_K": 16}


def h16(v: float) -> int:
    """binary16 bits of v (v must be representable)."""
    b = int(np.array([v], dtype=np.float16).view(np.uint16)[0])
    assert float(np.uint16(b).view(np.float16)) == v, v
    return b


def hb16(v: float) -> int:
    """bfloat16 bits of v (v must be representable)."""
    b = int(np.array([v], dtype=np.float32).view(np.uint32)[0]) >> 16
    assert np.uint32(b << 16).view(np.float32) == np.float32(v), v
    return b


def val16(bits: int) -> Fraction:
    return Fraction(float(np.uint16(bits).view(np.float16)))


def valb16(bits: int) -> Fraction:
    return Fraction(float(np.uint32(bits << 16).view(np.float32)))


def _put16(b: bytearray, off: int, v: int):
    b[off] = v & 255
    b[off + 1] = (v >> 8) & 255


def _get16(b, off: int) -> int:
    return b[off] | (b[off + 1] << 8)


def _put_bits(b: bytearray, off: int, pos: int, width: int, v: int):
    for t in range(width):
        p = pos + t
        if (v >> t) & 1:
            b[off + p // 8] |= 1 << (p % 8)
        else:
            b[off + p // 8] &= ~(1 << (p % 8)) & 255


def _get_bits(b, off: int, pos: int, width: int) -> int:
    v = 0
    for t in range(width):
        p = pos + t
        v |= ((b[off + p // 8] >> (p % 8)) & 1) << t
    return v


def pack(qtype: str, f: dict) -> bytes:
    """Build one block from fields: 'd', 'm', 'dmin', 's', 'b' (bit patterns), 'sc', 'mn' (lists of
    sub-block integers) and 'q' (list of per-element codes, unsigned as stored)."""
    b = bytearray(BYTES[qtype])
    q = f.get("q")
    if qtype in ("Q4_0", "Q4_1", "Q5_0", "Q5_1"):
        qs_off = {"Q4_0": 2, "Q4_1": 4, "Q5_0": 6, "Q5_1": 8}[qtype]
        _put16(b, 0, f["d"])
        if qtype in ("Q4_1", "Q5_1"):
            _put16(b, 2, f["m"])
        qh_off = {"Q5_0": 2, "Q5_1": 4}.get(qtype)
        for j in range(16):
            b[qs_off + j] = (q[j] & 15) | ((q[j + 16] & 15) << 4)
        if qh_off is not None:
            H = sum(((q[i] >> 4) & 1) << i for i in range(32))
            for t in range(4):
                b[qh_off + t] = (H >> (8 * t)) & 255
    elif qtype == "Q8_0":
        _put16(b, 0, f["d"])
        for i in range(32):
            b[2 + i] = q[i] & 255
    elif qtype == "A4G64":
        _put16(b, 0, f["s"])
        _put16(b, 2, f["b"])
        for j in range(32):
            b[4 + j] = (q[j] & 15) | ((q[j + 32] & 15) << 4)
    elif qtype == "Q2_K":
        for s in range(16):
            b[s] = f["sc"][s] | (f["mn"][s] << 4)
        for i in range(256):
            h, g, l = i // 128, (i % 128) // 32, i % 32
            b[16 + 32 * h + l] |= (q[i] & 3) << (2 * g)
        _put16(b, 80, f["d"])
        _put16(b, 82, f["dmin"])
    elif qtype == "Q3_K":
        for i in range(256):
            h, g, l = i // 128, (i % 128) // 32, i % 32
            b[32 + 32 * h + l] |= (q[i] & 3) << (2 * g)
            b[i % 32] |= ((q[i] >> 2) & 1) << (i // 32)
        for s in range(16):
            _put_bits(b, 96, 6 * s, 6, f["sc"][s])
        _put16(b, 108, f["d"])
    elif qtype in ("Q4_K", "Q5_K"):
        _put16(b, 0, f["d"])
        _put16(b, 2, f["dmin"])
        for s in range(8):
            _put_bits(b, 4, 6 * s, 6, f["sc"][s])
            _put_bits(b, 4, 48 + 6 * s, 6, f["mn"][s])
        qs_off = 16 if qtype == "Q4_K" else 48
        for i in range(256):
            c, l = i // 64, i % 32
            sh = 0 if (i % 64) < 32 else 4
            b[qs_off + 32 * c + l] |= (q[i] & 15) << sh
            if qtype == "Q5_K":
                b[16 + i % 32] |= ((q[i] >> 4) & 1) << (i // 32)
    elif qtype == "Q6_K":
        for i in range(256):
            h, j = i // 128, i % 128
            b[64 * h + j % 64] |= (q[i] & 15) << (4 * (j // 64))
            b[128 + 32 * h + j % 32] |= ((q[i] >> 4) & 3) << (2 * (j // 32))
        for s in range(16):
            b[192 + s] = f["sc"][s] & 255
        _put16(b, 208, f["d"])
    else:
        raise ValueError(qtype)
    return bytes(b)


def unpack(qtype: str, blk) -> dict:
    """Inverse of pack(): fields and codes of one block."""
    b = bytes(blk)
    out = {}
    if qtype in ("Q4_0", "Q4_1", "Q5_0", "Q5_1"):
        qs_off = {"Q4_0": 2, "Q4_1": 4, "Q5_0": 6, "Q5_1": 8}[qtype]
        out["d"] = _get16(b, 0)
        if qtype in ("Q4_1", "Q5_1"):
            out["m"] = _get16(b, 2)
        q = [b[qs_off + j] & 15 for j in range(16)] + [b[qs_off + j] >> 4 for j in range(16)]
        qh_off = {"Q5_0": 2, "Q5_1": 4}.get(qtype)
        if qh_off is not None:
            H = sum(b[qh_off + t] << (8 * t) for t in range(4))
            q = [q[i] + 16 * ((H >> i) & 1) for i in range(32)]
        out["q"] = q
    elif qtype == "Q8_0":
        out["d"] = _get16(b, 0)
        out["q"] = [int(np.int8(np.uint8(b[2 + i]))) for i in range(32)]
    elif qtype == "A4G64":
        out["s"], out["b"] = _get16(b, 0), _get16(b, 2)
        out["q"] = [b[4 + j] & 15 for j in range(32)] + [b[4 + j] >> 4 for j in range(32)]
    elif qtype == "Q2_K":
        out["sc"] = [b[s] & 15 for s in range(16)]
        out["mn"] = [b[s] >> 4 for s in range(16)]
        out["q"] = [(b[16 + 32 * (i // 128) + i % 32] >> (2 * ((i % 128) // 32))) & 3 for i in range(256)]
        out["d"], out["dmin"] = _get16(b, 80), _get16(b, 82)
    elif qtype == "Q3_K":
        out["sc"] = [_get_bits(b, 96, 6 * s, 6) for s in range(16)]
        out["q"] = [((b[32 + 32 * (i // 128) + i % 32] >> (2 * ((i % 128) // 32))) & 3)
                    + 4 * ((b[i % 32] >> (i // 32)) & 1) for i in range(256)]
        out["d"] = _get16(b, 108)
    elif qtype in ("Q4_K", "Q5_K"):
        out["d"], out["dmin"] = _get16(b, 0), _get16(b, 2)
        out["sc"] = [_get_bits(b, 4, 6 * s, 6) for s in range(8)]
        out["mn"] = [_get_bits(b, 4, 48 + 6 * s, 6) for s in range(8)]
        qs_off = 16 if qtype == "Q4_K" else 48
        q = []
        for i in range(256):
            v = b[qs_off + 32 * (i // 64) + i % 32]
            v = (v & 15) if (i % 64) < 32 else (v >> 4)
            if qtype == "Q5_K":
                v += 16 * ((b[16 + i % 32] >> (i // 32)) & 1)
            q.append(v)
        out["q"] = q
    elif qtype == "Q6_K":
        q = []
        for i in range(256):
            h, j = i // 128, i % 128
            lo = (b[64 * h + j % 64] >> (4 * (j // 64))) & 15
            hi = (b[128 + 32 * h + j % 32] >> (2 * (j // 32))) & 3
            q.append(lo + 16 * hi)
        out["q"] = q
        out["sc"] = [int(np.int8(np.uint8(b[192 + s]))) for s in range(16)]
        out["d"] = _get16(b, 208)
    else:
        raise ValueError(qtype)
    return out


def values(qtype: str, f: dict):
    """Exact weights (Fractions) of a block from its fields: the formulas of the specification's section 1
    table, evaluated on exact rationals."""
    q = f["q"]
    if qtype == "Q4_0":
        return [val16(f["d"]) * (qi - 8) for qi in q]
    if qtype == "Q4_1":
        return [val16(f["d"]) * qi + val16(f["m"]) for qi in q]
    if qtype == "Q5_0":
        return [val16(f["d"]) * (qi - 16) for qi in q]
    if qtype == "Q5_1":
        return [val16(f["d"]) * qi + val16(f["m"]) for qi in q]
    if qtype == "Q8_0":
        return [val16(f["d"]) * qi for qi in q]
    if qtype == "A4G64":
        return [valb16(f["s"]) * qi + valb16(f["b"]) for qi in q]
    sub = SUB[qtype]
    if qtype in ("Q2_K", "Q4_K", "Q5_K"):
        d, dm = val16(f["d"]), val16(f["dmin"])
        return [d * f["sc"][i // sub] * q[i] - dm * f["mn"][i // sub] for i in range(256)]
    if qtype == "Q3_K":
        d = val16(f["d"])
        return [d * (f["sc"][i // sub] - 32) * (q[i] - 4) for i in range(256)]
    if qtype == "Q6_K":
        d = val16(f["d"])
        return [d * f["sc"][i // sub] * (q[i] - 32) for i in range(256)]
    raise ValueError(qtype)


def random_fields(qtype: str, g: np.random.Generator) -> dict:
    """Random valid fields: normal binary16 scales of either sign, every code and sub-scale in range."""
    def rh():
        return h16(float(np.float16(g.choice([-1, 1]) * g.uniform(1e-3, 2.0))))
    if qtype in ("Q4_0", "Q4_1"):
        f = {"d": rh(), "q": list(g.integers(0, 16, 32))}
    elif qtype in ("Q5_0", "Q5_1"):
        f = {"d": rh(), "q": list(g.integers(0, 32, 32))}
    elif qtype == "Q8_0":
        f = {"d": rh(), "q": list(g.integers(-128, 128, 32))}
    elif qtype == "A4G64":
        # bfloat16 patterns: the upper halves of random binary32 values
        f = {"s": int(np.float32(g.uniform(1e-3, 1.0)).view(np.uint32)) >> 16,
             "b": int(np.float32(-g.uniform(0, 1.0)).view(np.uint32)) >> 16,
             "q": list(g.integers(0, 16, 64))}
    elif qtype == "Q2_K":
        f = {"d": rh(), "dmin": rh(), "sc": list(g.integers(0, 16, 16)), "mn": list(g.integers(0, 16, 16)),
             "q": list(g.integers(0, 4, 256))}
    elif qtype == "Q3_K":
        f = {"d": rh(), "sc": list(g.integers(0, 64, 16)), "q": list(g.integers(0, 8, 256))}
    elif qtype in ("Q4_K", "Q5_K"):
        f = {"d": rh(), "dmin": rh(), "sc": list(g.integers(0, 64, 8)), "mn": list(g.integers(0, 64, 8)),
             "q": list(g.integers(0, 16 if qtype == "Q4_K" else 32, 256))}
    elif qtype == "Q6_K":
        f = {"d": rh(), "sc": list(g.integers(-128, 128, 16)), "q": list(g.integers(0, 64, 256))}
    else:
        raise ValueError(qtype)
    if qtype in ("Q4_1", "Q5_1"):
        f["m"] = rh()
    f["q"] = [int(v) for v in f["q"]]
    for k in ("sc", "mn"):
        if k in f:
            f[k] = [int(v) for v in f[k]]
    return f

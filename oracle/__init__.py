"""CPU oracle for the block-quantized weight matmul (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import this
package. The product library never loads it, and it never loads the product library: the two share no
code, header or table (see ``oracle.c`` for the full statement of what is computed and from which
passages).

This module is a thin ctypes wrapper around ``liboracle.so`` built from ``oracle.c`` with gcc (``build()``);
all arithmetic lives in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

TYPES = ["F32", "F16", "BF16", "Q4_0", "Q4_1", "Q5_0", "Q5_1", "Q8_0",
         "Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K", "A4G64"]
TYPE_ID = {n: i for i, n in enumerate(TYPES)}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (OpenMP if the compiler has it). Returns the library path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f64.restype = ctypes.c_double
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_f16.restype = ctypes.c_uint16
        lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_type_info.argtypes = [I, ctypes.POINTER(I), ctypes.POINTER(I)]
        lib.orc_num_threads.restype = I
        lib.orc_quantize.argtypes = [I, P, I64, I64, P]
        lib.orc_dequant_f64.argtypes = [I, P, I64, I64, P]
        lib.orc_dequant_f32.argtypes = [I, P, I64, I64, P]
        lib.orc_qmm.argtypes = [I, I, P, I64, I64, P, I64, P, P]
        lib.orc_matmul_f64.argtypes = [P, I64, I64, I, P, I64, P, P]
        lib.orc_qmm_sampled.argtypes = [I, I, P, I64, I64, P, I64, I64, P, P, P, P]
        lib.orc_qmm_id.argtypes = [I, I, P, I64, I64, I64, P, P, I64, I, P, P]
        lib.orc_qmm_id_slots.argtypes = [I, I, P, I64, I64, I64, P, P, I64, I, P, P]
        for f in ("orc_type_info", "orc_quantize", "orc_dequant_f64", "orc_dequant_f32", "orc_qmm",
                  "orc_qmm_sampled", "orc_qmm_id", "orc_qmm_id_slots", "orc_matmul_f64"):
            getattr(lib, f).restype = I
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _qt(qtype) -> int:
    return TYPE_ID[qtype] if isinstance(qtype, str) else int(qtype)


def num_threads() -> int:
    return _load().orc_num_threads()


def type_info(qtype):
    """(weights per block, bytes per block)."""
    qk, nb = ctypes.c_int(), ctypes.c_int()
    if _load().orc_type_info(_qt(qtype), ctypes.byref(qk), ctypes.byref(nb)) != 0:
        raise ValueError("bad qtype %r" % (qtype,))
    return qk.value, nb.value


def row_bytes(qtype, K: int) -> int:
    qk, nb = type_info(qtype)
    return (K // qk) * nb


def f16_to_f64(h: int) -> float:
    return _load().orc_f16_to_f64(int(h) & 0xFFFF)


def bf16_to_f64(h: int) -> float:
    return _load().orc_bf16_to_f64(int(h) & 0xFFFF)


def f32_to_f16(v) -> int:
    return _load().orc_f32_to_f16(float(np.float32(v)))


def f32_to_bf16(v) -> int:
    return _load().orc_f32_to_bf16(float(np.float32(v)))


def quantize(qtype, w: np.ndarray) -> np.ndarray:
    """Encode an (N, K) float32 matrix; returns (N, row_bytes) uint8."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    out = np.zeros((N, row_bytes(qtype, K)), dtype=np.uint8)
    if _load().orc_quantize(_qt(qtype), _ptr(w), N, K, _ptr(out)) != 0:
        raise ValueError("quantize: K=%d not a multiple of the block size" % K)
    return out


def dequant_f64(qtype, wq: np.ndarray, N: int, K: int) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    assert wq.size == N * row_bytes(qtype, K)
    out = np.empty((N, K), dtype=np.float64)
    if _load().orc_dequant_f64(_qt(qtype), _ptr(wq), N, K, _ptr(out)) != 0:
        raise ValueError("dequant: bad arguments")
    return out


def dequant_f32(qtype, wq: np.ndarray, N: int, K: int) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    assert wq.size == N * row_bytes(qtype, K)
    out = np.empty((N, K), dtype=np.float32)
    if _load().orc_dequant_f32(_qt(qtype), _ptr(wq), N, K, _ptr(out)) != 0:
        raise ValueError("dequant: bad arguments")
    return out


def _x_arg(x: np.ndarray):
    """Activations: float32, or bfloat16 bit patterns given as uint16."""
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), 1
    return np.ascontiguousarray(x, dtype=np.float32), 0


def qmm(qtype, wq: np.ndarray, N: int, K: int, x: np.ndarray):
    """(y, bound): y[m,n] = sum_k w[n,k] x[m,k] in binary64; bound = sum_k |w x|. Shapes (M, N)."""
    x, xb = _x_arg(x)
    M = x.shape[0]
    assert x.shape == (M, K)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    y = np.empty((M, N), dtype=np.float64)
    bnd = np.empty((M, N), dtype=np.float64)
    if _load().orc_qmm(_qt(qtype), xb, _ptr(wq), N, K, _ptr(x), M, _ptr(y), _ptr(bnd)) != 0:
        raise ValueError("qmm: bad arguments or out of memory")
    return y, bnd


def matmul_f64(w: np.ndarray, x: np.ndarray):
    """The product step alone on an (N, K) binary64 matrix of decoded weights (e.g. dequant_f64's):
    (y, bound) as qmm() returns them."""
    x, xb = _x_arg(x)
    w = np.ascontiguousarray(w, dtype=np.float64)
    N, K = w.shape
    M = x.shape[0]
    assert x.shape == (M, K)
    y = np.empty((M, N), dtype=np.float64)
    bnd = np.empty((M, N), dtype=np.float64)
    if _load().orc_matmul_f64(_ptr(w), N, K, xb, _ptr(x), M, _ptr(y), _ptr(bnd)) != 0:
        raise ValueError("matmul_f64: out of memory")
    return y, bnd


def qmm_sampled(qtype, wq: np.ndarray, N: int, K: int, x: np.ndarray, ms, ns):
    """The same sums for the listed (m, n) pairs only."""
    x, xb = _x_arg(x)
    M = x.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    y = np.empty(ms.size, dtype=np.float64)
    bnd = np.empty(ms.size, dtype=np.float64)
    if _load().orc_qmm_sampled(_qt(qtype), xb, _ptr(wq), N, K, _ptr(x), M, ms.size, _ptr(ms), _ptr(ns),
                               _ptr(y), _ptr(bnd)) != 0:
        raise ValueError("qmm_sampled: bad arguments")
    return y, bnd


def qmm_id(qtype, wqs, N: int, K: int, x: np.ndarray, ids: np.ndarray):
    """Expert-indexed product. wqs: list of E (N, row_bytes) uint8 arrays; x is (M, K), one row per token
    shared by its slots, or (M, topk, K), one row per (token, slot). Returns (y, bound) of shape
    (M, topk, N)."""
    per_slot = x.ndim == 3
    x, xb = _x_arg(x)
    M = x.shape[0]
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    topk = ids.shape[1]
    assert x.shape == ((M, topk, K) if per_slot else (M, K))
    wqs = [np.ascontiguousarray(w, dtype=np.uint8) for w in wqs]
    ptrs = (ctypes.c_void_p * len(wqs))(*[w.ctypes.data for w in wqs])
    y = np.empty((M, topk, N), dtype=np.float64)
    bnd = np.empty((M, topk, N), dtype=np.float64)
    fn = _load().orc_qmm_id_slots if per_slot else _load().orc_qmm_id
    rc = fn(_qt(qtype), xb, ctypes.cast(ptrs, ctypes.c_void_p), len(wqs), N, K, _ptr(x), _ptr(ids), M, topk,
            _ptr(y), _ptr(bnd))
    if rc != 0:
        raise ValueError("qmm_id: bad arguments")
    return y, bnd

"""Python binding of libqmm, the block-quantized weight matmul for GB300 (sm_103a).

Argument marshalling only: every function takes torch tensors (device memory owned by the caller),
passes their pointers and the current CUDA stream to the C-ABI function of the same name (declared in
include/qmm.h), and raises QmmError on a non-zero return code. All computation happens in the library's
CUDA kernels; there is no other code path. If libqmm.so has not been built (``build()``), every call
raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["QmmError", "TYPES", "TYPE_ID", "X_BF16", "X_PER_SLOT", "W_STATIC", "build", "lib", "qmm", "qmm_ws", "qmm_batch", "qmm_workspace_size",
           "qmm_launch_count", "qmm_plan_info", "qmm_noalloc", "NOALLOC_SCRATCH_BYTES",
           "qmm_id", "qmm_id_with_path", "qmm_id_pick_path", "qmm_with_tile", "qmm_pick_tile", "qmm_pick_path", "qmm_dequant", "qmm_quantize",
           "qmm_type_info", "qmm_get_status", "qmm_debug_stall", "qmm_strerror", "row_bytes", "EXPORTS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmm.so")

TYPES = ["F32", "F16", "BF16", "Q4_0", "Q4_1", "Q5_0", "Q5_1", "Q8_0",
         "Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K", "A4G64"]
TYPE_ID = {n: i for i, n in enumerate(TYPES)}
X_BF16 = 0x100
X_PER_SLOT = 0x200
W_STATIC = 0x400      # the kernel launched just before the call does not write the weights
STATUS_BAD_ID, STATUS_TIMEOUT = 0x1, 0x2

# Every symbol include/qmm.h declares.
EXPORTS = ["qmm", "qmm_ws", "qmm_workspace_size", "qmm_noalloc", "qmm_batch", "qmm_id", "qmm_id_with_path", "qmm_id_pick_path",
           "qmm_with_tile", "qmm_pick_tile",
           "qmm_pick_path", "qmm_launch_count", "qmm_plan_info", "qmm_dequant", "qmm_quantize", "qmm_type_info", "qmm_get_status",
           "qmm_debug_stall", "qmm_strerror"]
NOALLOC_SCRATCH_BYTES = 64 << 20   # QMM_NOALLOC_SCRATCH_BYTES


class QmmError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s failed: %s (%d)" % (what, qmm_strerror(code), code))
        self.code = code


def build(force: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force)


_lib = None


def lib():
    """The loaded libqmm (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libqmm.so is not built: run weight_quantized_matmul_fly_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sig = {
            "qmm": ([P, I, I64, I64, P, I64, P, P], I),
            "qmm_ws": ([P, I, I64, I64, P, I64, P, P, SZ, P], I),
            "qmm_noalloc": ([P, I, I64, I64, P, I64, P, P], I),
            "qmm_batch": ([I, P, P, P, I, I64, P, I64, P], I),
            "qmm_workspace_size": ([I, I64, I64, I64], SZ),
            "qmm_id": ([P, I64, I, I64, I64, P, P, I64, I, P, P], I),
            "qmm_id_with_path": ([P, I64, I, I64, I64, P, P, I64, I, P, I, P], I),
            "qmm_id_pick_path": ([I, I64, I64, I64, I], I),
            "qmm_with_tile": ([P, I, I64, I64, P, I64, P, I, P], I),
            "qmm_pick_tile": ([I64], I),
            "qmm_pick_path": ([I, I64, I64, I64], I),
            "qmm_launch_count": ([I, I64, I64, I64], I),
            "qmm_plan_info": ([I, I64, I64, I64, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "qmm_dequant": ([P, I, I64, I64, P, P], I),
            "qmm_quantize": ([P, I, I64, I64, P, P], I),
            "qmm_type_info": ([I, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "qmm_get_status": ([P], I),
            "qmm_debug_stall": ([P, I, I64, I64, P, I64, P, P], I),
            "qmm_strerror": ([I], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _qt(qtype) -> int:
    return TYPE_ID[qtype] if isinstance(qtype, str) else int(qtype)


def _stream(stream):
    if stream is not None:
        # a torch.cuda.Stream, or a raw cudaStream_t as an integer
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check(rc: int, what: str):
    if rc != 0:
        raise QmmError(rc, what)


def _xflag(x) -> int:
    import torch
    if x.dtype == torch.bfloat16:
        return X_BF16
    if x.dtype != torch.float32:
        raise TypeError("activations must be float32 or bfloat16, got %s" % x.dtype)
    return 0


def qmm_strerror(code: int) -> str:
    return lib().qmm_strerror(int(code)).decode()


def qmm_type_info(qtype):
    qk, nb = ctypes.c_int(), ctypes.c_int()
    _check(lib().qmm_type_info(_qt(qtype), ctypes.byref(qk), ctypes.byref(nb)), "qmm_type_info")
    return qk.value, nb.value


def row_bytes(qtype, K: int) -> int:
    qk, nb = qmm_type_info(qtype)
    return (K // qk) * nb


def qmm_pick_tile(M: int) -> int:
    return lib().qmm_pick_tile(int(M))


def qmm_pick_path(qtype, N: int, K: int, M: int) -> int:
    return lib().qmm_pick_path(_qt(qtype), int(N), int(K), int(M))


def qmm_launch_count(qtype, N: int, K: int, M: int, x_bf16: bool = False) -> int:
    return lib().qmm_launch_count(_qt(qtype) | (X_BF16 if x_bf16 else 0), int(N), int(K), int(M))


def qmm_plan_info(qtype, N: int, K: int, M: int, x_bf16: bool = False):
    """(path, K split, token columns per CTA) of the work plan (0, 0, 0 on the mat-vec path)."""
    S, c = ctypes.c_int(), ctypes.c_int()
    rc = lib().qmm_plan_info(_qt(qtype) | (X_BF16 if x_bf16 else 0), int(N), int(K), int(M), ctypes.byref(S),
                             ctypes.byref(c))
    if rc < 0:
        raise QmmError(rc, "qmm_plan_info")
    return rc, S.value, c.value


def qmm_workspace_size(qtype, N: int, K: int, M: int, x_bf16: bool = False) -> int:
    return lib().qmm_workspace_size(_qt(qtype) | (X_BF16 if x_bf16 else 0), int(N), int(K), int(M))


def qmm(wq, qtype, N: int, K: int, x, y, stream=None):
    """y[M, N] = x[M, K] @ dequant(wq)^T (x float32 or bfloat16, y float32; all CUDA tensors)."""
    M = x.shape[0]
    rc = lib().qmm(_ptr(wq), _qt(qtype) | _xflag(x), int(N), int(K), _ptr(x), int(M), _ptr(y), _stream(stream))
    _check(rc, "qmm")
    return y


def qmm_ws(wq, qtype, N: int, K: int, x, y, workspace, stream=None):
    M = x.shape[0]
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().qmm_ws(_ptr(wq), _qt(qtype) | _xflag(x), int(N), int(K), _ptr(x), int(M), _ptr(y),
                      _ptr(workspace), nbytes, _stream(stream))
    _check(rc, "qmm_ws")
    return y


def qmm_batch(wqs, qtype, Ns, K: int, x, ys, stream=None):
    """ys[i][M, N_i] = x[M, K] @ dequant(wqs[i])^T for matrices of one type that share x (one mat-vec launch
    for all of them when M <= 16)."""
    M = x.shape[0]
    n = len(wqs)
    W = (ctypes.c_void_p * n)(*[w.data_ptr() for w in wqs])
    NN = (ctypes.c_int64 * n)(*[int(v) for v in Ns])
    Y = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    rc = lib().qmm_batch(n, ctypes.cast(W, ctypes.c_void_p), ctypes.cast(NN, ctypes.c_void_p),
                         ctypes.cast(Y, ctypes.c_void_p), _qt(qtype) | _xflag(x), int(K), _ptr(x), int(M),
                         _stream(stream))
    _check(rc, "qmm_batch")
    return ys


def qmm_noalloc(wq, qtype, N: int, K: int, x, y, stream=None):
    """qmm() without any allocation: for callers that cannot allocate device memory while they run (the
    scratch of the tensor-core path comes from one device array the library owns; see include/qmm.h)."""
    M = x.shape[0]
    rc = lib().qmm_noalloc(_ptr(wq), _qt(qtype) | _xflag(x), int(N), int(K), _ptr(x), int(M), _ptr(y),
                           _stream(stream))
    _check(rc, "qmm_noalloc")
    return y


def qmm_with_tile(wq, qtype, N: int, K: int, x, y, tile: int, stream=None):
    M = x.shape[0]
    rc = lib().qmm_with_tile(_ptr(wq), _qt(qtype) | _xflag(x), int(N), int(K), _ptr(x), int(M), _ptr(y),
                             int(tile), _stream(stream))
    _check(rc, "qmm_with_tile")
    return y


def qmm_id(wqs, qtype, N: int, K: int, x, ids, y, stream=None, path: int = 0):
    """y[M, topk, N]: for each token t and slot j, x[t] @ dequant(wqs[ids[t, j]])^T; x of shape (M, K), or
    (M, topk, K) for one activation row per (token, slot), which is then x[t, j]. path 0 lets the library
    pick the kernel (qmm_id); 1 / 2 force the mat-vec / tensor-core expert kernel (qmm_id_with_path)."""
    M, topk = ids.shape
    flags = _xflag(x) | (X_PER_SLOT if x.dim() == 3 else 0)
    arr = (ctypes.c_void_p * len(wqs))(*[w.data_ptr() for w in wqs])
    if path == 0:
        rc = lib().qmm_id(ctypes.cast(arr, ctypes.c_void_p), len(wqs), _qt(qtype) | flags, int(N), int(K),
                          _ptr(x), _ptr(ids), int(M), int(topk), _ptr(y), _stream(stream))
    else:
        rc = lib().qmm_id_with_path(ctypes.cast(arr, ctypes.c_void_p), len(wqs), _qt(qtype) | flags, int(N),
                                    int(K), _ptr(x), _ptr(ids), int(M), int(topk), _ptr(y), int(path),
                                    _stream(stream))
    _check(rc, "qmm_id")
    return y


def qmm_id_pick_path(qtype, E: int, K: int, M: int, topk: int) -> int:
    return lib().qmm_id_pick_path(_qt(qtype), int(E), int(K), int(M), int(topk))


def qmm_dequant(wq, qtype, N: int, K: int, w_out, stream=None):
    _check(lib().qmm_dequant(_ptr(wq), _qt(qtype), int(N), int(K), _ptr(w_out), _stream(stream)), "qmm_dequant")
    return w_out


def qmm_quantize(w_in, qtype, N: int, K: int, wq_out, stream=None):
    _check(lib().qmm_quantize(_ptr(w_in), _qt(qtype), int(N), int(K), _ptr(wq_out), _stream(stream)),
           "qmm_quantize")
    return wq_out


def qmm_get_status(stream=None) -> int:
    """The device status bits (QMM_STATUS_*) since the last call, read and cleared (synchronises)."""
    rc = lib().qmm_get_status(_stream(stream))
    if rc < 0:
        raise QmmError(rc, "qmm_get_status")
    return rc


def qmm_debug_stall(wq, qtype, N: int, K: int, x, y, stream=None):
    """Test hook: a mat-vec call in which one bounded wait is made to run out (see include/qmm.h)."""
    M = x.shape[0]
    rc = lib().qmm_debug_stall(_ptr(wq), _qt(qtype) | _xflag(x), int(N), int(K), _ptr(x), int(M), _ptr(y),
                               _stream(stream))
    _check(rc, "qmm_debug_stall")
    return y

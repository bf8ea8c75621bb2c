"""Host-side checks of the C-ABI library: it loads without a GPU, exports every function include/qmm.h
declares, and rejects bad arguments with the documented codes before touching any device memory."""
import ctypes
import os
import re

import pytest

import weight_quantized_matmul_fly_gb300 as qmm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    qmm.build()
    return qmm.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "qmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(qmm[a-z_]*)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "qmm" in names and "qmm_id" in names and len(names) >= 10
    assert sorted(qmm.EXPORTS) == names
    for n in names:
        assert hasattr(L, n), n


def test_type_info_table(L):
    want = {"F32": (1, 4), "F16": (1, 2), "BF16": (1, 2), "Q4_0": (32, 18), "Q4_1": (32, 20), "Q5_0": (32, 22),
            "Q5_1": (32, 24), "Q8_0": (32, 34), "Q2_K": (256, 84), "Q3_K": (256, 110), "Q4_K": (256, 144),
            "Q5_K": (256, 176), "Q6_K": (256, 210), "A4G64": (64, 36)}
    for t, v in want.items():
        assert qmm.qmm_type_info(t) == v


def test_strerror(L):
    for c in range(-8, 1):
        assert isinstance(qmm.qmm_strerror(c), str) and qmm.qmm_strerror(c) != "unknown error"


P = ctypes.c_void_p
A = 0x1000  # a 16-byte aligned fake address; never dereferenced: every call below fails its checks first


@pytest.mark.parametrize("args,code", [
    ((P(A), 14, 64, 64, P(A), 1, P(A), None), -1),           # bad type
    ((P(A), 0x203, 64, 64, P(A), 1, P(A), None), -1),        # not a flag of qmm (per-slot x is qmm_id's)
    ((P(A), 0x803, 64, 64, P(A), 1, P(A), None), -1),        # unknown flag bit
    ((P(A), 3, 64, 48, P(A), 1, P(A), None), -2),            # K not a multiple of 32 for Q4_0
    ((P(A), 10, 64, 512 + 32, P(A), 1, P(A), None), -2),     # K not a multiple of 256 for Q4_K
    ((P(A), 3, 0, 64, P(A), 1, P(A), None), -3),             # N = 0
    ((P(A), 3, 64, 64, P(A), 0, P(A), None), -3),            # M = 0
    ((P(A), 3, 64, -32, P(A), 1, P(A), None), -3),           # K < 0
    ((None, 3, 64, 64, P(A), 1, P(A), None), -4),            # null wq
    ((P(A), 3, 64, 64, None, 1, P(A), None), -4),            # null x
    ((P(A + 8), 3, 64, 64, P(A), 1, P(A), None), -5),        # misaligned wq
    ((P(A), 3, 64, 64, P(A), 1, P(A + 4), None), -5),        # misaligned y
])
def test_qmm_argument_errors(L, args, code):
    assert L.qmm(*args) == code


def test_with_tile_bad_tile(L):
    assert L.qmm_with_tile(P(A), 3, 64, 64, P(A), 40, P(A), 48, None) == -7


def test_qmm_id_errors(L):
    ptrs = (ctypes.c_void_p * 2)(A, A)
    arr = ctypes.cast(ptrs, P)
    assert L.qmm_id(arr, 0, 3, 64, 64, P(A), P(A), 1, 8, P(A), None) == -7          # E = 0
    assert L.qmm_id(arr, 2, 3, 64, 64, P(A), P(A), 1000, 8, P(A), None) == -7       # M*topk too large
    assert L.qmm_id(arr, 2, 3, 64, 48, P(A), P(A), 1, 8, P(A), None) == -2          # K
    assert L.qmm_id(None, 2, 3, 64, 64, P(A), P(A), 1, 8, P(A), None) == -4
    bad = (ctypes.c_void_p * 2)(A, A + 2)
    assert L.qmm_id(ctypes.cast(bad, P), 2, 3, 64, 64, P(A), P(A), 1, 8, P(A), None) == -5


def test_qmm_id_flags(L):
    ptrs = (ctypes.c_void_p * 2)(A, A)
    arr = ctypes.cast(ptrs, P)
    assert L.qmm_id(arr, 2, 3 | 0x800, 64, 64, P(A), P(A), 1, 8, P(A), None) == -1   # unknown flag
    assert L.qmm_id(arr, 2, 3 | 0x200, 64, 48, P(A), P(A), 1, 8, P(A), None) == -2   # per-slot x accepted
    assert L.qmm(P(A), 3 | 0x200, 64, 64, P(A), 1, P(A), None) == -1                # not a qmm flag


def test_debug_stall_errors(L):
    assert L.qmm_debug_stall(P(A), 0, 64, 64, P(A), 1, P(A), None) == -7    # plain type: no such path
    assert L.qmm_debug_stall(P(A), 3, 64, 64, P(A), 17, P(A), None) == -7   # tensor-core path
    assert L.qmm_debug_stall(P(A), 3, 64, 64, None, 1, P(A), None) == -4


def test_dequant_quantize_errors(L):
    assert L.qmm_dequant(P(A), 20, 4, 64, P(A), None) == -1
    assert L.qmm_dequant(P(A), 3, 4, 40, P(A), None) == -2
    assert L.qmm_quantize(P(A), 3, 4, 64, None, None) == -4
    assert L.qmm_quantize(P(A + 1), 3, 4, 64, P(A), None) == -5


def test_pick_path(L):
    # mat-vec up to 16 tokens, tensor-core tile above
    assert qmm.qmm_pick_path("Q4_K", 4096, 2560, 1) == 0
    assert qmm.qmm_pick_path("Q4_K", 4096, 2560, 16) == 0
    assert qmm.qmm_pick_path("Q4_K", 4096, 2560, 17) == 32
    assert qmm.qmm_pick_path("Q4_K", 4096, 2560, 2048) == 128
    # plain type whose rows cannot be read by TMA stays on the mat-vec path
    assert qmm.qmm_pick_path("F32", 64, 33, 512) == 0


def test_workspace_size(L):
    # the mat-vec path needs no scratch
    assert qmm.qmm_workspace_size("Q4_K", 4096, 2560, 1) == 0
    # tensor-core path with binary32 x: its bf16 copy (and the partial sums of a K split) ...
    assert qmm.qmm_workspace_size("Q4_K", 9728, 2560, 2048) >= 2048 * 2560 * 2
    ws = qmm.qmm_workspace_size("Q4_K", 1024, 2560, 100)
    assert qmm.qmm_plan_info("Q4_K", 1024, 2560, 100)[1] > 1 and ws >= 100 * 2560 * 2 + 2 * 100 * 1024 * 4
    # up to 32 tokens the kernel converts x itself (measured as fast as the copy there)
    assert qmm.qmm_workspace_size("Q4_K", 1024, 2560, 32) == 0
    # ... and nothing with bf16 x (a K split is added inside a cluster)
    assert qmm.qmm_workspace_size("Q4_K", 9728, 2560, 2048, x_bf16=True) == 0
    assert qmm.qmm_workspace_size("Q6_K", 1024, 2560, 33, x_bf16=True) == 0


def test_launch_count(L):
    assert qmm.qmm_launch_count("Q4_K", 9728, 2560, 1) == 1
    assert qmm.qmm_launch_count("Q4_K", 9728, 2560, 2048) == 2            # bf16 copy of x + mm (qmm_ws)
    assert qmm.qmm_launch_count("Q4_K", 9728, 2560, 2048, x_bf16=True) == 1
    assert qmm.qmm_launch_count("Q4_K", 1024, 2560, 100, x_bf16=True) == 1   # K split inside a cluster
    assert qmm.qmm_launch_count("Q4_K", 1024, 2560, 100) == 3             # copy of x + mm + split reduction


def test_noalloc_checks_arguments_first(L):
    # a null x with a large M is a null pointer, not an oversized workspace
    assert L.qmm_noalloc(P(A), 3, 64, 8192, None, 1 << 20, P(A), None) == -4
    assert L.qmm_noalloc(P(A), 3, 64, -64, P(A), 1 << 20, P(A), None) == -3


def test_qmm_id_path_choice(L):
    # a few pairs per expert: the mat-vec expert kernel; many (prefill): the tensor-core one
    assert qmm.qmm_id_pick_path("Q4_0", 128, 512, 24, 8) == 1
    assert qmm.qmm_id_pick_path("Q4_0", 128, 512, 256, 8) == 1
    assert qmm.qmm_id_pick_path("Q4_0", 16, 512, 256, 8) == 2
    assert qmm.qmm_id_pick_path("F32", 1, 256, 128, 1) == 2
    ptrs = (ctypes.c_void_p * 2)(A, A)
    arr = ctypes.cast(ptrs, P)
    assert L.qmm_id_with_path(arr, 2, 3, 64, 64, P(A), P(A), 1, 8, P(A), 3, None) == -7   # no such path

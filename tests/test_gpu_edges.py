"""GPU parity on the edges of the input space, against the oracle element by element.

- qmm_id with plain F32 / F16 / BF16 experts (the CUDA-core expert kernel), K = 256 and 768,
  1 / 7 / 24 tokens, binary32 and bfloat16 activations (llama.cpp PR 28086, "metal : fix idle threads in
  mul_mv_iq3_xxs for ne00 < 1024", "Additional information": GPU against the CPU backend for MUL_MAT and
  MUL_MAT_ID at K = 256 and 768).
- K that is not a multiple of 256 for the 32- and 64-weight block types: the last macro block of a row
  holds fewer than 8 (4) blocks, on the mat-vec path, the tensor-core path (every token tile, bit-identical
  to one another: candle PR 4056, "Metal: 64-token tile for the quantized matrix-matrix kernel", section
  "Same results, bit for bit") and the expert-indexed path; the 1 x 32 x 1 case included.
- Blocks whose scales are NaN, infinite, subnormal or zero, through qmm, qmm_with_tile and qmm_id.
  Reading of the format specification for these: the dequantized weight is the IEEE value of the formula,
  so outputs that see no infinite scale must match the oracle's NaN pattern exactly (NaN == NaN) and be
  within tolerance elsewhere. An infinite scale times a zero code is NaN per weight in the oracle, while the
  kernels apply a unit's scale once to its code sum (ds * sum(q x)), which resolves such a row to a NaN or an
  infinity; for those outputs the test requires a non-finite value wherever the oracle's is non-finite.
"""
import numpy as np
import pytest

import oracle
import synthetic
import weight_quantized_matmul_fly_gb300 as qmm
from gpu_util import TOL_BF16, TOL_FP32, bit_differences, check_tol, dev, torch_cuda, x_dev

pytestmark = pytest.mark.gpu

LEGACY = ["Q4_0", "Q4_1", "Q5_0", "Q5_1", "Q8_0"]


def _run_qmm(fn, wq, qtype, N, K, x, **kw):
    torch = torch_cuda()
    M = x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fn(dev(wq), qtype, N, K, x_dev(x), y, **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _run_id(wqs, qtype, N, K, x, ids):
    torch = torch_cuda()
    M, topk = ids.shape
    y = torch.full((M, topk, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_id([dev(w) for w in wqs], qtype, N, K, x_dev(x), dev(ids), y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


# ------------------------------------------------------------------ plain-type experts

@pytest.mark.parametrize("qtype", ["F32", "F16", "BF16"])
@pytest.mark.parametrize("K", [256, 768])
@pytest.mark.parametrize("M", [1, 7, 24])
@pytest.mark.parametrize("bf16", [False, True])
def test_qmm_id_plain_types(qtype, K, M, bf16):
    E, N, topk = 16, 130, 8
    wqs = [oracle.quantize(qtype, synthetic.weights(N, K, seed=300 + e)) for e in range(E)]
    x = synthetic.activations(M, K, seed=M + K, bf16=bf16)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=M + K)
    y = _run_id(wqs, qtype, N, K, x, ids)
    ref, bnd = oracle.qmm_id(qtype, wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, "%s K=%d M=%d bf16=%s" % (qtype, K, M, bf16))


def test_qmm_id_plain_bad_ids():
    torch_cuda()
    E, N, K = 3, 40, 256
    wqs = [oracle.quantize("F16", synthetic.weights(N, K, seed=400 + e)) for e in range(E)]
    x = synthetic.activations(2, K, seed=4)
    ids = np.array([[0, 5], [2, -3]], dtype=np.int32)
    qmm.qmm_get_status()
    y = _run_id(wqs, "F16", N, K, x, ids)
    assert qmm.qmm_get_status() & qmm.STATUS_BAD_ID
    ref, bnd = oracle.qmm_id("F16", wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, "plain bad ids")


# ------------------------------------------------------------------ K tails (K not a multiple of 256)

TAIL_CASES = [(qt, K) for qt in LEGACY for K in (32, 96, 800)] + [("A4G64", 64), ("A4G64", 192)]


@pytest.mark.parametrize("qtype,K", TAIL_CASES)
def test_k_tail_matvec(qtype, K):
    N = 150
    wq = oracle.quantize(qtype, synthetic.weights(N, K, seed=K))
    for M in (1, 7, 16):
        x = synthetic.activations(M, K, seed=M)
        assert qmm.qmm_pick_path(qtype, N, K, M) == 0
        y = _run_qmm(qmm.qmm, wq, qtype, N, K, x)
        ref, bnd = oracle.qmm(qtype, wq, N, K, x)
        check_tol(y, ref, bnd, TOL_FP32, "%s K=%d M=%d" % (qtype, K, M))


@pytest.mark.parametrize("qtype,K", TAIL_CASES)
def test_k_tail_tensor_core(qtype, K):
    N = 150
    wq = oracle.quantize(qtype, synthetic.weights(N, K, seed=K + 1))
    for M in (17, 33, 130):
        x = synthetic.activations(M, K, seed=M + 1)
        outs = [_run_qmm(qmm.qmm_with_tile, wq, qtype, N, K, x, tile=t) for t in (32, 64, 128)]
        ref, bnd = oracle.qmm(qtype, wq, N, K, x)
        check_tol(outs[0], ref, bnd, TOL_BF16, "%s K=%d M=%d" % (qtype, K, M))
        assert np.any(outs[0] != 0)
        for t, o in zip((64, 128), outs[1:]):
            assert bit_differences(o, outs[0]) == 0, "%s K=%d M=%d: tile %d differs from tile 32" % (
                qtype, K, M, t)
        y = _run_qmm(qmm.qmm, wq, qtype, N, K, x)
        assert bit_differences(y, outs[0]) == 0


@pytest.mark.parametrize("qtype,K", TAIL_CASES)
def test_k_tail_qmm_id(qtype, K):
    E, N, topk = 6, 90, 3
    wqs = [oracle.quantize(qtype, synthetic.weights(N, K, seed=500 + e)) for e in range(E)]
    for M in (1, 9):
        x = synthetic.activations(M, K, seed=M + 2)
        ids = synthetic.expert_ids(M, E=E, topk=topk, seed=M + 2)
        y = _run_id(wqs, qtype, N, K, x, ids)
        ref, bnd = oracle.qmm_id(qtype, wqs, N, K, x, ids)
        check_tol(y, ref, bnd, TOL_FP32, "%s K=%d M=%d" % (qtype, K, M))


@pytest.mark.parametrize("qtype", LEGACY + ["A4G64", "F32", "F16", "BF16"])
def test_one_row_one_block_one_token(qtype):
    """N = 1, K = one block (32 weights; 64 for A4G64), M = 1: the smallest call."""
    K = 64 if qtype == "A4G64" else 32
    wq = oracle.quantize(qtype, synthetic.weights(1, K, seed=1))
    x = synthetic.activations(1, K, seed=1)
    y = _run_qmm(qmm.qmm, wq, qtype, 1, K, x)
    ref, bnd = oracle.qmm(qtype, wq, 1, K, x)
    check_tol(y, ref, bnd, TOL_FP32, qtype)


# ------------------------------------------------------------------ special scale values

# (offset, width) of the scale-like fields of one block, from the block format specification's layout
SCALE_FIELDS = {
    "Q4_0": [(0, "h")], "Q4_1": [(0, "h"), (2, "h")], "Q5_0": [(0, "h")], "Q5_1": [(0, "h"), (2, "h")],
    "Q8_0": [(0, "h")], "Q2_K": [(80, "h"), (82, "h")], "Q3_K": [(108, "h")], "Q4_K": [(0, "h"), (2, "h")],
    "Q5_K": [(0, "h"), (2, "h")], "Q6_K": [(208, "h")], "A4G64": [(0, "b"), (2, "b")],
}
H_NAN, H_INF, H_NINF = 0x7E00, 0x7C00, 0xFC00
H_SUB = [0x0001, 0x03FF, 0x8001, 0x0000, 0x8000]
B_NAN, B_INF, B_NINF = 0x7FC0, 0x7F80, 0xFF80
B_SUB = [0x0001, 0x007F, 0x8001, 0x0000, 0x8000]


def _special(qtype, N, K, seed, with_inf):
    """A normally quantized matrix in which the odd rows have about two blocks (at most a quarter of
    their blocks) whose scale fields are replaced by NaN, +-infinity (when with_inf), subnormal or zero
    bit patterns. Plain types: a third of the rows have 1 % of their elements replaced likewise."""
    g = np.random.default_rng(seed)
    w = synthetic.weights(N, K, seed=seed)
    if qtype in ("F32", "F16", "BF16"):
        if qtype == "F32":
            specials = [np.float32(np.nan), np.float32(1e-40), np.float32(-3e-45), np.float32(0)]
            if with_inf:
                specials += [np.float32(np.inf), np.float32(-np.inf)]
            wq = oracle.quantize(qtype, w).view(np.float32).reshape(N, K).copy()
        else:
            hs = (H_NAN, *H_SUB[:3]) if qtype == "F16" else (B_NAN, *B_SUB[:3])
            if with_inf:
                hs += (H_INF, H_NINF) if qtype == "F16" else (B_INF, B_NINF)
            specials = [np.uint16(v) for v in hs]
            wq = oracle.quantize(qtype, w).view(np.uint16).reshape(N, K).copy()
        # a third of the rows carry special elements (1 % of their elements), the others stay finite
        mask = (g.random((N, K)) < 0.01) & (np.arange(N) % 3 == 0)[:, None]
        picks = g.integers(0, len(specials), int(mask.sum()))
        wq[mask] = np.array(specials, dtype=wq.dtype)[picks]
        return wq.view(np.uint8).reshape(N, -1).copy()
    wq = oracle.quantize(qtype, w).copy()
    qk, nbytes = oracle.type_info(qtype)
    nb = K // qk
    blocks = wq.reshape(N, nb, nbytes)
    fields = SCALE_FIELDS[qtype]
    pblk = min(0.25, 2.0 / nb)            # about two special blocks in each odd row; even rows stay finite
    for n in range(1, N, 2):
        for b in range(nb):
            if g.random() >= pblk:
                continue
            off, kind = fields[g.integers(0, len(fields))]
            nan, inf, ninf, sub = (H_NAN, H_INF, H_NINF, H_SUB) if kind == "h" else (B_NAN, B_INF, B_NINF, B_SUB)
            choices = [nan] + sub + ([inf, ninf] if with_inf else [])
            v = int(choices[g.integers(0, len(choices))])
            blocks[n, b, off] = v & 255
            blocks[n, b, off + 1] = v >> 8
    return wq


def _check_special(y, ref, bnd, tol, what, with_inf):
    if not with_inf:
        check_tol(y, ref, bnd, tol, what)
        return
    fin = np.isfinite(ref)
    assert np.all(~np.isfinite(y[~fin])), what + ": finite output where the oracle's is not"
    assert np.all(np.isfinite(y[fin])), what + ": non-finite output where the oracle's is finite"
    check_tol(np.where(fin, y, 0.0), np.where(fin, ref, 0.0), np.where(fin, bnd, 1.0), tol, what)


SPECIAL_TYPES = LEGACY + ["Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K", "A4G64", "F32", "F16", "BF16"]


@pytest.mark.parametrize("qtype", SPECIAL_TYPES)
@pytest.mark.parametrize("with_inf", [False, True])
def test_special_scales_matvec(qtype, with_inf):
    N, K = 96, 1024
    wq = _special(qtype, N, K, seed=11, with_inf=with_inf)
    for M in (1, 7):
        x = synthetic.activations(M, K, seed=M + 20)
        y = _run_qmm(qmm.qmm, wq, qtype, N, K, x)
        ref, bnd = oracle.qmm(qtype, wq, N, K, x)
        assert np.isnan(ref).any()
        _check_special(y, ref, bnd, TOL_FP32, "%s M=%d" % (qtype, M), with_inf)


@pytest.mark.parametrize("qtype", SPECIAL_TYPES)
@pytest.mark.parametrize("with_inf", [False, True])
def test_special_scales_tensor_core(qtype, with_inf):
    N, K, M = 96, 1024, 40
    wq = _special(qtype, N, K, seed=12, with_inf=with_inf)
    x = synthetic.activations(M, K, seed=21)
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    outs = [_run_qmm(qmm.qmm_with_tile, wq, qtype, N, K, x, tile=t) for t in (32, 64, 128)]
    _check_special(outs[0], ref, bnd, TOL_BF16, "%s tile 32" % qtype, with_inf)
    for t, o in zip((64, 128), outs[1:]):
        # bit identity across tiles, NaN payloads aside
        same = (o.view(np.uint32) == outs[0].view(np.uint32)) | (np.isnan(o) & np.isnan(outs[0]))
        assert same.all(), "%s: tile %d differs from tile 32 at %d outputs" % (qtype, t, int((~same).sum()))
    y = _run_qmm(qmm.qmm, wq, qtype, N, K, x)
    _check_special(y, ref, bnd, TOL_BF16, "%s qmm" % qtype, with_inf)


@pytest.mark.parametrize("qtype", ["Q4_0", "Q4_1", "Q4_K", "Q6_K", "A4G64", "F16", "F32"])
@pytest.mark.parametrize("with_inf", [False, True])
def test_special_scales_qmm_id(qtype, with_inf):
    E, N, K, M, topk = 5, 64, 512, 6, 3
    wqs = [_special(qtype, N, K, seed=30 + e, with_inf=with_inf) for e in range(E)]
    x = synthetic.activations(M, K, seed=22)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=22)
    y = _run_id(wqs, qtype, N, K, x, ids)
    ref, bnd = oracle.qmm_id(qtype, wqs, N, K, x, ids)
    _check_special(y, ref, bnd, TOL_FP32, "%s qmm_id" % qtype, with_inf)

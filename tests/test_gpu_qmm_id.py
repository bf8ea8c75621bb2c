"""qmm_id (expert-indexed mat-vec) on the GPU against the oracle: K = 256 / 512 / 768 / 1024 (row split
2 and 4, the plain mapping at 24 chunks), 1..24 tokens, top-8 of 16 experts (so experts are shared by
several tokens), and out-of-range ids."""
import numpy as np
import pytest

import oracle
import synthetic
import weight_quantized_matmul_fly_gb300 as qmm
from gpu_util import TOL_FP32, check_tol, dev, torch_cuda, x_dev

pytestmark = pytest.mark.gpu


def _experts(qtype, E, N, K, seed):
    return [oracle.quantize(qtype, synthetic.weights(N, K, seed=seed + e)) for e in range(E)]


def _run(wqs, qtype, N, K, x, ids):
    torch = torch_cuda()
    M, topk = ids.shape
    y = torch.full((M, topk, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_id([dev(w) for w in wqs], qtype, N, K, x_dev(x), dev(ids), y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("K", [256, 512, 768, 1024])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 12, 16, 24])
def test_qmm_id_q4_0(K, M):
    E, N, topk = 16, 200, 8
    wqs = _experts("Q4_0", E, N, K, seed=K)
    x = synthetic.activations(M, K, seed=M)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=M)
    y = _run(wqs, "Q4_0", N, K, x, ids)
    ref, bnd = oracle.qmm_id("Q4_0", wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, "K=%d M=%d" % (K, M))


@pytest.mark.parametrize("qtype", ["Q4_K", "Q6_K", "Q8_0", "A4G64"])
def test_qmm_id_other_types(qtype):
    E, N, K, M, topk = 8, 130, 1024, 6, 3
    wqs = _experts(qtype, E, N, K, seed=50)
    x = synthetic.activations(M, K, seed=2, bf16=(qtype == "A4G64"))
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=2)
    y = _run(wqs, qtype, N, K, x, ids)
    ref, bnd = oracle.qmm_id(qtype, wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, qtype)


def test_qmm_id_duplicate_and_bad_ids():
    torch_cuda()
    E, N, K = 4, 70, 512
    wqs = _experts("Q4_0", E, N, K, seed=9)
    x = synthetic.activations(3, K, seed=9)
    ids = np.array([[0, 0, 3], [2, 7, 1], [-1, 3, 3]], dtype=np.int32)
    qmm.qmm_get_status()  # clear
    y = _run(wqs, "Q4_0", N, K, x, ids)
    st = qmm.qmm_get_status()
    assert st & qmm.STATUS_BAD_ID
    ref, bnd = oracle.qmm_id("Q4_0", wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, "dup/bad ids")
    assert np.all(np.isnan(y[1, 1])) and np.all(np.isnan(y[2, 0]))
    assert qmm.qmm_get_status() == 0


def test_qmm_id_long_k_cluster_split():
    """K = 8192 (32 macro blocks): the work split takes 4 K segments per cluster, whose partial sums are
    added in rank order; 5 tokens routed to 2 of 4 experts."""
    E, N, K, M, topk = 4, 64, 8192, 5, 2
    wqs = _experts("Q4_0", E, N, K, seed=77)
    x = synthetic.activations(M, K, seed=77)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=77)
    y = _run(wqs, "Q4_0", N, K, x, ids)
    ref, bnd = oracle.qmm_id("Q4_0", wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, "K=8192")


@pytest.mark.parametrize("bf16", [False, True])
def test_qmm_id_many_slots_per_expert(bf16):
    """64 tokens over 4 experts (about 64 slots each): many passes of 4 (8 for bf16 activations) tokens."""
    E, N, K, M, topk = 4, 96, 512, 64, 4
    wqs = _experts("Q4_K", E, N, K, seed=5)
    x = synthetic.activations(M, K, seed=5, bf16=bf16)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=5)
    y = _run(wqs, "Q4_K", N, K, x, ids)
    ref, bnd = oracle.qmm_id("Q4_K", wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, "many slots bf16=%s" % bf16)


@pytest.mark.parametrize("qtype", ["Q4_0", "Q4_K", "Q6_K", "A4G64", "F16", "BF16"])
@pytest.mark.parametrize("M", [1, 5, 24])
def test_qmm_id_per_slot_activations(qtype, M):
    """x of shape M x topk x K (one activation row per routed pair, the experts' down projection:
    llama.cpp PR 28086, "Test methodology", ffn_down_exps), on both expert kernels."""
    E, N, K, topk = 12, 140, 512, 8
    wqs = _experts(qtype, E, N, K, seed=60)
    bf16 = qtype == "A4G64"
    x = synthetic.activations(M * topk, K, seed=M + 60, bf16=bf16).reshape(M, topk, K)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=M + 60)
    y = _run(wqs, qtype, N, K, x, ids)
    ref, bnd = oracle.qmm_id(qtype, wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_FP32, "%s per-slot M=%d" % (qtype, M))
    # the broadcast form is the per-slot form with every slot given its token's row
    xb = synthetic.activations(M, K, seed=M + 61, bf16=bf16)
    y1 = _run(wqs, qtype, N, K, xb, ids)
    y2 = _run(wqs, qtype, N, K, np.ascontiguousarray(np.repeat(xb[:, None, :], topk, axis=1)), ids)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))

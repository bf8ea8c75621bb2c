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
    """64 tokens over 4 experts (about 64 slots each): on the tensor-core expert kernel (bf16 class), and on
    the mat-vec expert kernel, many passes of 4 (8 for bf16 activations) tokens (binary32 class)."""
    from gpu_util import TOL_BF16
    E, N, K, M, topk = 4, 96, 512, 64, 4
    wqs = _experts("Q4_K", E, N, K, seed=5)
    x = synthetic.activations(M, K, seed=5, bf16=bf16)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=5)
    ref, bnd = oracle.qmm_id("Q4_K", wqs, N, K, x, ids)
    y = _run_path(wqs, "Q4_K", N, K, x, ids, 2)
    check_tol(y, ref, bnd, TOL_BF16, "many slots, tensor-core, bf16=%s" % bf16)
    y1 = _run_path(wqs, "Q4_K", N, K, x, ids, 1)
    check_tol(y1, ref, bnd, TOL_FP32, "many slots, mat-vec, bf16=%s" % bf16)


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
    from gpu_util import TOL_BF16
    tol = TOL_BF16 if qmm.qmm_id_pick_path(qtype, E, K, M, topk) == 2 else TOL_FP32
    check_tol(y, ref, bnd, tol, "%s per-slot M=%d" % (qtype, M))
    # the broadcast form is the per-slot form with every slot given its token's row
    xb = synthetic.activations(M, K, seed=M + 61, bf16=bf16)
    y1 = _run(wqs, qtype, N, K, xb, ids)
    y2 = _run(wqs, qtype, N, K, np.ascontiguousarray(np.repeat(xb[:, None, :], topk, axis=1)), ids)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


# ------------------------------------------------------------------ tensor-core expert path (many pairs per expert)

def _run_path(wqs, qtype, N, K, x, ids, path):
    torch = torch_cuda()
    M, topk = ids.shape
    y = torch.full((M, topk, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.qmm_id([dev(w) for w in wqs], qtype, N, K, x_dev(x), dev(ids), y, path=path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("n", [32, 64, 256])
def test_qmm_id_tensor_core_128_experts(n):
    """Prefill-sized routing (llama.cpp PR 28086, "Test methodology": MUL_MAT_ID): n tokens, top-8 of 128
    experts, on the tensor-core expert kernel, element by element against the oracle (bf16 class), and
    the mat-vec expert kernel on the same inputs (binary32 class)."""
    from gpu_util import TOL_BF16
    E, N, K, topk = 128, 256, 512, 8
    wqs = _experts("Q4_0", E, N, K, seed=700)
    x = synthetic.activations(n, K, seed=n)
    ids = synthetic.expert_ids(n, E=E, topk=topk, seed=n)
    ref, bnd = oracle.qmm_id("Q4_0", wqs, N, K, x, ids)
    y2 = _run_path(wqs, "Q4_0", N, K, x, ids, 2)
    check_tol(y2, ref, bnd, TOL_BF16, "tensor-core n=%d" % n)
    y1 = _run_path(wqs, "Q4_0", N, K, x, ids, 1)
    check_tol(y1, ref, bnd, TOL_FP32, "mat-vec n=%d" % n)
    assert qmm.qmm_id_pick_path("Q4_0", E, K, n, topk) == (2 if n * topk >= 128 * min(E, n * topk) else 1)


@pytest.mark.parametrize("qtype", ["Q4_K", "Q6_K", "Q8_0", "A4G64", "Q5_1", "F16", "F32"])
def test_qmm_id_tensor_core_types_and_passes(qtype):
    """Few experts and many tokens, so that experts get more pairs than one pass holds (several passes
    into the same accumulator), with a duplicate id and ragged rows."""
    from gpu_util import TOL_BF16
    E, N, K, M, topk = 4, 200, 512, 150, 2
    wqs = _experts(qtype, E, N, K, seed=800)
    bf16 = qtype == "A4G64"
    x = synthetic.activations(M, K, seed=8, bf16=bf16)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=8)
    ids[3] = [1, 1]
    ref, bnd = oracle.qmm_id(qtype, wqs, N, K, x, ids)
    y = _run_path(wqs, qtype, N, K, x, ids, 2)
    check_tol(y, ref, bnd, TOL_BF16, qtype)


@pytest.mark.parametrize("bf16", [False, True])
def test_qmm_id_tensor_core_per_slot_and_k_tail(bf16):
    """Per-slot activation rows (M x topk x K) and K = 96 (the last K step half full), plus bad ids."""
    from gpu_util import TOL_BF16
    torch_cuda()
    E, N, K, M, topk = 6, 130, 96, 40, 3
    wqs = _experts("Q4_0", E, N, K, seed=900)
    x = synthetic.activations(M * topk, K, seed=9, bf16=bf16).reshape(M, topk, K)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=9)
    ids[5, 1] = 77
    ids[7, 0] = -2
    qmm.qmm_get_status()
    y = _run_path(wqs, "Q4_0", N, K, x, ids, 2)
    assert qmm.qmm_get_status() & qmm.STATUS_BAD_ID
    ref, bnd = oracle.qmm_id("Q4_0", wqs, N, K, x, ids)
    check_tol(y, ref, bnd, TOL_BF16, "per-slot bf16=%s" % bf16)

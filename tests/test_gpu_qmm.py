"""qmm on the GPU against the oracle, element by element, and bit-identity across token tiles.

Tolerances: |y - y_ref| <= 1e-5 * sum_k |w x| on the mat-vec path (binary32 products of the exactly
rounded weights) and <= 4e-3 * sum_k |w x| on the tensor-core path (x and w rounded to bfloat16).
Shapes span several tiles with ragged tails in rows (N = 300, 200), tokens and K."""
import numpy as np
import pytest

import oracle
import synthetic
import weight_quantized_matmul_fly_gb300 as qmm
from gpu_util import TOL_BF16, TOL_FP32, bit_differences, check_tol, dev, torch_cuda, x_dev

pytestmark = pytest.mark.gpu
TYPES = oracle.TYPES


def _case(qtype, N, K, M, seed, bf16=False):
    wq = oracle.quantize(qtype, synthetic.weights(N, K, seed=seed))
    x = synthetic.activations(M, K, seed=seed, bf16=bf16)
    return wq, x


def _run(fn, wq, qtype, N, K, x, **kw):
    torch = torch_cuda()
    M = x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fn(dev(wq), qtype, N, K, x_dev(x), y, **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M", [1, 2, 3, 7, 16])
def test_gemv_path(qtype, M):
    N, K = 300, 512
    wq, x = _case(qtype, N, K, M, seed=M)
    assert qmm.qmm_pick_path(qtype, N, K, M) == 0
    y = _run(qmm.qmm, wq, qtype, N, K, x)
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    check_tol(y, ref, bnd, TOL_FP32, "%s M=%d" % (qtype, M))


@pytest.mark.parametrize("qtype", ["Q4_0", "Q4_K", "Q6_K", "Q3_K", "Q8_0", "A4G64", "F16"])
@pytest.mark.parametrize("K", [256, 768, 1024, 2560])
def test_gemv_narrow_and_wide_k(qtype, K):
    """K = 256 (4 rows per warp), 768 (24 chunks, plain mapping), 1024 and 2560."""
    if K % oracle.type_info(qtype)[0]:
        pytest.skip("K not a multiple of the block size")
    N, M = 130, 5
    wq, x = _case(qtype, N, K, M, seed=K)
    y = _run(qmm.qmm, wq, qtype, N, K, x)
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    check_tol(y, ref, bnd, TOL_FP32, "%s K=%d" % (qtype, K))


@pytest.mark.parametrize("qtype", ["F32", "F16", "BF16"])
@pytest.mark.parametrize("K", [1, 33, 100])
def test_plain_types_odd_k(qtype, K):
    N = 70
    for M in (1, 9, 40):
        wq, x = _case(qtype, N, K, M, seed=K + M)
        y = _run(qmm.qmm, wq, qtype, N, K, x)
        ref, bnd = oracle.qmm(qtype, wq, N, K, x)
        check_tol(y, ref, bnd, TOL_FP32, "%s K=%d M=%d" % (qtype, K, M))


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("M", [17, 33, 100, 130])
def test_tensor_core_path(qtype, M):
    N, K = 200, 512
    wq, x = _case(qtype, N, K, M, seed=100 + M)
    assert qmm.qmm_pick_path(qtype, N, K, M) in (32, 64, 128)
    y = _run(qmm.qmm, wq, qtype, N, K, x)
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    check_tol(y, ref, bnd, TOL_BF16, "%s M=%d" % (qtype, M))


@pytest.mark.parametrize("qtype", ["A4G64", "Q4_0", "Q4_K"])
@pytest.mark.parametrize("M", [1, 4, 16, 48])
def test_bf16_activations(qtype, M):
    N, K = 260, 1024
    wq, x = _case(qtype, N, K, M, seed=7, bf16=True)
    y = _run(qmm.qmm, wq, qtype, N, K, x)
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    check_tol(y, ref, bnd, TOL_FP32 if M <= 16 else TOL_BF16, "%s bf16 M=%d" % (qtype, M))


@pytest.mark.parametrize("qtype,N,K,M", [("Q4_K", 9728, 2560, 512), ("Q6_K", 2560, 9728, 600), ("Q4_0", 256, 2560, 64)])
def test_workspace_entry_point(qtype, N, K, M):
    """qmm_ws with its scratch (a bf16 copy of x read at the plan's full width, K splits added by a second
    kernel) and qmm (no scratch: x converted inside the kernel, splits added in a cluster): both within the
    tolerance of the oracle on sampled outputs, and a call repeated gives the same bits."""
    torch = torch_cuda()
    wq, x = _case(qtype, N, K, M, seed=5)
    nb = qmm.qmm_workspace_size(qtype, N, K, M)
    assert nb >= M * K * 2
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda") if nb else None
    y = _run(qmm.qmm_ws, wq, qtype, N, K, x, workspace=ws)
    y1 = _run(qmm.qmm_ws, wq, qtype, N, K, x, workspace=ws)
    y2 = _run(qmm.qmm, wq, qtype, N, K, x)
    assert np.array_equal(y.view(np.uint32), y1.view(np.uint32))
    g = np.random.default_rng(M)
    ms, ns = g.integers(0, M, 500), g.integers(0, N, 500)
    ref, bnd = oracle.qmm_sampled(qtype, wq, N, K, x, ms, ns)
    check_tol(y[ms, ns], ref, bnd, TOL_BF16, qtype + " qmm_ws")
    check_tol(y2[ms, ns], ref, bnd, TOL_BF16, qtype + " qmm")


@pytest.mark.parametrize("qtype", ["Q4_K", "Q6_K", "Q4_0", "Q8_0", "A4G64"])
@pytest.mark.parametrize("M", [17, 40, 100, 130, 260])
def test_k_split_in_cluster(qtype, M):
    """Few row blocks and a long K make the plan split K over a cluster of up to 8 CTAs that add their
    partials in split order in shared memory: element-wise parity with the oracle, bit-identity across the
    token tiles, with binary32 (converted in the kernel) and bf16 activations."""
    N, K = 200, 4096
    wq, x = _case(qtype, N, K, M, seed=M + 3)
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    outs = [_run(qmm.qmm_with_tile, wq, qtype, N, K, x, tile=t) for t in (32, 64, 128)]
    check_tol(outs[0], ref, bnd, TOL_BF16, "%s M=%d" % (qtype, M))
    for t, o in zip((64, 128), outs[1:]):
        assert bit_differences(o, outs[0]) == 0, "%s M=%d: tile %d differs" % (qtype, M, t)
    y = _run(qmm.qmm, wq, qtype, N, K, x)
    assert bit_differences(y, outs[0]) == 0
    # with scratch (M > 32): the partial tiles go through global memory to a second kernel, in split order
    torch = torch_cuda()
    nb = qmm.qmm_workspace_size(qtype, N, K, M)
    assert (nb > 0) == (M > 32)
    if nb:
        assert qmm.qmm_plan_info(qtype, N, K, M)[1] > 1
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        yw = _run(qmm.qmm_ws, wq, qtype, N, K, x, workspace=ws)
        check_tol(yw, ref, bnd, TOL_BF16, "%s qmm_ws M=%d" % (qtype, M))
    xb = synthetic.activations(M, K, seed=M + 3, bf16=True)
    yb = _run(qmm.qmm, wq, qtype, N, K, xb)
    refb, bndb = oracle.qmm(qtype, wq, N, K, xb)
    check_tol(yb, refb, bndb, TOL_BF16, "%s bf16 M=%d" % (qtype, M))


@pytest.mark.parametrize("tile", [0, 32, 64, 128])
def test_forced_tiles_parity(tile):
    N, K, M = 136, 768, 45
    qtype = "Q5_K"
    wq, x = _case(qtype, N, K, M, seed=tile)
    y = _run(qmm.qmm_with_tile, wq, qtype, N, K, x, tile=tile)
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    check_tol(y, ref, bnd, TOL_FP32 if tile == 0 else TOL_BF16, "tile %d" % tile)


# ------------------------------------------------------------------ bit-identity across token tiles

INVARIANCE_SHAPES = [  # (batch, tokens, rows, K): candle PR 4056, section "Same results, bit for bit"
    (1, 7, 96, 512), (1, 32, 96, 512), (1, 33, 96, 512), (1, 130, 96, 512), (2, 65, 128, 768)]


@pytest.mark.parametrize("qtype", oracle.TYPES[:13])
def test_tile_invariance(qtype):
    for batch, M, N, K in INVARIANCE_SHAPES:
        if K % oracle.type_info(qtype)[0]:
            continue
        for b in range(batch):
            wq, x = _case(qtype, N, K, M, seed=1000 + 7 * b + M)
            outs = [_run(qmm.qmm_with_tile, wq, qtype, N, K, x, tile=t) for t in (32, 64, 128)]
            assert np.any(outs[0] != 0), "all-zero output"
            for t, o in zip((64, 128), outs[1:]):
                d = bit_differences(o, outs[0])
                assert d == 0, "%s %dx%dx%dx%d: %d of %d outputs differ between tiles 32 and %d" % (
                    qtype, batch, M, N, K, d, o.size, t)


@pytest.mark.parametrize("qtype", ["Q4_K", "Q6_K", "Q4_0"])
@pytest.mark.parametrize("M", [1, 7, 40, 300])
def test_static_weights_flag_same_bits(qtype, M):
    """QMM_W_STATIC only moves the weight reads before the wait for the preceding kernel: same bits."""
    torch = torch_cuda()
    N, K = 260, 1024
    wq, x = _case(qtype, N, K, M, seed=M + 11)
    a = _run(qmm.qmm, wq, qtype, N, K, x)
    b = _run(qmm.qmm, wq, qmm.TYPE_ID[qtype] | qmm.W_STATIC, N, K, x)
    assert bit_differences(a, b) == 0
    nb = qmm.qmm_workspace_size(qtype, N, K, M)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    c = _run(qmm.qmm_ws, wq, qtype, N, K, x, workspace=ws)
    d = _run(qmm.qmm_ws, wq, qmm.TYPE_ID[qtype] | qmm.W_STATIC, N, K, x, workspace=ws)
    assert bit_differences(c, d) == 0
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    check_tol(b, ref, bnd, TOL_FP32 if M <= 16 else TOL_BF16, "%s M=%d" % (qtype, M))

"""qmm_noalloc: the allocation-free entry point, for callers that cannot allocate device memory while
they run (its scratch lives in one device array the library owns).

Checked through the C-ABI against qmm() on the same inputs, within the tolerance the parity tests use
(the tensor-core class, 4e-3 * sum |w x| with the bound from the oracle), on two calls in a row with
different inputs — the second call runs on whatever the first left in the shared array. Shapes cover the
tensor-core path that reads a bf16 copy of x from the array, without and with a K split added inside a
cluster, and the mat-vec path that needs no scratch.
This file is collected last so that a failure here stops a run only after every other test has run.
"""
import numpy as np
import pytest

import oracle
import synthetic
import weight_quantized_matmul_fly_gb300 as qmm
from gpu_util import TOL_BF16, TOL_FP32, check_tol, dev, torch_cuda

pytestmark = pytest.mark.gpu

CASES = [
    ("Q4_K", 9728, 2560, 512),   # tensor-core path, bf16 copy of x in the array
    ("Q6_K", 1024, 2560, 100),   # tensor-core path, bf16 copy of x; K split over a cluster
    ("Q4_0", 256, 512, 7),       # mat-vec path: no scratch
]


@pytest.mark.parametrize("qtype,N,K,M", CASES)
def test_noalloc_matches_qmm_twice(qtype, N, K, M):
    torch = torch_cuda()
    qmm.build()
    need = qmm.qmm_workspace_size(qtype, N, K, M)
    assert need <= qmm.NOALLOC_SCRATCH_BYTES
    if M > 32:
        assert need >= M * K * 2          # these cases use the array
    if qtype == "Q6_K":
        assert qmm.qmm_plan_info(qtype, N, K, M)[1] > 1      # the plan splits K
    wq_h = oracle.quantize(qtype, synthetic.weights(N, K, seed=N + M))
    wq = dev(wq_h)
    tol = TOL_FP32 if M <= 16 else TOL_BF16
    for call in range(2):
        x_h = synthetic.activations(M, K, seed=100 * call + M)
        x = dev(x_h)
        y_ref = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        y_na = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        qmm.qmm(wq, qtype, N, K, x, y_ref)
        qmm.qmm_noalloc(wq, qtype, N, K, x, y_na)
        torch.cuda.synchronize()
        a, b = y_na.cpu().numpy(), y_ref.cpu().numpy()
        g = np.random.default_rng(call)
        ms = g.integers(0, M, 200)
        ns = g.integers(0, N, 200)
        _, bnd = oracle.qmm_sampled(qtype, wq_h, N, K, x_h, ms, ns)
        check_tol(a[ms, ns], b[ms, ns].astype(np.float64), bnd, tol, "noalloc vs qmm, call %d" % call)
        assert np.all(np.isfinite(a))


def test_noalloc_allocates_nothing_in_a_graph():
    """Two qmm_noalloc calls (one using the static array) captured in a CUDA graph after a warm-up call:
    replaying the graph leaves the device's free memory unchanged."""
    torch = torch_cuda()
    qmm.build()
    qtype, N, K = "Q4_K", 1024, 2560
    wq = dev(oracle.quantize(qtype, synthetic.weights(N, K, seed=3)))
    xs = [dev(synthetic.activations(M, K, seed=M)) for M in (7, 100)]
    ys = [torch.empty((x.shape[0], N), dtype=torch.float32, device="cuda") for x in xs]
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for x, y in zip(xs, ys):
            qmm.qmm_noalloc(wq, qtype, N, K, x, y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for x, y in zip(xs, ys):
            qmm.qmm_noalloc(wq, qtype, N, K, x, y)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert all(bool(torch.isfinite(y).all()) for y in ys)


def test_noalloc_refuses_oversized_scratch():
    torch = torch_cuda()
    qmm.build()
    M, N, K = 8192, 128, 8192            # bf16 copy of x alone: 128 MiB
    assert qmm.qmm_workspace_size("Q4_0", N, K, M) > qmm.NOALLOC_SCRATCH_BYTES
    wq = torch.zeros(qmm.row_bytes("Q4_0", K) * N, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), dtype=torch.float32, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_noalloc(wq, "Q4_0", N, K, x, y)
    assert e.value.code == -8

"""Failure path on the GPU without a fault: a bounded wait is made to run out on purpose (the test hook
qmm_debug_stall points one warp's first weight wait at a barrier nothing signals). The call must return
within a few seconds, the status word must carry QMM_STATUS_TIMEOUT, and the next ordinary call on the same
device must match the oracle, with a clean status word.

Nothing here faults, traps or hangs the GPU: the stalled warp gives up after about one second, waits
(bounded) for its own weight copies that are in flight, and leaves; the other warps run to completion."""
import time

import numpy as np
import pytest

import oracle
import synthetic
import weight_quantized_matmul_fly_gb300 as qmm
from gpu_util import TOL_FP32, check_tol, dev, torch_cuda, x_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("qtype,N,K,M", [("Q4_K", 256, 2560, 1), ("Q6_K", 512, 9728, 16), ("Q4_0", 64, 512, 7)])
def test_bounded_wait_runs_out_and_device_stays_usable(qtype, N, K, M):
    torch = torch_cuda()
    wq = oracle.quantize(qtype, synthetic.weights(N, K, seed=3))
    x = synthetic.activations(M, K, seed=3)
    wq_d, x_d = dev(wq), x_dev(x)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert qmm.qmm_get_status() == 0
    t0 = time.perf_counter()
    qmm.qmm_debug_stall(wq_d, qtype, N, K, x_d, y)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert 0.5 < dt < 20.0, dt
    assert qmm.qmm_get_status() & qmm.STATUS_TIMEOUT
    # the device and the library are still usable, and the next call is right
    y.fill_(float("nan"))
    qmm.qmm(wq_d, qtype, N, K, x_d, y)
    torch.cuda.synchronize()
    ref, bnd = oracle.qmm(qtype, wq, N, K, x)
    check_tol(y.cpu().numpy(), ref, bnd, TOL_FP32, "after the timeout")
    assert qmm.qmm_get_status() == 0

"""GPU decoders and encoder against the oracle, bit for bit.

Dequantization must equal the oracle's binary32 rounding of the exact formula value for every type
(the block-format specification's decoding rule), including blocks of arbitrary bytes whose scales are
NaN or infinite. The device encoder must write exactly the oracle encoder's bytes."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_util import dev, torch_cuda

pytestmark = pytest.mark.gpu
TYPES = oracle.TYPES


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("N,K", [(37, 512), (3, 1536)])
def test_dequant_bitexact(qtype, N, K):
    torch = torch_cuda()
    wq = oracle.quantize(qtype, synthetic.weights(N, K, seed=N + K))
    want = oracle.dequant_f32(qtype, wq, N, K)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    import weight_quantized_matmul_fly_gb300 as qmm
    qmm.qmm_dequant(dev(wq), qtype, N, K, out)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("qtype", TYPES)
def test_dequant_arbitrary_bytes(qtype):
    """Random bytes: every code pattern, and scales that may be NaN, infinite or subnormal."""
    torch = torch_cuda()
    import weight_quantized_matmul_fly_gb300 as qmm
    N, K = 16, 1024
    g = np.random.default_rng(7)
    wq = g.integers(0, 256, (N, oracle.row_bytes(qtype, K)), dtype=np.uint8)
    want = oracle.dequant_f32(qtype, wq, N, K)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    qmm.qmm_dequant(dev(wq), qtype, N, K, out)
    got = out.cpu().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("dist", ["normal", "uniform", "sparse"])
def test_quantize_matches_oracle(qtype, dist):
    torch = torch_cuda()
    import weight_quantized_matmul_fly_gb300 as qmm
    N, K = 24, 1024
    g = np.random.default_rng(len(dist) * 31 + len(qtype))
    if dist == "normal":
        w = synthetic.weights(N, K, seed=3)
    elif dist == "uniform":
        w = g.uniform(-2, 2, (N, K)).astype(np.float32)
    else:
        w = (0.05 * g.standard_normal((N, K))).astype(np.float32)
        w[g.random((N, K)) < 0.6] = 0
    want = oracle.quantize(qtype, w)
    out = torch.zeros(want.shape, dtype=torch.uint8, device="cuda")
    qmm.qmm_quantize(dev(w), qtype, N, K, out)
    got = out.cpu().numpy()
    assert np.array_equal(got, want), int((got != want).sum())

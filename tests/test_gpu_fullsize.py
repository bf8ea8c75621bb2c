"""Parity at the workloads' full sizes, in the launch configuration the benchmark times (qmm / qmm_ws /
qmm_id on the default stream), checked on sampled outputs that the oracle computes one by one, plus the
tile-invariance check of the all-type sweep at full size.

Workloads: one Qwen3-Embedding-4B layer (Q4_K / Q6_K, binary32 activations), the Qwen3-0.6B output head
(group-64 affine 4-bit, bf16 activations), the 128-expert narrow-K expert-indexed mat-vec, and the
13-type sweep on a 9728 x 2560 ffn_gate matrix."""
import numpy as np
import pytest

import oracle
import synthetic
import weight_quantized_matmul_fly_gb300 as qmm
from gpu_util import TOL_BF16, TOL_FP32, check_tol, dev, torch_cuda, x_dev

pytestmark = pytest.mark.gpu
SAMPLES = 384


def _sample(M, N, seed):
    g = np.random.default_rng(seed)
    ms = g.integers(0, M, SAMPLES)
    ns = g.integers(0, N, SAMPLES)
    # always include the corners and the last row / token
    ms[:4] = [0, 0, M - 1, M - 1]
    ns[:4] = [0, N - 1, 0, N - 1]
    return ms, ns


def _check_call(qtype, wq, N, K, M, seed, bf16=False):
    torch = torch_cuda()
    x = synthetic.activations(M, K, seed=seed, bf16=bf16)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    qmm.qmm(dev(wq), qtype, N, K, x_dev(x), y)
    torch.cuda.synchronize()
    ms, ns = _sample(M, N, seed)
    ref, bnd = oracle.qmm_sampled(qtype, wq, N, K, x, ms, ns)
    got = y.cpu().numpy()[ms, ns]
    tol = TOL_FP32 if M <= 16 else TOL_BF16
    return check_tol(got, ref, bnd, tol, "%s %dx%dx%d" % (qtype, M, N, K))


@pytest.mark.parametrize("name,N,K,qtype", synthetic.QWEN3_EMB_4B_LAYER)
def test_qwen3_emb_4b_layer(name, N, K, qtype):
    wq = oracle.quantize(qtype, synthetic.weights(N, K, seed=0))
    for M in (1, 2, 7, 33, 130, 2048):
        _check_call(qtype, wq, N, K, M, seed=M)


def test_qwen3_06b_lm_head():
    N, K = 151936, 1024
    wq = oracle.quantize("A4G64", synthetic.weights(N, K, seed=0))
    for M in (1, 16):
        _check_call("A4G64", wq, N, K, M, seed=M, bf16=True)


@pytest.mark.parametrize("K", synthetic.MOE_K)
def test_moe_narrow_k(K):
    torch = torch_cuda()
    E, N, topk = synthetic.MOE_EXPERTS, synthetic.MOE_ROWS, synthetic.MOE_TOPK
    wqs = [oracle.quantize("Q4_0", synthetic.weights(N, K, seed=1000 + e)) for e in range(E)]
    wd = [dev(w) for w in wqs]
    for M in (1, 24):
        x = synthetic.activations(M, K, seed=M)
        ids = synthetic.expert_ids(M, seed=M)
        y = torch.empty((M, topk, N), dtype=torch.float32, device="cuda")
        qmm.qmm_id(wd, "Q4_0", N, K, x_dev(x), dev(ids), y)
        torch.cuda.synchronize()
        # sample rows of every slot through the oracle's single-matrix sampled product
        got = y.cpu().numpy()
        g = np.random.default_rng(K + M)
        for t in range(M):
            for j in range(topk):
                ns = g.integers(0, N, 8)
                ref, bnd = oracle.qmm_sampled("Q4_0", wqs[ids[t, j]], N, K, x[t:t + 1], np.zeros(8, np.int64), ns)
                check_tol(got[t, j, ns], ref, bnd, TOL_FP32, "moe K=%d t=%d j=%d" % (K, t, j))


@pytest.mark.parametrize("qtype", synthetic.SWEEP_TYPES)
def test_type_sweep_ffn_gate(qtype):
    torch = torch_cuda()
    N, K = synthetic.SWEEP_SHAPE
    wq = oracle.quantize(qtype, synthetic.weights(N, K, seed=0))
    wd = dev(wq)
    for M in synthetic.SWEEP_TOKENS:
        _check_call(qtype, wq, N, K, M, seed=M)
        if M >= 64:
            # bit-identical across every token-tile variant at this size
            x = x_dev(synthetic.activations(M, K, seed=M))
            outs = []
            for t in (32, 64, 128):
                y = torch.empty((M, N), dtype=torch.float32, device="cuda")
                qmm.qmm_with_tile(wd, qtype, N, K, x, y, tile=t)
                outs.append(y)
            assert bool(torch.any(outs[0] != 0))
            for o in outs[1:]:
                assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32)), qtype

"""A layer's projections chained on one stream, against the oracle element by element.

- qmm_batch: matrices of one type and K that take the same activations (q/k, gate/up) in one mat-vec
  launch (M <= 16), or one qmm call after the other (M > 16).
- A Qwen3-Embedding-4B-shaped layer at reduced width (candle PR 4056, "This branch, kernel level": a layer
  timed as its seven projections back to back) captured into one CUDA graph: q/k batched, v, the output
  projection on an input computed on the GPU inside the graph, gate/up batched, and the down projection
  on silu(gate) * up computed inside the graph; replayed twice with new activations copied in. So every
  call follows a kernel that writes its input, and the chained launches' ordering is checked.
- A kernel that writes the weights immediately before a call: the call must see the new weights.
"""
import numpy as np
import pytest

import oracle
import synthetic
import weight_quantized_matmul_fly_gb300 as qmm
from gpu_util import TOL_BF16, TOL_FP32, check_tol, dev, torch_cuda, x_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("qtype", ["Q4_K", "Q4_0", "A4G64", "Q6_K"])
@pytest.mark.parametrize("M", [1, 2, 7, 16, 40])
def test_batch_shared_activations(qtype, M):
    torch = torch_cuda()
    K = 1024
    Ns = [300, 77, 520]
    bf16 = qtype == "A4G64"
    wqs = [oracle.quantize(qtype, synthetic.weights(N, K, seed=20 + i)) for i, N in enumerate(Ns)]
    x = synthetic.activations(M, K, seed=M, bf16=bf16)
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for N in Ns]
    qmm.qmm_batch([dev(w) for w in wqs], qtype, Ns, K, x_dev(x), ys)
    torch.cuda.synchronize()
    tol = TOL_FP32 if M <= 16 else TOL_BF16
    for i, (w, N) in enumerate(zip(wqs, Ns)):
        ref, bnd = oracle.qmm(qtype, w, N, K, x)
        check_tol(ys[i].cpu().numpy(), ref, bnd, tol, "%s M=%d matrix %d" % (qtype, M, i))


def test_batch_argument_errors():
    torch_cuda()
    import ctypes
    L = qmm.lib()
    P = ctypes.c_void_p
    A = 0x1000
    W = (P * 2)(A, A)
    NN = (ctypes.c_int64 * 2)(64, 64)
    Y = (P * 2)(A, A + 4)
    assert L.qmm_batch(0, ctypes.cast(W, P), ctypes.cast(NN, P), ctypes.cast(Y, P), 3, 64, P(A), 1, None) == -7
    assert L.qmm_batch(9, ctypes.cast(W, P), ctypes.cast(NN, P), ctypes.cast(Y, P), 3, 64, P(A), 1, None) == -7
    assert L.qmm_batch(2, ctypes.cast(W, P), ctypes.cast(NN, P), ctypes.cast(Y, P), 3, 64, P(A), 1, None) == -5


LAYER = [("q", 512, 768, "Q4_K"), ("k", 128, 768, "Q4_K"), ("v", 128, 768, "Q6_K"), ("o", 768, 512, "Q4_K"),
         ("gate", 1024, 768, "Q4_K"), ("up", 1024, 768, "Q4_K"), ("down", 768, 1024, "Q6_K")]


@pytest.mark.parametrize("M", [1, 7, 33])
def test_layer_graph(M):
    torch = torch_cuda()
    W = {name: oracle.quantize(qt, synthetic.weights(N, K, seed=40 + i)) for i, (name, N, K, qt) in enumerate(LAYER)}
    S = {name: (N, K, qt) for name, N, K, qt in LAYER}
    Wd = {name: dev(w) for name, w in W.items()}
    x = torch.empty((M, 768), dtype=torch.float32, device="cuda")
    y = {name: torch.empty((M, N), dtype=torch.float32, device="cuda") for name, N, K, qt in LAYER}
    att = torch.empty((M, 512), dtype=torch.float32, device="cuda")
    act = torch.empty((M, 1024), dtype=torch.float32, device="cuda")

    def layer():
        qmm.qmm_batch([Wd["q"], Wd["k"]], "Q4_K", [512, 128], 768, x, [y["q"], y["k"]])
        qmm.qmm(Wd["v"], "Q6_K", 128, 768, x, y["v"])
        # a stand-in for attention: the output projection's input written right before it
        torch.tanh(y["q"], out=att)
        qmm.qmm(Wd["o"], "Q4_K", 768, 512, att, y["o"])
        qmm.qmm_batch([Wd["gate"], Wd["up"]], "Q4_K", [1024, 1024], 768, x, [y["gate"], y["up"]])
        torch.mul(torch.nn.functional.silu(y["gate"]), y["up"], out=act)
        qmm.qmm(Wd["down"], "Q6_K", 768, 1024, act, y["down"])

    stream = torch.cuda.Stream()
    x.copy_(torch.from_numpy(synthetic.activations(M, 768, seed=1)))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        layer()                                      # warm-up: kernel attributes, plans
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer()
    tol = TOL_FP32 if M <= 16 else TOL_BF16
    for rep in range(2):
        xh = synthetic.activations(M, 768, seed=100 + rep)
        x.copy_(torch.from_numpy(xh))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ins = {"q": xh, "k": xh, "v": xh, "gate": xh, "up": xh, "o": att.cpu().numpy(), "down": act.cpu().numpy()}
        for name, (N, K, qt) in S.items():
            ref, bnd = oracle.qmm(qt, W[name], N, K, ins[name])
            check_tol(y[name].cpu().numpy(), ref, bnd, tol, "M=%d replay %d %s" % (M, rep, name))


@pytest.mark.parametrize("M", [1, 7, 40])
def test_weight_writer_immediately_before(M):
    """An ordinary kernel writes the weights and the call follows at once on the same stream: the call must
    use the new weights (before its predecessor completes it only prefetches them into L2)."""
    torch = torch_cuda()
    N, K, qt = 384, 2560, "Q4_K"
    A = oracle.quantize(qt, synthetic.weights(N, K, seed=61))
    B = oracle.quantize(qt, synthetic.weights(N, K, seed=62))
    Ad, Bd = dev(A), dev(B)
    zero = torch.zeros_like(Ad)
    wq = torch.empty_like(Ad)
    xh = synthetic.activations(M, K, seed=63)
    x = x_dev(xh)
    refs = {0: oracle.qmm(qt, A, N, K, xh), 1: oracle.qmm(qt, B, N, K, xh)}
    ys = []
    for r in range(6):
        torch.bitwise_or(Ad if r % 2 == 0 else Bd, zero, out=wq)      # the weight writer
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        qmm.qmm(wq, qt, N, K, x, y)                                   # launched right after it
        ys.append(y)
    torch.cuda.synchronize()
    tol = TOL_FP32 if M <= 16 else TOL_BF16
    for r, y in enumerate(ys):
        ref, bnd = refs[r % 2]
        check_tol(y.cpu().numpy(), ref, bnd, tol, "M=%d round %d" % (M, r))

"""Pins for the oracle's matmul y[m, n] = sum_k w[n, k] x[m, k] and its expert-indexed form.

- brute force on tiny inputs with exact rational arithmetic (every weight and activation is a dyadic
  rational, so the exact dot product is a Fraction);
- the plain types reduce to numpy's binary64 x @ W.T;
- Q8_0 with d = 1 and integer activations is an exact integer matmul;
- permuting weight rows permutes y's columns exactly; permuting tokens permutes y's rows exactly;
- the bound sum_k |w x| is numpy's |x| @ |W|.T;
- the sampled and expert-indexed entry points agree with the full product.
"""
from fractions import Fraction

import numpy as np
import pytest

import spec_fields as sf
import synthetic

QTYPES = ["Q4_0", "Q4_1", "Q5_0", "Q5_1", "Q8_0", "Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K", "A4G64"]
EPS64 = 2.0 ** -53


def _random_blocks(qtype, g, nblk):
    fields = [sf.random_fields(qtype, g) for _ in range(nblk)]
    blob = b"".join(sf.pack(qtype, f) for f in fields)
    vals = [v for f in fields for v in sf.values(qtype, f)]
    return np.frombuffer(blob, dtype=np.uint8).copy(), vals


@pytest.mark.parametrize("qtype", QTYPES)
def test_brute_force_exact_rational(orc, qtype):
    """1 x QK x 1 and 3 x 2QK x 2: the oracle's binary64 sum is within K * 2^-53 * bound of the exact
    rational dot product of the block's exact weights with the activations."""
    g = np.random.default_rng(100 + len(qtype) * 7 + sf.QK[qtype])
    qk = sf.QK[qtype]
    for (M, N, nblk_row) in [(1, 1, 1), (3, 2, 2)]:
        K = qk * nblk_row
        wq, vals = _random_blocks(qtype, g, N * nblk_row)
        x = g.standard_normal((M, K)).astype(np.float32)
        y, bnd = orc.qmm(qtype, wq, N, K, x)
        for m in range(M):
            for n in range(N):
                exact = sum(vals[n * K + k] * Fraction(float(x[m, k])) for k in range(K))
                absum = sum(abs(vals[n * K + k] * Fraction(float(x[m, k]))) for k in range(K))
                assert abs(Fraction(y[m, n]) - exact) <= K * EPS64 * absum
                assert abs(Fraction(bnd[m, n]) - absum) <= K * EPS64 * absum


@pytest.mark.parametrize("qtype", ["F32", "F16", "BF16"])
def test_plain_types_reduce_to_numpy(orc, qtype):
    g = np.random.default_rng(3)
    N, K, M = 37, 96, 5
    w = (0.02 * g.standard_normal((N, K))).astype(np.float32)
    x = g.standard_normal((M, K)).astype(np.float32)
    wq = orc.quantize(qtype, w)
    if qtype == "F32":
        W = w.astype(np.float64)
    elif qtype == "F16":
        W = w.astype(np.float16).astype(np.float64)
    else:
        import torch
        W = torch.from_numpy(w).to(torch.bfloat16).to(torch.float64).numpy()
    y, bnd = orc.qmm(qtype, wq, N, K, x)
    ref = x.astype(np.float64) @ W.T
    refb = np.abs(x.astype(np.float64)) @ np.abs(W).T
    assert np.all(np.abs(y - ref) <= 2 * K * EPS64 * refb)
    assert np.all(np.abs(bnd - refb) <= 2 * K * EPS64 * refb)


def test_q8_0_unit_scale_is_integer_matmul(orc):
    g = np.random.default_rng(8)
    N, K, M = 19, 128, 4
    codes = g.integers(-128, 128, (N, K))
    blocks = []
    for n in range(N):
        for b in range(K // 32):
            blocks.append(sf.pack("Q8_0", {"d": sf.h16(1.0), "q": [int(c) for c in codes[n, 32 * b:32 * b + 32]]}))
    wq = np.frombuffer(b"".join(blocks), dtype=np.uint8).copy()
    xi = g.integers(-50, 51, (M, K))
    y, _ = orc.qmm("Q8_0", wq, N, K, xi.astype(np.float32))
    assert np.array_equal(y, (xi @ codes.T).astype(np.float64))


@pytest.mark.parametrize("qtype", ["Q4_0", "Q4_K", "Q6_K", "A4G64"])
def test_permutation_invariance(orc, qtype):
    g = np.random.default_rng(21)
    N, K, M = 24, 2 * sf.QK[qtype] if sf.QK[qtype] > 32 else 128, 6
    w = synthetic.weights(N, K, seed=4)
    x = synthetic.activations(M, K, seed=4)
    wq = orc.quantize(qtype, w)
    y, bnd = orc.qmm(qtype, wq, N, K, x)
    pr = g.permutation(N)
    pt = g.permutation(M)
    y2, b2 = orc.qmm(qtype, np.ascontiguousarray(wq[pr]), N, K, np.ascontiguousarray(x[pt]))
    assert np.array_equal(y2, y[pt][:, pr])
    assert np.array_equal(b2, bnd[pt][:, pr])


@pytest.mark.parametrize("qtype", QTYPES)
def test_bound_is_abs_product(orc, qtype):
    N, K, M = 8, 512, 3
    w = synthetic.weights(N, K, seed=6)
    x = synthetic.activations(M, K, seed=6)
    wq = orc.quantize(qtype, w)
    W = orc.dequant_f64(qtype, wq, N, K)
    y, bnd = orc.qmm(qtype, wq, N, K, x)
    refb = np.abs(x.astype(np.float64)) @ np.abs(W).T
    assert np.all(np.abs(bnd - refb) <= 2 * K * EPS64 * refb)
    assert np.all(np.abs(y - x.astype(np.float64) @ W.T) <= 2 * K * EPS64 * refb)


def test_bf16_activations(orc):
    import torch
    N, K, M = 16, 256, 4
    w = synthetic.weights(N, K, seed=9)
    xb = synthetic.activations(M, K, seed=9, bf16=True)
    wq = orc.quantize("A4G64", w)
    W = orc.dequant_f64("A4G64", wq, N, K)
    X = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    y, bnd = orc.qmm("A4G64", wq, N, K, xb)
    refb = np.abs(X) @ np.abs(W).T
    assert np.all(np.abs(y - X @ W.T) <= 2 * K * EPS64 * refb)


def test_sampled_matches_full(orc):
    N, K, M = 40, 512, 5
    w = synthetic.weights(N, K, seed=2)
    x = synthetic.activations(M, K, seed=2)
    wq = orc.quantize("Q5_K", w) if K % 256 == 0 else None
    y, bnd = orc.qmm("Q5_K", wq, N, K, x)
    g = np.random.default_rng(0)
    ms = g.integers(0, M, 30)
    ns = g.integers(0, N, 30)
    ys, bs = orc.qmm_sampled("Q5_K", wq, N, K, x, ms, ns)
    assert np.array_equal(ys, y[ms, ns])
    assert np.array_equal(bs, bnd[ms, ns])


def test_qmm_id_matches_per_slot(orc):
    E, N, K, M, topk = 6, 20, 512, 5, 3
    wqs = [orc.quantize("Q4_0", synthetic.weights(N, K, seed=30 + e)) for e in range(E)]
    x = synthetic.activations(M, K, seed=30)
    ids = synthetic.expert_ids(M, E=E, topk=topk, seed=30)
    y, bnd = orc.qmm_id("Q4_0", wqs, N, K, x, ids)
    for t in range(M):
        for j in range(topk):
            yr, br = orc.qmm("Q4_0", wqs[ids[t, j]], N, K, x[t:t + 1])
            assert np.array_equal(y[t, j], yr[0])
            assert np.array_equal(bnd[t, j], br[0])


def test_qmm_id_bad_id_gives_nan(orc):
    E, N, K = 2, 4, 32
    wqs = [orc.quantize("Q4_0", synthetic.weights(N, K, seed=e)) for e in range(E)]
    x = synthetic.activations(1, K, seed=1)
    y, _ = orc.qmm_id("Q4_0", wqs, N, K, x, np.array([[0, 5, -1]], dtype=np.int32))
    assert np.all(np.isfinite(y[0, 0])) and np.all(np.isnan(y[0, 1])) and np.all(np.isnan(y[0, 2]))


def test_expert_ids_distinct(orc):
    ids = synthetic.expert_ids(24)
    assert ids.shape == (24, 8)
    assert all(len(set(r)) == 8 for r in ids.tolist())
    assert ids.min() >= 0 and ids.max() < 128


def test_qmm_id_slots_unit_scale_is_integer_matmul(orc):
    """Per-slot activations (x of shape M x topk x K): with Q8_0 blocks of scale 1 and integer
    activations, slot (t, j) is the exact integer product of expert ids[t, j]'s codes with its own row
    x[t, j]; a slip to the token's first row, or to the wrong expert, changes the integers."""
    g = np.random.default_rng(12)
    E, N, K, M, topk = 4, 7, 64, 3, 2
    codes = [g.integers(-128, 128, (N, K)) for _ in range(E)]
    wqs = []
    for e in range(E):
        blocks = [sf.pack("Q8_0", {"d": sf.h16(1.0), "q": [int(c) for c in codes[e][n, 32 * b:32 * b + 32]]})
                  for n in range(N) for b in range(K // 32)]
        wqs.append(np.frombuffer(b"".join(blocks), dtype=np.uint8).copy())
    xi = g.integers(-50, 51, (M, topk, K))
    ids = np.array([[0, 3], [2, 2], [1, 0]], dtype=np.int32)
    y, bnd = orc.qmm_id("Q8_0", wqs, N, K, xi.astype(np.float32), ids)
    for t in range(M):
        for j in range(topk):
            c = codes[ids[t, j]]
            assert np.array_equal(y[t, j], (c @ xi[t, j]).astype(np.float64))
            assert np.array_equal(bnd[t, j], (np.abs(c) @ np.abs(xi[t, j])).astype(np.float64))


def test_qmm_id_slots_bad_id_gives_nan(orc):
    E, N, K = 2, 4, 32
    wqs = [orc.quantize("Q4_0", synthetic.weights(N, K, seed=e)) for e in range(E)]
    x = synthetic.activations(3, K, seed=1).reshape(1, 3, K)
    y, _ = orc.qmm_id("Q4_0", wqs, N, K, x, np.array([[1, 2, -1]], dtype=np.int32))
    assert np.all(np.isfinite(y[0, 0])) and np.all(np.isnan(y[0, 1])) and np.all(np.isnan(y[0, 2]))


def test_matmul_step_alone(orc):
    """The product step on decoded weights: the plain definition checked against numpy's binary64 x @ W.T
    (within its rounding bound), and the two-step form equals the one-call form bit for bit."""
    N, K, M = 30, 512, 4
    w = synthetic.weights(N, K, seed=13)
    x = synthetic.activations(M, K, seed=13)
    wq = orc.quantize("Q4_K", w)
    W = orc.dequant_f64("Q4_K", wq, N, K)
    y, bnd = orc.matmul_f64(W, x)
    refb = np.abs(x.astype(np.float64)) @ np.abs(W).T
    assert np.all(np.abs(y - x.astype(np.float64) @ W.T) <= 2 * K * EPS64 * refb)
    y1, b1 = orc.qmm("Q4_K", wq, N, K, x)
    assert np.array_equal(y, y1) and np.array_equal(bnd, b1)

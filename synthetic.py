"""Seeded synthetic inputs and workload shapes, shared by the tests and the benchmark.

This module draws random numbers and lists shapes; it holds none of the method's arithmetic (no
quantization, no dequantization, no products). Each stream of random numbers comes from
``numpy.random.default_rng([seed, stream])`` with stream 0 = weights, 1 = activations, 2 = expert ids,
so that every consumer that asks for the same (seed, shape) gets the same numbers.

Shapes and distributions follow the workloads the pages time:
  - the seven projections of one Qwen3-Embedding-4B layer with their weight types (candle PR 4056,
    "Metal: 64-token tile for the quantized matrix-matrix kernel", section "This branch, kernel level");
  - a Qwen3-0.6B decode layer plus its lm_head, with MLX-style group-64 4-bit weights and bf16
    activations (tiny-llm PR 122, "perf: Optimize quantized matmul for small decode batches", section
    "Benchmark setup");
  - expert-indexed mat-vecs with narrow K = 512 / 768 / 1024 over 4096 rows and verify batches of up to 24
    tokens, expert ids rotated between timed batches (llama.cpp PR 28086, "metal : fix idle threads in
    mul_mv_iq3_xxs for ne00 < 1024", sections "Overview", the M4 Max table, and "Test methodology").
The real models' weights are not available; weights are N(0, 0.02) and activations N(0, 1) stand-ins.
"""
from __future__ import annotations

import numpy as np

STREAM_W, STREAM_X, STREAM_IDS = 0, 1, 2

# (name, rows N, columns K, weight type): one Qwen3-Embedding-4B layer.
QWEN3_EMB_4B_LAYER = [
    ("attn_q", 4096, 2560, "Q4_K"),
    ("attn_k", 1024, 2560, "Q4_K"),
    ("attn_v", 1024, 2560, "Q6_K"),
    ("attn_output", 2560, 4096, "Q4_K"),
    ("ffn_gate", 9728, 2560, "Q4_K"),
    ("ffn_up", 9728, 2560, "Q4_K"),
    ("ffn_down", 2560, 9728, "Q6_K"),
]
QWEN3_EMB_4B_TOKENS = [1, 2, 7, 32, 33, 64, 96, 100, 128, 130, 136, 512, 2048]
QWEN3_EMB_4B_BATCH2_TOKENS = 65     # run as a batch of two sequences of 65 tokens

# One Qwen3-0.6B decode layer with group-64 affine 4-bit weights, plus the output head.
QWEN3_06B_LAYER = [
    ("q", 2048, 1024, "A4G64"),
    ("k", 1024, 1024, "A4G64"),
    ("v", 1024, 1024, "A4G64"),
    ("o", 1024, 2048, "A4G64"),
    ("gate", 3072, 1024, "A4G64"),
    ("up", 3072, 1024, "A4G64"),
    ("down", 1024, 3072, "A4G64"),
    ("lm_head", 151936, 1024, "A4G64"),
]
QWEN3_06B_TOKENS = [1, 2, 4, 8, 16]

# Expert-indexed mat-vec with narrow K.
MOE_EXPERTS, MOE_ROWS, MOE_TOPK = 128, 4096, 8
MOE_K = [512, 768, 1024]
MOE_TOKENS = [1, 2, 4, 8, 12, 16, 24]

# All-type sweep on one ffn_gate-shaped matrix.
SWEEP_SHAPE = (9728, 2560)
SWEEP_TYPES = ["F32", "F16", "BF16", "Q4_0", "Q4_1", "Q5_0", "Q5_1", "Q8_0",
               "Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K"]
SWEEP_TOKENS = [1, 16, 64, 512, 2048]

# Small single-matrix case: Q4_0, 256 rows x 512 columns, 1 and 7 tokens.
SMALL_Q4_0 = (256, 512)
SMALL_TOKENS = [1, 7]


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def weights(N: int, K: int, seed: int = 0, scale: float = 0.02) -> np.ndarray:
    """(N, K) float32 weights drawn N(0, scale^2) in binary64, then rounded to binary32."""
    return (scale * rng(seed, STREAM_W).standard_normal((N, K))).astype(np.float32)


def activations(M: int, K: int, seed: int = 0, bf16: bool = False) -> np.ndarray:
    """(M, K) activations N(0, 1): float32, or bfloat16 bit patterns (uint16) when bf16=True.

    The bf16 patterns are the float32 values rounded to nearest-even by torch's own conversion."""
    x = rng(seed, STREAM_X).standard_normal((M, K)).astype(np.float32)
    if not bf16:
        return x
    import torch
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def expert_ids(M: int, E: int = MOE_EXPERTS, topk: int = MOE_TOPK, seed: int = 0, batch: int = 0) -> np.ndarray:
    """(M, topk) int32: for each token, topk distinct experts drawn uniformly from E.

    `batch` selects an independent table, so that timed batches can rotate through different ids."""
    g = np.random.default_rng([seed, STREAM_IDS, batch])
    return np.stack([g.choice(E, size=topk, replace=False) for _ in range(M)]).astype(np.int32)

"""The tile-invariance check must catch a tile-boundary mistake (candle PR 4056, section "Same results, bit
for bit": the page plants a mutation in its 64-token kernel and shows the test failing on 1 x 33 x 200 x 512
Q4_0). Mistakes are planted on the CPU only: the oracle computes the product once with the right
activations and once with the mistake a token tile can make at its boundary — the 33rd token (the one a
32-token tile leaves to a second tile) reading the first token's activations — and the same bit-difference
count the GPU tile-invariance test uses must flag exactly that token's 200 outputs."""
import numpy as np

import oracle
import synthetic
from gpu_util import bit_differences


def test_planted_tile_boundary_mistake_is_caught():
    N, K, M = 200, 512, 33
    wq = oracle.quantize("Q4_0", synthetic.weights(N, K, seed=0))
    x = synthetic.activations(M, K, seed=1)
    y, _ = oracle.qmm("Q4_0", wq, N, K, x)
    x_bad = x.copy()
    x_bad[32] = x[0]
    y_bad, _ = oracle.qmm("Q4_0", wq, N, K, x_bad)
    y32 = np.asarray(y, dtype=np.float32)
    d = bit_differences(np.asarray(y_bad, dtype=np.float32), y32)
    assert (d, y32.size) == (200, 6600), "%d of %d outputs differ" % (d, y32.size)
    # and the unchanged run is identical to itself, with a non-zero output (the page's guard)
    assert bit_differences(y32, np.asarray(oracle.qmm("Q4_0", wq, N, K, x)[0], dtype=np.float32)) == 0
    assert np.any(y32 != 0)

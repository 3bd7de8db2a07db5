"""The test-side tensor-core scale layout helper against the layout's
per-byte definition, on CPU."""
import numpy as np

from gpu_helpers import to_mma_layout


def test_to_mma_layout_matches_index_formula():
    rng = np.random.default_rng(0)
    for G, R, C in ((1, 128, 4), (2, 200, 21), (1, 33, 3), (3, 256, 8)):
        lin = rng.integers(1, 255, size=(G, R, C), dtype=np.uint8)
        got = to_mma_layout(lin)
        nrb, ncb = -(-R // 128), -(-C // 4)
        assert got.size == G * nrb * ncb * 512
        want = np.zeros(got.size, np.uint8)
        for g in range(G):
            for r in range(R):
                for c in range(C):
                    off = ((g * nrb + r // 128) * ncb + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
                    want[off] = lin[g, r, c]
        assert (got == want).all()

"""The full-size wire test's sampling (test_gpu_configs.py): one oracle call of
W * m elements, sample i placed in its own segment at slot segment * m + i,
gives the full problem's bits at the sampled indices (checked here against the
oracle on a whole problem, uneven segments included)."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("W,n,wire,op", [(8, 100_003, "f16", "sum"), (5, 77_777, "bf16", "avg"),
                                         (3, 4_096, "f16", "avg")])
def test_embedded_samples_match_the_full_problem(W, n, wire, op):
    rng = np.random.default_rng(W * 7 + n)
    xs = [(rng.standard_normal(n) * 10.0 ** rng.integers(-6, 3, n)).astype(np.float32)
          for _ in range(W)]
    full = oracle.allreduce_wire(xs, wire, op)[0]
    idx = np.unique(np.concatenate([rng.integers(0, n, 2000), [0, n - 1]]))
    m = idx.size
    offs = np.array([oracle.segment(n, W, j)[0] for j in range(W)])
    seg = np.searchsorted(offs, idx, side="right") - 1
    pos = seg * m + np.arange(m)
    emb = [np.zeros(W * m, np.float32) for _ in range(W)]
    for u in range(W):
        emb[u][pos] = xs[u][idx]
    got = oracle.allreduce_wire(emb, wire, op)[0][pos]
    assert got.tobytes() == full[idx].tobytes()

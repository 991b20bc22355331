"""The full-size top-K check's restatement of SINGA's top-K sparsified
allreduce (tests/parity.py) against the oracle, bit for bit, on small cases:
ties straddling the cut, negative and zero values, every K from none to all,
with and without accumulations.  (The oracle itself is pinned in
test_oracle_pins.py; this ties the restatement to it.)"""
import numpy as np
import pytest

import oracle
from parity import topk_sparse_definition


def _case(W, n, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(W)]
    if kind == "ties":  # few distinct values: long runs of equal keys at the cut
        return [(rng.integers(-3, 4, n) * 0.25).astype(np.float32) for _ in range(W)]
    if kind == "zeros":  # mostly zeros of both signs
        xs = []
        for _ in range(W):
            x = np.where(rng.random(n) < 0.9, np.float32(0.0), rng.standard_normal(n)).astype(np.float32)
            x[rng.random(n) < 0.3] *= -1  # -0.0 among them
            xs.append(x)
        return xs
    raise ValueError(kind)


@pytest.mark.parametrize("W,n,kind,frac", [
    (3, 50_003, "normal", 0.01), (3, 50_003, "normal", 0.3), (4, 4_099, "ties", 0.01),
    (4, 4_099, "ties", 0.5), (2, 10_000, "zeros", 0.2), (5, 1_000, "normal", 0.0),
    (5, 1_000, "normal", 1.0), (1, 777, "ties", 0.1)])
@pytest.mark.parametrize("with_acc", [False, True])
def test_definition_matches_oracle(W, n, kind, frac, with_acc):
    ins = _case(W, n, kind, 1000 + n + W)
    acc = _case(W, n, "normal", 7 + n) if with_acc else None
    K = int(np.ceil(np.float32(frac) * np.float32(n)))
    xs = [ins[u] + acc[u] for u in range(W)] if with_acc else ins
    want, want_acc = topk_sparse_definition(xs, K, with_acc)
    acc_o = [a.copy() for a in acc] if with_acc else None
    got, nnz = oracle.sparse_allreduce(ins, frac, True, acc_o)
    assert list(nnz) == [K] * W
    for u in range(W):
        assert got[u].tobytes() == want.tobytes()
        if with_acc:
            assert acc_o[u].tobytes() == want_acc[u].tobytes()

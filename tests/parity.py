"""Comparison helpers for the GPU parity tests (host side, numpy).

Tolerances (the pages fix none numerically; these follow from the arithmetic):

* ring order, max, allgather, fusion copies: bit-exact.  NaN compares equal to
  NaN (payloads of a sum of NaNs are not specified by IEEE 754).
* prod in the fastest order: each multiply rounds relatively, so two orders
  differ by at most 2 (W - 1) u |result| (inputs kept away from overflow and
  underflow).
* fp32 in the library's fastest order: the result and the ring-order oracle
  are two orderings of the same W - 1 fp32 additions; each is within
  gamma_{W-1} * sum_r |x_r| of the exact sum (Higham, Accuracy and Stability of
  Numerical Algorithms, eq. 4.4), so they differ by at most
  2 (W - 1) u sum_r |x_r| (u = 2^-24), and never by more than the stated
  1e-6 relative to sum_r |x_r| for W <= 8:
      |gpu - oracle| <= max(1e-6, 2 (W - 1) 2^-24) * sum_r |x_r|   (* 1/W for avg)
* bf16 in the fastest order: the fp32 results obey the bound above before the
  final cast; rounding each to bf16 adds at most one bf16 ulp between them:
      ordered-bits distance <= 1, or
      |gpu - oracle| <= fp32 bound + ulp_bf16(max(|gpu|, |oracle|)).
"""
from __future__ import annotations

import numpy as np
import torch

U32 = np.float64(2.0 ** -24)


def to_np(t: torch.Tensor) -> np.ndarray:
    """CUDA/CPU tensor -> numpy (bf16 as uint16 bit patterns)."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def widen(a: np.ndarray) -> np.ndarray:
    """fp32 or bf16-bits array -> float64 values."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _isnan(a):
    return np.isnan(widen(a))


def assert_bit_exact(got: np.ndarray, want: np.ndarray, what: str = ""):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    gn, wn = _isnan(got), _isnan(want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    bad = np.nonzero((got.view(_uint(got)) != want.view(_uint(want))) & ~gn)[0]
    assert bad.size == 0, (f"{what}: {bad.size} elements differ; first at {bad[:5]}: "
                           f"got {got[bad[:5]]} want {want[bad[:5]]}")


def _uint(a):
    return np.uint32 if a.dtype == np.float32 else np.uint16


def fp32_bound(abs_sum: np.ndarray, W: int, op: str) -> np.ndarray:
    rel = max(1e-6, 2 * (W - 1) * U32)
    b = rel * abs_sum
    return b / W if op == "avg" else b


def _ordered(b16: np.ndarray) -> np.ndarray:
    b = b16.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_close_fast(got: np.ndarray, want: np.ndarray, abs_sum: np.ndarray, W: int, op: str,
                      what: str = ""):
    """Fastest-order result against the ring-order oracle (see module doc)."""
    assert got.shape == want.shape
    if op in ("max", "min"):
        return assert_bit_exact(got, want, what)
    gn, wn = _isnan(got), _isnan(want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    g, w = widen(got), widen(want)
    ok = gn | (g == w)
    if op == "prod":
        # products: each of the W - 1 multiplies rounds relatively, so two
        # orders differ by at most 2 (W - 1) u |result| (no overflow/underflow)
        bound = 2 * (W - 1) * U32 * np.abs(w) * (1 + 4 * (W - 1) * U32)
    else:
        bound = fp32_bound(abs_sum, W, op)
    diff = np.abs(g - w)
    if got.dtype == np.float32:
        ok |= diff <= bound
    else:
        ok |= np.abs(_ordered(got) - _ordered(want)) <= 1
        mag = np.maximum(np.abs(g), np.abs(w)).astype(np.float32)
        ulp = np.spacing(mag).astype(np.float64) * 65536.0
        ok |= diff <= bound + ulp
    bad = np.nonzero(~ok)[0]
    assert bad.size == 0, (f"{what}: {bad.size} elements outside tolerance; first at {bad[:5]}: "
                           f"got {g[bad[:5]]} want {w[bad[:5]]} bound {bound[bad[:5]]}")


def abs_sum(ins_np) -> np.ndarray:
    """sum_r |x_r| per element, float64."""
    acc = np.zeros(ins_np[0].shape, np.float64)
    for a in ins_np:
        acc += np.abs(widen(a))
    return acc


def topk_sparse_definition(xs, K: int, residuals: bool):
    """SINGA's top-K sparsified allreduce (Apache SINGA, Communicator::
    topKSparsAllReduce) from its definition, for arrays of any size: each rank
    sends the K entries of x (its input plus its accumulation) with the largest
    values -- values ordered by their order-preserving 32-bit keys, equal keys by
    lower index first; every result starts at zero and receives rank 0's sent
    values, then rank 1's, and so on, one fp32 add each; a rank's new
    accumulation is x - x where it sent and x elsewhere.  The oracle reaches the
    same by sorting every rank's (index, value) pairs; this form picks the K-th
    key with a partition and so runs at full size.

    xs: W fp32 arrays x.  Returns (result, [accumulations] or None)."""
    n = xs[0].size
    result = np.zeros(n, np.float32)
    accs = [] if residuals else None
    for x in xs:
        b = x.view(np.uint32)
        key = b ^ ((b >> np.uint32(31)) * np.uint32(0x7FFFFFFF) | np.uint32(0x80000000))
        if K <= 0:
            sent = np.zeros(n, bool)
        elif K >= n:
            sent = np.ones(n, bool)
        else:
            T = np.partition(key, n - K)[n - K]  # the K-th largest key
            sent = key > T
            need = K - int(np.count_nonzero(sent))
            sent[np.flatnonzero(key == T)[:need]] = True
        result[sent] = x[sent] + result[sent]
        if residuals:
            r = x.copy()
            r[sent] = x[sent] - x[sent]
            accs.append(r)
    return result, accs

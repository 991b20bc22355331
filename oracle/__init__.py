"""CPU oracle for virtual-rank ring reduce-scatter / allgather / allreduce and
Horovod-style tensor fusion (Python face of ``oracle.c``).

TEST INFRASTRUCTURE ONLY.  The oracle is the yardstick the CUDA library is
checked against.  It shares no code with ``collective_reduction_virtual_gb300``
and the library never imports it.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference arm of ``bench.py`` may import this package.

All arithmetic lives in ``oracle.c`` (see its header for the sources followed
and the readings taken where the pages are silent).  This module only builds
the shared object with gcc and marshals numpy arrays through ctypes.  bf16
arrays are carried as ``numpy.uint16`` bit patterns.

Parity pins: every routine here is pinned in ``tests/test_oracle_pins.py``
(worked schedule table of the NCCL page, hand-derived order-sensitive
examples, exact integer sums, exact rational sums within the reordering
bound, library routines for max and bf16 rounding, and the RS/AG/AR
identities).  No routine is unpinned.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, F16 = 0, 1, 2
SUM, MAX, AVG, MIN, PROD = 0, 1, 2, 3, 4
OPS = {"sum": SUM, "max": MAX, "avg": AVG, "min": MIN, "prod": PROD}
DTYPES = {"f32": F32, "float32": F32, "bf16": BF16, "bfloat16": BF16, "f16": F16,
          "float16": F16}
NP_DTYPE = {F32: np.float32, BF16: np.uint16, F16: np.uint16}
MAX_RANKS = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def load(path: str) -> ctypes.CDLL:
    """Open an oracle shared object and declare its entry points."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    PP = ctypes.POINTER(ctypes.c_void_p)
    I64 = ctypes.c_int64
    I = ctypes.c_int
    IP = ctypes.POINTER(ctypes.c_int)
    I64P = ctypes.POINTER(ctypes.c_int64)
    L.oracle_segment.argtypes = [I64, I, I, I64P, I64P]
    L.oracle_ring_schedule.argtypes = [I, IP, IP]
    L.oracle_reduce_scatter.argtypes = [PP, PP, I, I64, I, I, IP]
    L.oracle_allgather.argtypes = [PP, PP, I, I64, I, IP]
    L.oracle_allreduce.argtypes = [PP, PP, I, I64, I, I, IP]
    L.oracle_allgatherv.argtypes = [PP, I64P, PP, I, I, IP]
    L.oracle_allreduce_sampled.argtypes = [P, I64P, I64, I64, I, I, I, IP, P]
    L.oracle_f16_from_f32.argtypes = [ctypes.c_float]
    L.oracle_f16_from_f32.restype = ctypes.c_uint16
    L.oracle_f32_from_f16.argtypes = [ctypes.c_uint16]
    L.oracle_f32_from_f16.restype = ctypes.c_float
    L.oracle_reduce_scatter_hop.argtypes = [PP, PP, I, I64, I, I, IP]
    L.oracle_allreduce_wire.argtypes = [PP, PP, I, I64, I, I, IP]
    L.oracle_sparse_allreduce.argtypes = [PP, PP, PP, I, I64, ctypes.c_float, I, I64P]
    L.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
    L.oracle_bf16_from_f32.restype = ctypes.c_uint16
    L.oracle_fuse_plan.argtypes = [I64P, I, I, I64, IP, IP]
    L.oracle_fuse_pack.argtypes = [PP, I64P, I, PP, I, I]
    L.oracle_fuse_unpack.argtypes = [PP, I64P, I, PP, I, I]
    L.oracle_fusion_allreduce.argtypes = [PP, PP, I64P, I, I, I, I, I64, PP]
    for name in ("oracle_segment", "oracle_ring_schedule", "oracle_reduce_scatter",
                 "oracle_allgather", "oracle_allreduce", "oracle_allreduce_sampled",
                 "oracle_allgatherv", "oracle_reduce_scatter_hop", "oracle_allreduce_wire",
                 "oracle_sparse_allreduce",
                 "oracle_fuse_plan", "oracle_fuse_pack", "oracle_fuse_unpack",
                 "oracle_fusion_allreduce"):
        getattr(L, name).restype = I
    return L


def lib() -> ctypes.CDLL:
    """The oracle's shared object (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load(_LIB)
    return _lib


@contextlib.contextmanager
def using(path: str):
    """Temporarily route every oracle call through another build of oracle.c
    (the mutation tests use this to check that the pins catch planted
    mistakes)."""
    global _lib
    saved = lib()
    _lib = load(path)
    try:
        yield
    finally:
        _lib = saved


# ------------------------------------------------------------------ helpers

def _code(table, v):
    return table[v] if isinstance(v, str) else int(v)


def _ptrs(arrays):
    arr = (ctypes.c_void_p * max(1, len(arrays)))()
    for i, a in enumerate(arrays):
        arr[i] = a.ctypes.data
    return arr


def _ring(user_from_ring, W):
    if user_from_ring is None:
        return None
    a = (ctypes.c_int * W)(*[int(x) for x in user_from_ring])
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed (rc={rc})")


def _contig(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != NP_DTYPE[dtype]:
        raise TypeError(f"expected {np.dtype(NP_DTYPE[dtype])} array, got {a.dtype}")
    return a


# --------------------------------------------------------------- public API

def segment(n: int, W: int, j: int) -> tuple[int, int]:
    """(offset, length) of segment j of an n-element buffer split over W ranks."""
    off, ln = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().oracle_segment(n, W, j, ctypes.byref(off), ctypes.byref(ln)), "segment")
    return off.value, ln.value


def ring_schedule(W: int, user_from_ring=None) -> np.ndarray:
    """table[s, p] = block handled by ring position p at step s."""
    tab = (ctypes.c_int * (W * W))()
    _check(lib().oracle_ring_schedule(W, _ring(user_from_ring, W), tab), "ring_schedule")
    return np.array(tab[:], dtype=np.int64).reshape(W, W)


def reduce_scatter(ins, op="sum", dtype=F32, user_from_ring=None):
    """Ring reduce-scatter of the W rank arrays ``ins``; returns W segments."""
    dtype = _code(DTYPES, dtype)
    ins = [_contig(a, dtype) for a in ins]
    W, n = len(ins), int(ins[0].size)
    outs = [np.empty(segment(n, W, j)[1], NP_DTYPE[dtype]) for j in range(W)]
    rc = lib().oracle_reduce_scatter(_ptrs(ins), _ptrs(outs), W, n, dtype,
                                     _code(OPS, op), _ring(user_from_ring, W))
    _check(rc, "reduce_scatter")
    return outs


def allgather(segs, n: int, dtype=F32, user_from_ring=None):
    """Ring allgather: segs[u] holds segment u; returns W arrays of n elements."""
    dtype = _code(DTYPES, dtype)
    segs = [_contig(a, dtype) for a in segs]
    W = len(segs)
    outs = [np.empty(n, NP_DTYPE[dtype]) for _ in range(W)]
    _check(lib().oracle_allgather(_ptrs(segs), _ptrs(outs), W, n, dtype,
                                  _ring(user_from_ring, W)), "allgather")
    return outs


def allgatherv(pieces, dtype=F32, user_from_ring=None):
    """Ring allgather with per-rank sizes: pieces[u] (any length) -> W arrays
    holding all pieces in rank order."""
    dtype = _code(DTYPES, dtype)
    pieces = [_contig(a, dtype) for a in pieces]
    W = len(pieces)
    counts = np.array([a.size for a in pieces], dtype=np.int64)
    outs = [np.empty(int(counts.sum()), NP_DTYPE[dtype]) for _ in range(W)]
    rc = lib().oracle_allgatherv(_ptrs(pieces), counts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 _ptrs(outs), W, dtype, _ring(user_from_ring, W))
    _check(rc, "allgatherv")
    return outs


def allreduce(ins, op="sum", dtype=F32, user_from_ring=None):
    """Ring allreduce (reduce-scatter then allgather); returns W arrays."""
    dtype = _code(DTYPES, dtype)
    ins = [_contig(a, dtype) for a in ins]
    W, n = len(ins), int(ins[0].size)
    outs = [np.empty(n, NP_DTYPE[dtype]) for _ in range(W)]
    _check(lib().oracle_allreduce(_ptrs(ins), _ptrs(outs), W, n, dtype, _code(OPS, op),
                                  _ring(user_from_ring, W)), "allreduce")
    return outs


def allreduce_sampled(vals, idx, n: int, op="sum", dtype=F32, user_from_ring=None):
    """Allreduce output at indices ``idx`` of an n-element problem.

    ``vals[i, u]`` is rank u's input at ``idx[i]``.  Returns one value per
    sample (the same on every rank)."""
    dtype = _code(DTYPES, dtype)
    vals = _contig(vals, dtype)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    m, W = vals.shape
    res = np.empty(m, NP_DTYPE[dtype])
    rc = lib().oracle_allreduce_sampled(
        vals.ctypes.data, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), m, n, W,
        dtype, _code(OPS, op), _ring(user_from_ring, W), res.ctypes.data)
    _check(rc, "allreduce_sampled")
    return res


def bf16_from_f32(x) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bits, element by element."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    f = lib().oracle_bf16_from_f32
    return np.array([f(float(v)) for v in x], dtype=np.uint16)


def f16_from_f32(x) -> np.ndarray:
    """Round-to-nearest-even fp32 -> IEEE binary16 bits, element by element."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    f = lib().oracle_f16_from_f32
    return np.array([f(float(v)) for v in x], dtype=np.uint16)


def f32_from_f16(h) -> np.ndarray:
    """binary16 bits -> fp32 values (exact), element by element."""
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    f = lib().oracle_f32_from_f16
    return np.array([f(int(v)) for v in h], dtype=np.float32)


def reduce_scatter_hop(ins, op="sum", dtype=BF16, user_from_ring=None):
    """Ring reduce-scatter whose buffers hold the element type: every hop
    rounds to dtype (NCCL's T-typed ThisBuffer / NextBuffer)."""
    dtype = _code(DTYPES, dtype)
    ins = [_contig(a, dtype) for a in ins]
    W, n = len(ins), int(ins[0].size)
    outs = [np.empty(segment(n, W, j)[1], NP_DTYPE[dtype]) for j in range(W)]
    rc = lib().oracle_reduce_scatter_hop(_ptrs(ins), _ptrs(outs), W, n, dtype, _code(OPS, op),
                                         _ring(user_from_ring, W))
    _check(rc, "reduce_scatter_hop")
    return outs


def allreduce_wire(ins, wire="f16", op="sum", user_from_ring=None):
    """SINGA's reduced-precision allreduce: fp32 -> wire type, ring allreduce
    in the wire type (rounding every hop), wire type -> fp32."""
    ins = [_contig(a, F32) for a in ins]
    W, n = len(ins), int(ins[0].size)
    outs = [np.empty(n, np.float32) for _ in range(W)]
    rc = lib().oracle_allreduce_wire(_ptrs(ins), _ptrs(outs), W, n, _code(DTYPES, wire),
                                     _code(OPS, op), _ring(user_from_ring, W))
    _check(rc, "allreduce_wire")
    return outs


def sparse_allreduce(ins, threshold, topk=False, accum=None):
    """SINGA's sparsified allreduce of W fp32 arrays (threshold or top-K).
    accum: W fp32 arrays updated in place (error feedback), or None.
    Returns (outputs, nnz per rank)."""
    ins = [_contig(a, F32) for a in ins]
    W, n = len(ins), int(ins[0].size)
    outs = [np.empty(n, np.float32) for _ in range(W)]
    nnz = np.zeros(W, np.int64)
    if accum is not None:
        for a in accum:
            assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == n
    rc = lib().oracle_sparse_allreduce(_ptrs(ins), _ptrs(outs),
                                       _ptrs(accum) if accum is not None else None, W, n,
                                       float(threshold), 1 if topk else 0,
                                       nnz.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    _check(rc, "sparse_allreduce")
    return outs, nnz


def fuse_plan(counts, dtype=F32, threshold_bytes=64 * 1024 * 1024) -> list[int]:
    """Greedy fusion batches; returns batch_begin (first tensor per batch, then T)."""
    dtype = _code(DTYPES, dtype)
    c = np.ascontiguousarray(counts, dtype=np.int64)
    T = int(c.size)
    begin = (ctypes.c_int * (T + 1))()
    nb = ctypes.c_int()
    rc = lib().oracle_fuse_plan(c.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), T, dtype,
                                int(threshold_bytes), begin, ctypes.byref(nb))
    _check(rc, "fuse_plan")
    return list(begin[: nb.value + 1])


def fuse_pack(tensors, counts, W: int, dtype=F32):
    """tensors[u][t] -> W fused arrays (tensors back to back, no padding)."""
    dtype = _code(DTYPES, dtype)
    c = np.ascontiguousarray(counts, dtype=np.int64)
    T = int(c.size)
    flat = [_contig(tensors[u][t], dtype) for u in range(W) for t in range(T)]
    fused = [np.empty(int(c.sum()), NP_DTYPE[dtype]) for _ in range(W)]
    rc = lib().oracle_fuse_pack(_ptrs(flat), c.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                T, _ptrs(fused), W, dtype)
    _check(rc, "fuse_pack")
    return fused


def fuse_unpack(fused, counts, dtype=F32):
    """W fused arrays -> tensors[u][t]."""
    dtype = _code(DTYPES, dtype)
    c = np.ascontiguousarray(counts, dtype=np.int64)
    T, W = int(c.size), len(fused)
    fused = [_contig(a, dtype) for a in fused]
    outs = [[np.empty(int(c[t]), NP_DTYPE[dtype]) for t in range(T)] for _ in range(W)]
    flat = [outs[u][t] for u in range(W) for t in range(T)]
    rc = lib().oracle_fuse_unpack(_ptrs(fused), c.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                  T, _ptrs(flat), W, dtype)
    _check(rc, "fuse_unpack")
    return outs


def fusion_allreduce(tensors, counts, op="avg", dtype=F32,
                     threshold_bytes=64 * 1024 * 1024):
    """Plan batches, then pack -> in-place allreduce -> unpack per batch.

    tensors[u][t]: tensor t of rank u.  Returns outs[u][t]."""
    dtype = _code(DTYPES, dtype)
    c = np.ascontiguousarray(counts, dtype=np.int64)
    T, W = int(c.size), len(tensors)
    begin = fuse_plan(c, dtype, threshold_bytes)
    biggest = max((int(c[begin[b]:begin[b + 1]].sum()) for b in range(len(begin) - 1)), default=0)
    fused = [np.empty(max(1, biggest), NP_DTYPE[dtype]) for _ in range(W)]
    flat_in = [_contig(tensors[u][t], dtype) for u in range(W) for t in range(T)]
    outs = [[np.empty(int(c[t]), NP_DTYPE[dtype]) for t in range(T)] for _ in range(W)]
    flat_out = [outs[u][t] for u in range(W) for t in range(T)]
    rc = lib().oracle_fusion_allreduce(_ptrs(flat_in), _ptrs(flat_out),
                                       c.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                       T, W, dtype, _code(OPS, op), int(threshold_bytes),
                                       _ptrs(fused))
    _check(rc, "fusion_allreduce")
    return outs

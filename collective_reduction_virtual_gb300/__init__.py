"""vcoll: virtual-rank collectives (reduce-scatter, allgather, allreduce,
tensor-fusion pack/unpack) on one GB300 GPU.

This module is a thin ctypes binding over ``libvcoll.so`` (C ABI in
``include/vcoll.h``).  It only marshals arguments -- device pointers from
``torch.Tensor.data_ptr()`` and the current CUDA stream -- every step of every
collective runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is not built, every call raises.

Two layers, same names as the C ABI:

* ``vcoll_reduce_scatter(in_ptrs, out_ptrs, W, n, dtype, op, flags, stream)``
  and friends take integer device pointers and return the status code
  (``VcollError`` is raised by the tensor layer, not here);
* ``reduce_scatter(ins, outs=None, op="sum", ring_order=False)`` and friends
  take lists of CUDA tensors (one per virtual rank) and raise ``VcollError``.
  Pinned host tensors are accepted as well: the kernels then read and write
  host memory directly over the CPU-GPU link (no staging copies).
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvcoll.so")

F32, BF16, F16 = 0, 1, 2
SUM, MAX, AVG, MIN, PROD = 0, 1, 2, 3, 4
FLAG_RING_ORDER, FLAG_STAGED, FLAG_DIRECT = 0x1, 0x2, 0x4
MAX_RANKS = 64
OK, ERR_INVALID_ARG, ERR_INVALID_TYPE, ERR_INVALID_OP, ERR_UNSUPPORTED, ERR_CUDA = range(6)
OPS = {"sum": SUM, "max": MAX, "avg": AVG, "min": MIN, "prod": PROD}
DEFAULT_FUSION_THRESHOLD = 64 * 1024 * 1024  # Horovod's tensor_fusion_threshold default

_lock = threading.Lock()
_lib = None


class VcollError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"vcoll error {status}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libvcoll.so is not built; run `python -c \"import __graft_entry__ as g; "
                    "g.build()\"` or `python collective_reduction_virtual_gb300/build.py`")
            L = ctypes.CDLL(LIB_PATH)
            PP = ctypes.POINTER(ctypes.c_void_p)
            I, I64, U, P = ctypes.c_int, ctypes.c_int64, ctypes.c_uint, ctypes.c_void_p
            I64P, IP = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int)
            for name in ("vcoll_reduce_scatter", "vcoll_allgather", "vcoll_allreduce"):
                getattr(L, name).argtypes = [PP, PP, I, I64, I, I, U, P]
                getattr(L, name).restype = I
            L.vcoll_fuse_plan.argtypes = [I64P, I, I, I64, IP, IP]
            L.vcoll_fuse_plan.restype = I
            L.vcoll_fuse_pack.argtypes = [PP, I64P, I, PP, I, I, P]
            L.vcoll_fuse_pack.restype = I
            L.vcoll_fuse_unpack.argtypes = [PP, I64P, I, PP, I, I, P]
            L.vcoll_fuse_unpack.restype = I
            L.vcoll_sparse_workspace_bytes.argtypes = [I, I64, I]
            L.vcoll_sparse_workspace_bytes.restype = ctypes.c_size_t
            L.vcoll_sparse_workspace_min_bytes.argtypes = [I, I64, I]
            L.vcoll_sparse_workspace_min_bytes.restype = ctypes.c_size_t
            L.vcoll_sparse_allreduce.argtypes = [PP, PP, PP, I, I64, ctypes.c_float, I, P, P,
                                                 ctypes.c_size_t, P]
            L.vcoll_sparse_allreduce.restype = I
            L.vcoll_sparse_allreduce_noalloc.argtypes = [PP, PP, PP, I, I64, ctypes.c_float, I, P,
                                                         P]
            L.vcoll_sparse_allreduce_noalloc.restype = I
            for name in ("vcoll_reduce_scatter_ring", "vcoll_allreduce_ring"):
                getattr(L, name).argtypes = [PP, PP, I, I64, I, I, IP, P]
                getattr(L, name).restype = I
            L.vcoll_allreduce_wire.argtypes = [PP, PP, I, I64, I, I, U, P]
            L.vcoll_allreduce_wire.restype = I
            L.vcoll_allgatherv.argtypes = [PP, I64P, PP, I, I, P]
            L.vcoll_allgatherv.restype = I
            L.vcoll_allreduce_multi.argtypes = [PP, PP, I64P, I, I, I, I, U, P]
            L.vcoll_allreduce_multi.restype = I
            L.vcoll_fusion_allreduce.argtypes = [PP, PP, I64P, I, I, I, I, U, I64, IP, P]
            L.vcoll_fusion_allreduce.restype = I
            L.vcoll_fusion_allreduce_buffered.argtypes = [PP, PP, I64P, I, PP, I64, I, I, I, U,
                                                          I64, IP, P]
            L.vcoll_fusion_allreduce_buffered.restype = I
            L.vcoll_segment.argtypes = [I64, I, I, I64P, I64P]
            L.vcoll_segment.restype = I
            L.vcoll_status_string.argtypes = [I]
            L.vcoll_status_string.restype = ctypes.c_char_p
            L.vcoll_last_error.argtypes = []
            L.vcoll_last_error.restype = ctypes.c_char_p
            L.vcoll_version.argtypes = []
            L.vcoll_version.restype = I
            L.vcoll_selftest_wait_timeout.argtypes = [U, P]
            L.vcoll_selftest_wait_timeout.restype = I
            L.vcoll_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
            L.vcoll_device_errors.restype = I
            _lib = L
    return _lib


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = int(p) if p else None
    return arr


def _i64_array(vals):
    return (ctypes.c_int64 * max(1, len(vals)))(*[int(v) for v in vals])


def last_error() -> str:
    return lib().vcoll_last_error().decode()


def status_string(status: int) -> str:
    return lib().vcoll_status_string(int(status)).decode()


def version() -> int:
    return lib().vcoll_version()


DEVICE_ERR_TIMEOUT = 0x1


def vcoll_device_errors(clear: bool = False):
    """Returns (status, flags): the current device's error word
    (DEVICE_ERR_* bits raised by kernels); synchronises the device."""
    f = ctypes.c_uint()
    rc = lib().vcoll_device_errors(ctypes.byref(f), 1 if clear else 0)
    return rc, f.value


def vcoll_selftest_wait_timeout(limit_us: int, stream=0) -> int:
    return lib().vcoll_selftest_wait_timeout(int(limit_us), stream or None)


def device_errors(clear: bool = False) -> int:
    rc, f = vcoll_device_errors(clear)
    _check(rc)
    return f


# ----------------------------------------------------------- raw C ABI layer

def vcoll_reduce_scatter(in_ptrs, out_ptrs, W, n, dtype, op, flags=0, stream=0) -> int:
    return lib().vcoll_reduce_scatter(_ptr_array(in_ptrs), _ptr_array(out_ptrs), W, n, dtype, op,
                                      flags, stream or None)


def _ring_array(user_from_ring):
    if user_from_ring is None:
        return None
    return (ctypes.c_int * max(1, len(user_from_ring)))(*[int(v) for v in user_from_ring])


def vcoll_reduce_scatter_ring(in_ptrs, out_ptrs, W, n, dtype, op, user_from_ring=None,
                              stream=0) -> int:
    return lib().vcoll_reduce_scatter_ring(_ptr_array(in_ptrs), _ptr_array(out_ptrs), W, n, dtype,
                                           op, _ring_array(user_from_ring), stream or None)


def vcoll_allreduce_ring(in_ptrs, out_ptrs, W, n, dtype, op, user_from_ring=None,
                         stream=0) -> int:
    return lib().vcoll_allreduce_ring(_ptr_array(in_ptrs), _ptr_array(out_ptrs), W, n, dtype, op,
                                      _ring_array(user_from_ring), stream or None)


def vcoll_allgather(in_ptrs, out_ptrs, W, n, dtype, op=SUM, flags=0, stream=0) -> int:
    return lib().vcoll_allgather(_ptr_array(in_ptrs), _ptr_array(out_ptrs), W, n, dtype, op,
                                 flags, stream or None)


def vcoll_allreduce_wire(in_ptrs, out_ptrs, W, n, wire, op, flags=0, stream=0) -> int:
    return lib().vcoll_allreduce_wire(_ptr_array(in_ptrs), _ptr_array(out_ptrs), W, n, wire, op,
                                      flags, stream or None)


def vcoll_sparse_workspace_bytes(W, n, topk) -> int:
    return int(lib().vcoll_sparse_workspace_bytes(W, n, 1 if topk else 0))


def vcoll_sparse_workspace_min_bytes(W, n, topk) -> int:
    return int(lib().vcoll_sparse_workspace_min_bytes(W, n, 1 if topk else 0))


def vcoll_sparse_allreduce(in_ptrs, out_ptrs, acc_ptrs, W, n, threshold, topk, nnz_ptr=0,
                           workspace=0, workspace_bytes=0, stream=0) -> int:
    return lib().vcoll_sparse_allreduce(_ptr_array(in_ptrs), _ptr_array(out_ptrs),
                                        _ptr_array(acc_ptrs) if acc_ptrs else None, W, n,
                                        float(threshold), 1 if topk else 0, nnz_ptr or None,
                                        workspace or None, workspace_bytes, stream or None)


def vcoll_sparse_allreduce_noalloc(in_ptrs, out_ptrs, acc_ptrs, W, n, threshold, topk, nnz_ptr=0,
                                   stream=0) -> int:
    """The sparsified allreduce with its top-K working memory in a fixed array
    inside the library (for callers that must not allocate device memory)."""
    return lib().vcoll_sparse_allreduce_noalloc(_ptr_array(in_ptrs), _ptr_array(out_ptrs),
                                                _ptr_array(acc_ptrs) if acc_ptrs else None, W, n,
                                                float(threshold), 1 if topk else 0,
                                                nnz_ptr or None, stream or None)


SPARSE_NOALLOC_BYTES = 1 << 20  # the fixed working memory of the no-allocation entry point


def vcoll_allgatherv(in_ptrs, counts, out_ptrs, W, dtype, stream=0) -> int:
    return lib().vcoll_allgatherv(_ptr_array(in_ptrs), _i64_array(counts), _ptr_array(out_ptrs), W,
                                  dtype, stream or None)


def vcoll_allreduce(in_ptrs, out_ptrs, W, n, dtype, op, flags=0, stream=0) -> int:
    return lib().vcoll_allreduce(_ptr_array(in_ptrs), _ptr_array(out_ptrs), W, n, dtype, op,
                                 flags, stream or None)


def vcoll_fuse_pack(tensor_ptrs, counts, T, fused_ptrs, W, dtype, stream=0) -> int:
    return lib().vcoll_fuse_pack(_ptr_array(tensor_ptrs), _i64_array(counts), T,
                                 _ptr_array(fused_ptrs), W, dtype, stream or None)


def vcoll_fuse_unpack(fused_ptrs, counts, T, tensor_ptrs, W, dtype, stream=0) -> int:
    return lib().vcoll_fuse_unpack(_ptr_array(fused_ptrs), _i64_array(counts), T,
                                   _ptr_array(tensor_ptrs), W, dtype, stream or None)


def vcoll_allreduce_multi(in_ptrs, out_ptrs, counts, T, W, dtype, op, flags=0, stream=0) -> int:
    return lib().vcoll_allreduce_multi(_ptr_array(in_ptrs), _ptr_array(out_ptrs), _i64_array(counts),
                                       T, W, dtype, op, flags, stream or None)


def vcoll_fuse_plan(counts, dtype=F32, threshold_bytes=DEFAULT_FUSION_THRESHOLD):
    """Returns (status, batch_begin list)."""
    T = len(counts)
    begin = (ctypes.c_int * (T + 1))()
    nb = ctypes.c_int()
    rc = lib().vcoll_fuse_plan(_i64_array(counts), T, dtype, int(threshold_bytes), begin,
                               ctypes.byref(nb))
    return rc, (list(begin[: nb.value + 1]) if rc == OK else [])


def vcoll_segment(n, W, j):
    """Returns (status, offset, length)."""
    off, ln = ctypes.c_int64(), ctypes.c_int64()
    rc = lib().vcoll_segment(int(n), int(W), int(j), ctypes.byref(off), ctypes.byref(ln))
    return rc, off.value, ln.value


# -------------------------------------------------------------- tensor layer

def _check(rc: int):
    if rc != OK:
        raise VcollError(rc, last_error() or status_string(rc))


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise VcollError(ERR_INVALID_TYPE, f"unsupported dtype {t.dtype}")


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_tensors(ts, what):
    for i, t in enumerate(ts):
        if not (t.is_cuda or t.is_pinned()):
            raise VcollError(ERR_INVALID_ARG,
                             f"{what}[{i}] is neither a CUDA tensor nor pinned host memory")
        if not t.is_contiguous():
            raise VcollError(ERR_INVALID_ARG, f"{what}[{i}] is not contiguous")


def segment(n: int, W: int, j: int) -> tuple[int, int]:
    rc, off, ln = vcoll_segment(n, W, j)
    _check(rc)
    return off, ln


def reduce_scatter(ins, outs=None, op="sum", ring_order=False, stream=None, flags=0,
                   user_from_ring=None):
    """ins: W CUDA tensors of n elements.  Returns W segment tensors.
    user_from_ring (W ints, the rank at each ring position): ring order on
    that ring (implies ring_order)."""
    torch = _torch()
    W, n = len(ins), ins[0].numel()
    _check_tensors(ins, "ins")
    if outs is None:
        outs = [torch.empty(segment(n, W, j)[1], dtype=ins[0].dtype, device=ins[0].device)
                for j in range(W)]
    _check_tensors(outs, "outs")
    opc = OPS[op] if isinstance(op, str) else op
    if user_from_ring is not None:
        _check(vcoll_reduce_scatter_ring([t.data_ptr() for t in ins], [t.data_ptr() for t in outs],
                                         W, n, _dtype_code(ins[0]), opc, list(user_from_ring),
                                         _stream_handle(stream)))
        return outs
    fl = flags | (FLAG_RING_ORDER if ring_order else 0)
    _check(vcoll_reduce_scatter([t.data_ptr() for t in ins], [t.data_ptr() for t in outs], W, n,
                                _dtype_code(ins[0]), opc, fl, _stream_handle(stream)))
    return outs


def allgather(segs, n: int, outs=None, stream=None, flags=0):
    """segs[j]: segment j (len_j elements).  Returns W tensors of n elements."""
    torch = _torch()
    W = len(segs)
    _check_tensors(segs, "segs")
    if outs is None:
        outs = [torch.empty(n, dtype=segs[0].dtype, device=segs[0].device) for _ in range(W)]
    _check_tensors(outs, "outs")
    _check(vcoll_allgather([t.data_ptr() for t in segs], [t.data_ptr() for t in outs], W, n,
                           _dtype_code(segs[0]), SUM, flags, _stream_handle(stream)))
    return outs


def allgatherv(pieces, outs=None, stream=None):
    """pieces[j]: rank j's tensor (any length).  Returns W tensors holding all
    pieces concatenated in rank order."""
    torch = _torch()
    W = len(pieces)
    _check_tensors(pieces, "pieces")
    counts = [p.numel() for p in pieces]
    if outs is None:
        outs = [torch.empty(sum(counts), dtype=pieces[0].dtype, device=pieces[0].device)
                for _ in range(W)]
    _check_tensors(outs, "outs")
    _check(vcoll_allgatherv([t.data_ptr() for t in pieces], counts, [t.data_ptr() for t in outs], W,
                            _dtype_code(pieces[0]), _stream_handle(stream)))
    return outs


def allreduce(ins, outs=None, op="sum", ring_order=False, stream=None, flags=0,
              user_from_ring=None):
    """ins: W CUDA tensors of n elements; outs defaults to new tensors
    (pass ``outs=ins`` for in place).  Returns outs.  user_from_ring: ring
    order on that ring (implies ring_order)."""
    torch = _torch()
    W, n = len(ins), ins[0].numel()
    _check_tensors(ins, "ins")
    if outs is None:
        outs = [torch.empty_like(t) for t in ins]
    _check_tensors(outs, "outs")
    if user_from_ring is not None:
        _check(vcoll_allreduce_ring([t.data_ptr() for t in ins], [t.data_ptr() for t in outs], W,
                                    n, _dtype_code(ins[0]), OPS[op] if isinstance(op, str) else op,
                                    list(user_from_ring), _stream_handle(stream)))
        return outs
    fl = flags | (FLAG_RING_ORDER if ring_order else 0)
    _check(vcoll_allreduce([t.data_ptr() for t in ins], [t.data_ptr() for t in outs], W, n,
                           _dtype_code(ins[0]), OPS[op] if isinstance(op, str) else op, fl,
                           _stream_handle(stream)))
    return outs


def allreduce_wire(ins, outs=None, wire="f16", op="sum", ring_order=False, stream=None):
    """SINGA's reduced-precision allreduce of W fp32 tensors: values travel
    and accumulate in fp16 (or bf16), rounding every hop; fp32 results."""
    torch = _torch()
    W, n = len(ins), ins[0].numel()
    _check_tensors(ins, "ins")
    if any(t.dtype != torch.float32 for t in ins):
        raise VcollError(ERR_INVALID_TYPE, "the wire allreduce takes fp32 tensors")
    if outs is None:
        outs = [torch.empty_like(t) for t in ins]
    _check_tensors(outs, "outs")
    wcode = {"f16": F16, "fp16": F16, "bf16": BF16}[wire] if isinstance(wire, str) else wire
    _check(vcoll_allreduce_wire([t.data_ptr() for t in ins], [t.data_ptr() for t in outs], W, n,
                                wcode, OPS[op] if isinstance(op, str) else op,
                                FLAG_RING_ORDER if ring_order else 0, _stream_handle(stream)))
    return outs


def sparse_allreduce(ins, outs=None, accum=None, threshold=0.0, topk=False, nnz=None,
                     workspace=None, stream=None):
    """SINGA's sparsified allreduce of W fp32 CUDA tensors (threshold mode, or
    top-K with K = ceil(threshold * n)).  accum: W fp32 tensors updated in
    place (error feedback) or None.  nnz: int64 CUDA tensor of W survivor
    counts (optional).  workspace: a uint8 CUDA tensor of at least
    sparse_workspace_min_bytes(W, n, topk) bytes; sparse_workspace_bytes
    (allocated here when omitted) adds room for the faster candidate path."""
    torch = _torch()
    W, n = len(ins), ins[0].numel()
    _check_tensors(ins, "ins")
    if outs is None:
        outs = [torch.empty_like(t) for t in ins]
    _check_tensors(outs, "outs")
    need = vcoll_sparse_workspace_bytes(W, n, topk)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=ins[0].device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(vcoll_sparse_allreduce([t.data_ptr() for t in ins], [t.data_ptr() for t in outs],
                                  [t.data_ptr() for t in accum] if accum is not None else None,
                                  W, n, threshold, topk, nnz.data_ptr() if nnz is not None else 0,
                                  ws_ptr, ws_bytes, _stream_handle(stream)))
    return outs


def sparse_workspace_bytes(W, n, topk=True) -> int:
    return vcoll_sparse_workspace_bytes(W, n, topk)


def sparse_workspace_min_bytes(W, n, topk=True) -> int:
    return vcoll_sparse_workspace_min_bytes(W, n, topk)


def fuse_plan(counts, dtype=F32, threshold_bytes=DEFAULT_FUSION_THRESHOLD) -> list[int]:
    rc, begin = vcoll_fuse_plan(list(counts), dtype, threshold_bytes)
    _check(rc)
    return begin


def fuse_pack(tensors, fused, stream=None):
    """tensors[u][t] -> fused[u] (back to back, no padding)."""
    W, T = len(tensors), len(tensors[0])
    counts = [tensors[0][t].numel() for t in range(T)]
    flat = [tensors[u][t] for u in range(W) for t in range(T)]
    _check_tensors(flat, "tensors")
    _check_tensors(fused, "fused")
    _check(vcoll_fuse_pack([t.data_ptr() for t in flat], counts, T, [f.data_ptr() for f in fused],
                           W, _dtype_code(fused[0]), _stream_handle(stream)))
    return fused


def fuse_unpack(fused, tensors, stream=None):
    """fused[u] -> tensors[u][t]."""
    W, T = len(tensors), len(tensors[0])
    counts = [tensors[0][t].numel() for t in range(T)]
    flat = [tensors[u][t] for u in range(W) for t in range(T)]
    _check_tensors(flat, "tensors")
    _check_tensors(fused, "fused")
    _check(vcoll_fuse_unpack([f.data_ptr() for f in fused], counts, T, [t.data_ptr() for t in flat],
                             W, _dtype_code(fused[0]), _stream_handle(stream)))
    return tensors


def allreduce_multi(tensors, outs=None, op="sum", ring_order=False, stream=None, flags=0):
    """tensors[u][t]: tensor t of rank u.  Allreduce of each rank's tensors
    taken as one concatenated buffer, written to outs[u][t] (new tensors by
    default; pass outs=tensors for in place).  One pass, no fusion buffer."""
    torch = _torch()
    W, T = len(tensors), len(tensors[0])
    if outs is None:
        outs = [[torch.empty_like(t) for t in tensors[u]] for u in range(W)]
    counts = [tensors[0][t].numel() for t in range(T)]
    flat_in = [tensors[u][t] for u in range(W) for t in range(T)]
    flat_out = [outs[u][t] for u in range(W) for t in range(T)]
    _check_tensors(flat_in, "tensors")
    _check_tensors(flat_out, "outs")
    dt = _dtype_code(flat_in[0]) if flat_in else F32
    fl = flags | (FLAG_RING_ORDER if ring_order else 0)
    _check(vcoll_allreduce_multi([t.data_ptr() for t in flat_in], [t.data_ptr() for t in flat_out],
                                 counts, T, W, dt, OPS[op] if isinstance(op, str) else op, fl,
                                 _stream_handle(stream)))
    return outs


def vcoll_fusion_allreduce(in_ptrs, out_ptrs, counts, T, W, dtype, op, flags=0,
                           threshold_bytes=DEFAULT_FUSION_THRESHOLD, stream=0):
    """Returns (status, number of batches)."""
    nb = ctypes.c_int()
    rc = lib().vcoll_fusion_allreduce(_ptr_array(in_ptrs), _ptr_array(out_ptrs), _i64_array(counts),
                                      T, W, dtype, op, flags, int(threshold_bytes),
                                      ctypes.byref(nb), stream or None)
    return rc, nb.value


def vcoll_fusion_allreduce_buffered(in_ptrs, out_ptrs, counts, T, fused_ptrs, fused_bytes, W,
                                    dtype, op, flags=0, threshold_bytes=DEFAULT_FUSION_THRESHOLD,
                                    stream=0):
    """Returns (status, number of batches)."""
    nb = ctypes.c_int()
    rc = lib().vcoll_fusion_allreduce_buffered(
        _ptr_array(in_ptrs), _ptr_array(out_ptrs), _i64_array(counts), T, _ptr_array(fused_ptrs),
        int(fused_bytes), W, dtype, op, flags, int(threshold_bytes), ctypes.byref(nb),
        stream or None)
    return rc, nb.value


class FusionPlan:
    """Device pointers of a fixed set of tensors marshalled once, so that
    repeated fusion allreduces (one per training step) cost one C call."""

    def __init__(self, tensors, outs, op="avg", ring_order=False,
                 threshold_bytes=DEFAULT_FUSION_THRESHOLD, flags=0):
        W, T = len(tensors), len(tensors[0])
        flat_in = [tensors[u][t] for u in range(W) for t in range(T)]
        flat_out = [outs[u][t] for u in range(W) for t in range(T)]
        _check_tensors(flat_in, "tensors")
        _check_tensors(flat_out, "outs")
        self.W, self.T = W, T
        self.counts = [tensors[0][t].numel() for t in range(T)]
        self._in = _ptr_array([t.data_ptr() for t in flat_in])
        self._out = _ptr_array([t.data_ptr() for t in flat_out])
        self._counts = _i64_array(self.counts)
        self.dtype = _dtype_code(flat_in[0])
        self.op = OPS[op] if isinstance(op, str) else op
        self.flags = flags | (FLAG_RING_ORDER if ring_order else 0)
        self.threshold = int(threshold_bytes)
        self._keep = (flat_in, flat_out)
        self.nbatches = 0

    def __call__(self, stream=None):
        nb = ctypes.c_int()
        _check(lib().vcoll_fusion_allreduce(self._in, self._out, self._counts, self.T, self.W,
                                            self.dtype, self.op, self.flags, self.threshold,
                                            ctypes.byref(nb), _stream_handle(stream) or None))
        self.nbatches = nb.value


def fusion_allreduce_direct(tensors, outs, op="avg", ring_order=False,
                            threshold_bytes=DEFAULT_FUSION_THRESHOLD, stream=None):
    """The same batches and bits as fusion_allreduce, straight from the
    tensors to the outputs (no fusion buffer), planned and launched in C."""
    FusionPlan(tensors, outs, op, ring_order, threshold_bytes)(stream)
    return outs


class FusionBufferPlan:
    """Horovod-style tensor fusion through fusion buffers with the device
    pointers marshalled once: each call plans the greedy batches and runs,
    per batch of two or more tensors, pack into ``fused[u]`` -> in-place
    allreduce -> unpack (a batch of one tensor is allreduced straight), all
    in one C call."""

    def __init__(self, tensors, outs, fused, op="avg", ring_order=False,
                 threshold_bytes=DEFAULT_FUSION_THRESHOLD):
        W, T = len(tensors), len(tensors[0])
        flat_in = [tensors[u][t] for u in range(W) for t in range(T)]
        flat_out = [outs[u][t] for u in range(W) for t in range(T)]
        _check_tensors(flat_in, "tensors")
        _check_tensors(flat_out, "outs")
        _check_tensors(fused, "fused")
        self.W, self.T = W, T
        self.counts = [tensors[0][t].numel() for t in range(T)]
        self._in = _ptr_array([t.data_ptr() for t in flat_in])
        self._out = _ptr_array([t.data_ptr() for t in flat_out])
        self._fused = _ptr_array([f.data_ptr() for f in fused])
        self._counts = _i64_array(self.counts)
        self.fused_bytes = min(f.numel() * f.element_size() for f in fused)
        self.dtype = _dtype_code(fused[0])
        self.op = OPS[op] if isinstance(op, str) else op
        self.flags = FLAG_RING_ORDER if ring_order else 0
        self.threshold = int(threshold_bytes)
        self._keep = (flat_in, flat_out, list(fused))
        self.nbatches = 0

    def __call__(self, stream=None):
        nb = ctypes.c_int()
        _check(lib().vcoll_fusion_allreduce_buffered(
            self._in, self._out, self._counts, self.T, self._fused, self.fused_bytes, self.W,
            self.dtype, self.op, self.flags, self.threshold, ctypes.byref(nb),
            _stream_handle(stream) or None))
        self.nbatches = nb.value


def fusion_allreduce(tensors, outs, fused, op="avg", ring_order=False,
                     threshold_bytes=DEFAULT_FUSION_THRESHOLD, stream=None):
    """Horovod-style tensor fusion through fusion buffers, one C call: plan
    greedy batches, then per batch of two or more tensors pack every rank's
    tensors into its fusion buffer ``fused[u]`` (at least the largest batch),
    allreduce the buffers in place and unpack into ``outs[u][t]``; a batch of
    one tensor is allreduced straight into its output.  (Repeated calls on
    the same tensors: FusionBufferPlan marshals the pointers once.)"""
    FusionBufferPlan(tensors, outs, fused, op, ring_order, threshold_bytes)(stream)
    return outs

"""Host-only checks of the C ABI: the library builds and loads without a GPU,
exports every entry point include/vcoll.h declares, and rejects bad
arguments with the documented status codes before touching the device.
No call here reaches a kernel launch."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vcoll.h")


@pytest.fixture(scope="module")
def v():
    from collective_reduction_virtual_gb300 import build
    build.build()
    import collective_reduction_virtual_gb300 as vc
    return vc


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vcoll_[a-z_0-9]+)\s*\(", text)))


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(v):
    names = declared_functions()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", v.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (vcoll_[a-z_0-9]+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(v.LIB_PATH)
    for n in names:
        assert getattr(lib, n)


def test_build_targets_sm103a_only():
    from collective_reduction_virtual_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("fast-math" in f or "use_fast_math" in f for f in build.NVCC_FLAGS)


def test_version_and_status_strings(v):
    assert v.version() == 200  # 0.2.0: vcoll_sparse_workspace_min_bytes added
    assert v.status_string(v.OK) == "success"
    assert "operation" in v.status_string(v.ERR_INVALID_OP)
    assert v.status_string(99) == "unknown status"


FAKE_IN = [0x100000 * (u + 1) for u in range(8)]
FAKE_OUT = [0x10000000 + 0x100000 * u for u in range(8)]


@pytest.mark.parametrize("fn", ["vcoll_reduce_scatter", "vcoll_allreduce", "vcoll_allgather"])
def test_argument_errors(v, fn):
    f = getattr(v, fn)
    # unknown op / dtype (NCCL: ncclInvalidOperation / ncclInvalidType)
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F32, 9, 0, 0) == v.ERR_INVALID_OP
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, 7, v.SUM, 0, 0) == v.ERR_INVALID_TYPE
    # rank count and size
    assert f(FAKE_IN[:1], FAKE_OUT[:1], 0, 64, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG
    assert f(FAKE_IN * 9, FAKE_OUT * 9, 65, 64, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, -1, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG
    # null and misaligned pointers
    assert f([0] + FAKE_IN[1:4], FAKE_OUT[:4], 4, 64, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG
    assert f(FAKE_IN[:4], FAKE_OUT[:3] + [0], 4, 64, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG
    assert f([FAKE_IN[0] + 2] + FAKE_IN[1:4], FAKE_OUT[:4], 4, 64, v.F32, v.SUM, 0, 0) \
        == v.ERR_INVALID_ARG
    assert "aligned" in v.last_error()
    # unknown flag bits, conflicting variant flags
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F32, v.SUM, 0x80, 0) == v.ERR_INVALID_ARG
    # empty message: success, nothing enqueued, null pointers allowed
    assert f([0] * 4, [0] * 4, 4, 0, v.F32, v.SUM, 0, 0) == v.OK


def test_conflicting_variant_flags(v):
    assert v.vcoll_allreduce(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F32, v.SUM,
                             v.FLAG_STAGED | v.FLAG_DIRECT, 0) == v.ERR_INVALID_ARG


def test_overlap_rules(v):
    n, W = 1000, 4
    # two outputs overlapping
    outs = [FAKE_OUT[0], FAKE_OUT[0] + 64, FAKE_OUT[2], FAKE_OUT[3]]
    assert v.vcoll_allreduce(FAKE_IN[:W], outs, W, n, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG
    assert "output" in v.last_error()
    # output overlapping an input at a shifted offset
    outs = [FAKE_IN[1] + 4] + FAKE_OUT[1:W]
    assert v.vcoll_allreduce(FAKE_IN[:W], outs, W, n, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG
    # reduce-scatter: out[j] aliasing in[j] one element away from NCCL's
    # in-place position in[j] + off_j must fail
    offs = [oracle.segment(n, W, j)[0] for j in range(W)]
    outs = [FAKE_IN[j] + 4 * offs[j] + 4 for j in range(W)]
    assert v.vcoll_reduce_scatter(FAKE_IN[:W], outs, W, n, v.F32, v.SUM, 0, 0) \
        == v.ERR_INVALID_ARG
    # allgather: input overlapping an output away from its own segment
    segs = [FAKE_OUT[0] + 8] + FAKE_IN[1:W]
    assert v.vcoll_allgather(segs, FAKE_OUT[:W], W, n, v.F32, v.SUM, 0, 0) == v.ERR_INVALID_ARG


def test_fuse_errors(v):
    counts = [10, 20]
    ptrs = [0x100000, 0x200000]
    assert v.vcoll_fuse_pack(ptrs, counts, 2, [0x300000], 1, 9, 0) == v.ERR_INVALID_TYPE
    assert v.vcoll_fuse_pack(ptrs, [10, -1], 2, [0x300000], 1, v.F32, 0) == v.ERR_INVALID_ARG
    assert v.vcoll_fuse_pack([0x100000, 0], counts, 2, [0x300000], 1, v.F32, 0) \
        == v.ERR_INVALID_ARG
    # overlapping tensors
    assert v.vcoll_fuse_pack([0x100000, 0x100010], counts, 2, [0x300000], 1, v.F32, 0) \
        == v.ERR_INVALID_ARG
    # fused buffer overlapping a tensor
    assert v.vcoll_fuse_unpack([0x100004], counts, 2, ptrs, 1, v.F32, 0) == v.ERR_INVALID_ARG
    # nothing to copy
    assert v.vcoll_fuse_pack([0, 0], [0, 0], 2, [0], 1, v.F32, 0) == v.OK


def test_segment_matches_oracle(v):
    rng = np.random.default_rng(1)
    for _ in range(200):
        W = int(rng.integers(1, 65))
        n = int(rng.integers(0, 10 ** 6))
        j = int(rng.integers(0, W))
        assert v.segment(n, W, j) == oracle.segment(n, W, j)
    assert v.vcoll_segment(10, 0, 0)[0] == v.ERR_INVALID_ARG
    assert v.vcoll_segment(10, 4, 4)[0] == v.ERR_INVALID_ARG


def test_fuse_plan_matches_oracle(v):
    rng = np.random.default_rng(2)
    for trial in range(50):
        T = int(rng.integers(0, 300))
        counts = list(np.round(np.exp(rng.uniform(0, 16, T))).astype(np.int64))
        thr = int(rng.integers(1, 1 << 28))
        for dt in (v.F32, v.BF16):
            assert v.fuse_plan(counts, dt, thr) == oracle.fuse_plan(counts, dt, thr)
    assert v.vcoll_fuse_plan([1, 2], 5)[0] == v.ERR_INVALID_TYPE
    assert v.vcoll_fuse_plan([1, -2], v.F32)[0] == v.ERR_INVALID_ARG


def test_product_package_does_not_touch_oracle():
    # the CUDA library and its binding never import, load or name the oracle
    pkg = os.path.join(ROOT, "collective_reduction_virtual_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                hit = re.search(r"import\s+oracle|from\s+oracle|liboracle|oracle\.(c|so)\b|oracle/",
                                text)
                assert not hit, os.path.join(dirpath, f)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import collective_reduction_virtual_gb300 as vc
    monkeypatch.setattr(vc, "_lib", None)
    monkeypatch.setattr(vc, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        vc.lib()


def test_allreduce_multi_argument_errors(v):
    ins = [0x100000 * (i + 1) for i in range(4)]    # W=2, T=2
    outs = [0x10000000 + 0x100000 * i for i in range(4)]
    f = v.vcoll_allreduce_multi
    assert f(ins, outs, [10, 20], 2, 2, v.F32, 9) == v.ERR_INVALID_OP
    assert f(ins, outs, [10, 20], 2, 2, 5, v.SUM) == v.ERR_INVALID_TYPE
    assert f(ins, outs, [10, -1], 2, 2, v.F32, v.SUM) == v.ERR_INVALID_ARG
    assert f(ins, outs, [10, 20], 2, 0, v.F32, v.SUM) == v.ERR_INVALID_ARG
    assert f([0] + ins[1:], outs, [10, 20], 2, 2, v.F32, v.SUM) == v.ERR_INVALID_ARG
    assert f([ins[0] + 2] + ins[1:], outs, [10, 20], 2, 2, v.F32, v.SUM) == v.ERR_INVALID_ARG
    # output of tensor 0 overlapping input of tensor 1 at a different fused offset
    bad = [ins[1]] + outs[1:]
    assert f(ins, bad, [10, 10], 2, 2, v.F32, v.SUM) == v.ERR_INVALID_ARG
    # two outputs overlapping
    bad = [outs[0], outs[0] + 8] + outs[2:]
    assert f(ins, bad, [10, 20], 2, 2, v.F32, v.SUM) == v.ERR_INVALID_ARG
    # empty tensors need no pointers
    assert f([0] * 4, [0] * 4, [0, 0], 2, 2, v.F32, v.SUM) == v.OK


def test_new_ops_and_allgatherv_errors(v):
    # min and prod are valid ops; 5 is not
    assert v.vcoll_allreduce([0] * 4, [0] * 4, 4, 0, v.F32, v.MIN, 0, 0) == v.OK
    assert v.vcoll_allreduce([0] * 4, [0] * 4, 4, 0, v.F32, v.PROD, 0, 0) == v.OK
    assert v.vcoll_allreduce(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F32, 5, 0, 0) == v.ERR_INVALID_OP
    f = v.vcoll_allgatherv
    assert f(FAKE_IN[:2], [10, -1], FAKE_OUT[:2], 2, v.F32) == v.ERR_INVALID_ARG
    assert f(FAKE_IN[:2], [10, 20], FAKE_OUT[:2], 2, 3) == v.ERR_INVALID_TYPE
    assert f(FAKE_IN[:2], [10, 20], FAKE_OUT[:2], 0, v.F32) == v.ERR_INVALID_ARG
    assert f([0, FAKE_IN[1]], [10, 20], FAKE_OUT[:2], 2, v.F32) == v.ERR_INVALID_ARG
    # a zero-length piece needs no pointer; an empty total is a no-op
    assert f([0, 0], [0, 0], [0, 0], 2, v.F32) == v.OK
    # piece overlapping an output away from its own offset
    assert f([FAKE_OUT[0] + 4, FAKE_IN[1]], [10, 20], FAKE_OUT[:2], 2, v.F32) == v.ERR_INVALID_ARG


def test_fusion_allreduce_errors(v):
    ins = [0x100000 * (i + 1) for i in range(4)]
    outs = [0x10000000 + 0x100000 * i for i in range(4)]
    f = v.vcoll_fusion_allreduce
    assert f(ins, outs, [10, 20], 2, 2, v.F32, 9)[0] == v.ERR_INVALID_OP
    assert f(ins, outs, [10, 20], 2, 2, 5, v.SUM)[0] == v.ERR_INVALID_TYPE
    assert f(ins, outs, [10, -1], 2, 2, v.F32, v.SUM)[0] == v.ERR_INVALID_ARG
    assert f(ins, outs, [10, 20], -1, 2, v.F32, v.SUM)[0] == v.ERR_INVALID_ARG
    rc, nb = f([0] * 4, [0] * 4, [0, 0], 2, 2, v.F32, v.SUM, 0, 64)
    assert rc == v.OK and nb == 1


def test_ring_permutation_errors(v):
    W = 4
    for f in (v.vcoll_reduce_scatter_ring, v.vcoll_allreduce_ring):
        assert f(FAKE_IN[:W], FAKE_OUT[:W], W, 64, v.F32, v.SUM, [0, 1, 1, 3]) == \
            v.ERR_INVALID_ARG
        assert "permutation" in v.last_error()
        assert f(FAKE_IN[:W], FAKE_OUT[:W], W, 64, v.F32, v.SUM, [0, 1, 2, 4]) == \
            v.ERR_INVALID_ARG
        assert f(FAKE_IN[:W], FAKE_OUT[:W], W, 64, 7, v.SUM, [0, 1, 2, 3]) == v.ERR_INVALID_TYPE
        assert f(FAKE_IN[:W], FAKE_OUT[:W], W, 64, v.F32, 9, [0, 1, 2, 3]) == v.ERR_INVALID_OP
        # n == 0 enqueues nothing
        assert f(FAKE_IN[:W], FAKE_OUT[:W], W, 0, v.F32, v.SUM, [3, 2, 1, 0]) == v.OK


def test_fusion_allreduce_buffered_errors(v):
    ins = [0x100000 * (i + 1) for i in range(4)]
    outs = [0x10000000 + 0x100000 * i for i in range(4)]
    fused = [0x20000000, 0x21000000]
    f = v.vcoll_fusion_allreduce_buffered
    assert f(ins, outs, [10, 20], 2, fused, 120, 2, v.F32, 9)[0] == v.ERR_INVALID_OP
    assert f(ins, outs, [10, 20], 2, fused, 120, 2, 5, v.SUM)[0] == v.ERR_INVALID_TYPE
    assert f(ins, outs, [10, -1], 2, fused, 120, 2, v.F32, v.SUM)[0] == v.ERR_INVALID_ARG
    assert f(ins, outs, [10, 20], 2, [0, 0], 120, 2, v.F32, v.SUM)[0] == v.ERR_INVALID_ARG
    assert f(ins, outs, [10, 20], 2, fused, -1, 2, v.F32, v.SUM)[0] == v.ERR_INVALID_ARG
    # the plan's one batch of two tensors needs 120 bytes per rank: refused
    # before anything is enqueued
    rc, _ = f(ins, outs, [10, 20], 2, fused, 119, 2, v.F32, v.SUM)
    assert rc == v.ERR_INVALID_ARG and "fusion buffer" in v.last_error()
    # zero-length tensors: nothing to do
    rc, nb = f([0] * 4, [0] * 4, [0, 0], 2, fused, 0, 2, v.F32, v.SUM, 0, 64)
    assert rc == v.OK and nb == 1


def test_allreduce_wire_errors(v):
    f = v.vcoll_allreduce_wire
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F32, v.SUM) == v.ERR_INVALID_TYPE
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, 7, v.SUM) == v.ERR_INVALID_TYPE
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F16, v.MAX) == v.ERR_UNSUPPORTED
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F16, 9) == v.ERR_INVALID_OP
    assert f(FAKE_IN[:4], FAKE_OUT[:4], 0, 64, v.F16, v.SUM) == v.ERR_INVALID_ARG
    assert f([0] * 4, [0] * 4, 4, 0, v.BF16, v.AVG) == v.OK
    # fp16 is only a wire type: the plain collectives reject it
    assert v.vcoll_allreduce(FAKE_IN[:4], FAKE_OUT[:4], 4, 64, v.F16, v.SUM, 0, 0) \
        == v.ERR_INVALID_TYPE


def test_sparse_allreduce_errors(v):
    f = v.vcoll_sparse_allreduce
    assert v.vcoll_sparse_workspace_bytes(8, 64, 0) == 0
    need = v.vcoll_sparse_workspace_bytes(8, 64, 1)
    least = v.vcoll_sparse_workspace_min_bytes(8, 64, 1)
    assert need >= least >= 8 * 2048 * 4
    assert v.vcoll_sparse_workspace_min_bytes(8, 64, 0) == 0
    # the recommended size adds, per rank, a list offset per tile of 4096
    # entries and two candidate lists of (up to) n entries
    assert need - least >= 8 * 64 * 8
    big = v.vcoll_sparse_workspace_bytes(8, 1 << 26, 1) - v.vcoll_sparse_workspace_min_bytes(8, 1 << 26, 1)
    assert big == 8 * 4 * ((1 << 26) // 4096) + 8 * 8 * ((1 << 26) // 8 + 4096)
    ins, outs = FAKE_IN[:4], FAKE_OUT[:4]
    assert f(ins, outs, None, 0, 64, 0.5, 0) == v.ERR_INVALID_ARG
    assert f(ins, outs, None, 4, -1, 0.5, 0) == v.ERR_INVALID_ARG
    assert f(ins, outs, None, 4, 64, 1.5, 1) == v.ERR_INVALID_ARG        # fraction > 1
    assert f(ins, outs, None, 4, 64, 0.5, 1, 0, 0, 0) == v.ERR_INVALID_ARG  # no workspace
    assert f(ins, outs, None, 4, 64, 0.5, 1, 0, 0x100000, 16) == v.ERR_INVALID_ARG  # too small
    assert f([ins[0] + 2] + ins[1:], outs, None, 4, 64, 0.5, 0) == v.ERR_INVALID_ARG
    # accumulation overlapping an output
    assert f(ins, outs, [outs[1]] + FAKE_OUT[4:7], 4, 64, 0.5, 0) == v.ERR_INVALID_ARG
    assert f([0] * 4, [0] * 4, None, 4, 0, 0.5, 1) == v.OK

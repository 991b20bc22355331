"""Seeded random configurations across the C ABI, each checked against the
oracle: rank counts from 1 to 64, sizes around the tile boundaries, 16-byte
phases shared or different per rank, fp32 and bf16, every op, ring and
fastest order, in place, the TMA-staged forms, allgather(v), the
reduced-precision wire allreduce, the sparsified allreduce, tensor fusion and
user ring permutations.  Ring order,
max, min and bit copies must match bit for bit; the fastest order within
the reordering bound (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
from parity import abs_sum, assert_bit_exact, assert_close_fast, to_np

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
ODT = {"f32": oracle.F32, "bf16": oracle.BF16}
WS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 17, 31, 64]
NS = [0, 1, 2, 3, 5, 17, 255, 256, 257, 1023, 4095, 4096, 4097, 8191, 8193, 65535, 65537, 100_003]


@pytest.fixture(scope="module")
def v():
    from collective_reduction_virtual_gb300 import build
    build.build()
    import collective_reduction_virtual_gb300 as vc
    return vc


def _inputs(rng, W, n, dtype, shifts, op):
    """W rank buffers of n elements; rank u's starts shifts[u] elements into
    its allocation (a 16-byte phase of its own when the shifts differ)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(int(rng.integers(1 << 30)))
    outs = []
    for u in range(W):
        if op == "prod":  # sign * 2^U(-1, 1): products stay in range
            x = torch.pow(2.0, torch.rand(n, generator=g, device="cuda") * 2 - 1)
            x = x * torch.where(torch.rand(n, generator=g, device="cuda") < 0.5, -1.0, 1.0)
        else:  # wide dynamic range, so that different orders give different bits
            x = torch.randn(n, generator=g, device="cuda") * (10.0 ** torch.randint(
                -3, 4, (n,), generator=g, device="cuda").float())
        buf = torch.empty(n + shifts[u], dtype=DT[dtype], device="cuda")
        buf[shifts[u]:] = x.to(DT[dtype])
        outs.append(buf[shifts[u]:])
    return outs


def _check(got, want, s, W, op, ring, what):
    if ring or op in ("max", "min"):
        assert_bit_exact(got, want, what)
    else:
        assert_close_fast(got, want, s, W, op, what)


@pytest.mark.parametrize("case", range(160))
def test_random_collectives(v, case):
    rng = np.random.default_rng(7000 + case)
    W = int(rng.choice(WS))
    n = int(rng.choice(NS))
    dtype = str(rng.choice(["f32", "bf16"]))
    op = str(rng.choice(["sum", "avg", "max", "min", "prod"]))
    ring = bool(rng.integers(2))
    shifts = [int(rng.integers(4))] * W if rng.integers(2) else [int(x) for x in rng.integers(0, 4, W)]
    staged = W in (2, 4, 8, 16) and n > 1000 and bool(rng.integers(2))
    flags = v.FLAG_STAGED if staged else 0
    what = f"W={W} n={n} {dtype} {op} ring={ring} shifts={shifts[:4]} staged={staged}"
    ins = _inputs(rng, W, n, dtype, shifts, op)
    ins_np = [to_np(t) for t in ins]
    s = abs_sum(ins_np) if n else np.zeros(0)  # (the avg bound divides by W itself)
    want = oracle.allreduce(ins_np, op, ODT[dtype])
    rs_want = oracle.reduce_scatter(ins_np, op, ODT[dtype])
    # reduce-scatter, then allgather of its segments
    rs = v.reduce_scatter(ins, op=op, ring_order=ring, flags=flags)
    for j in range(W):
        off, ln = oracle.segment(n, W, j)
        _check(to_np(rs[j]), rs_want[j], s[off:off + ln], W, op, ring, "RS " + what)
    ag = v.allgather(rs, n, flags=flags)
    cat = torch.cat(rs) if n else torch.empty(0, dtype=DT[dtype], device="cuda")
    for u in range(W):
        assert to_np(ag[u]).tobytes() == to_np(cat).tobytes(), "AG " + what
    # allreduce, out of place or in place
    if rng.integers(2):
        outs = [t.clone() for t in ins]
        v.allreduce(outs, outs, op=op, ring_order=ring, flags=flags)
    else:
        outs = v.allreduce(ins, op=op, ring_order=ring, flags=flags)
    for u in range(W):
        _check(to_np(outs[u]), want[u], s, W, op, ring, "AR " + what)
    if ring:
        assert to_np(outs[0]).tobytes() == to_np(cat).tobytes(), "AR = RS + AG " + what


@pytest.mark.parametrize("case", range(24))
def test_random_allgatherv(v, case):
    rng = np.random.default_rng(7500 + case)
    W = int(rng.choice(WS))
    dtype = str(rng.choice(["f32", "bf16"]))
    counts = [int(rng.choice(NS[:12])) for _ in range(W)]
    shifts = [int(x) for x in rng.integers(0, 4, W)]
    pieces = [_inputs(rng, 1, c, dtype, [shifts[j]], "sum")[0] for j, c in enumerate(counts)]
    want = oracle.allgatherv([to_np(p) for p in pieces], ODT[dtype])
    outs = v.allgatherv(pieces)
    for u in range(W):
        assert to_np(outs[u]).tobytes() == want[u].tobytes(), f"AGV W={W} counts={counts[:6]}"


@pytest.mark.parametrize("case", range(24))
def test_random_wire(v, case):
    rng = np.random.default_rng(7700 + case)
    W = int(rng.choice(WS[:-1]))
    n = int(rng.choice(NS[1:]))
    wire = str(rng.choice(["f16", "bf16"]))
    op = str(rng.choice(["sum", "avg"]))
    shifts = [int(x) for x in rng.integers(0, 4, W)] if rng.integers(2) else [0] * W
    ins = _inputs(rng, W, n, "f32", shifts, "sum")
    ins_np = [to_np(t) for t in ins]
    want = oracle.allreduce_wire(ins_np, wire, op)
    ring = v.allreduce_wire(ins, wire=wire, op=op, ring_order=True)
    for u in range(W):
        assert_bit_exact(to_np(ring[u]), want[u], f"wire W={W} n={n} {wire} {op}")


@pytest.mark.parametrize("case", range(40))
def test_random_sparse(v, case):
    rng = np.random.default_rng(7900 + case)
    W = int(rng.choice(WS))
    n = int(rng.choice(NS[1:]))
    topk = bool(rng.integers(4))  # mostly top-K
    frac = float(rng.choice([0.0, 0.001, 0.01, 0.05, 0.2, 0.3, 0.7, 1.0])) if topk else float(rng.choice([0.0, 0.5, 1.5]))
    with_acc = bool(rng.integers(2))
    ws_kind = str(rng.choice(["full", "min", "between"]))
    shifts = [int(x) for x in rng.integers(0, 4, W)] if rng.integers(2) else [0] * W
    ins = _inputs(rng, W, n, "f32", shifts, "sum")
    acc = [t * 0.3 for t in _inputs(rng, W, n, "f32", shifts, "sum")] if with_acc else None
    ins_np = [to_np(t) for t in ins]
    acc_np = [to_np(a).copy() for a in acc] if acc is not None else None
    want, want_nnz = oracle.sparse_allreduce(ins_np, frac, topk, acc_np)
    ws = None
    if topk:
        lo = v.sparse_workspace_min_bytes(W, n, True)
        hi = v.sparse_workspace_bytes(W, n, True)
        nbytes = {"full": hi, "min": lo, "between": (lo + (hi - lo) // 5 + 15) // 16 * 16}[ws_kind]
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    nnz = torch.empty(W, dtype=torch.int64, device="cuda")
    outs = v.sparse_allreduce(ins, accum=acc, threshold=frac, topk=topk, nnz=nnz, workspace=ws)
    torch.cuda.synchronize()
    what = f"W={W} n={n} topk={topk} frac={frac} acc={with_acc} ws={ws_kind} shifts={shifts[:4]}"
    for u in range(W):
        assert_bit_exact(to_np(outs[u]), want[u], "sparse out " + what)
        if acc is not None:
            assert_bit_exact(to_np(acc[u]), acc_np[u], "sparse accum " + what)
    assert nnz.cpu().tolist() == list(want_nnz), "sparse nnz " + what


@pytest.mark.parametrize("case", range(24))
def test_random_fusion(v, case):
    # Horovod tensor fusion: random tensor lists (empty and one-element
    # tensors among them, each tensor at its own 16-byte phase), a threshold
    # that makes several batches, through the fusion buffers and in one pass
    rng = np.random.default_rng(8100 + case)
    W = int(rng.choice([1, 2, 3, 4, 8, 16]))
    T = int(rng.integers(1, 60))
    dtype = str(rng.choice(["f32", "bf16"]))
    op = str(rng.choice(["sum", "avg", "max", "min"]))
    ring = bool(rng.integers(2))
    counts = [int(rng.choice([0, 1, 2, 3, 5, 17, 255, 1023, 4097, 20000])) for _ in range(T)]
    es = 4 if dtype == "f32" else 2
    thr = int(rng.choice([64, 4096, 40_000, 1 << 26])) * es
    g = torch.Generator(device="cuda")
    g.manual_seed(int(rng.integers(1 << 30)))
    tens = []
    for u in range(W):
        row = []
        for c in counts:
            sh = int(rng.integers(4))
            base = torch.randn(c + 4, generator=g, device="cuda") * (10.0 ** torch.randint(
                -2, 3, (c + 4,), generator=g, device="cuda").float())
            row.append(base.to(DT[dtype])[sh:sh + c])
        tens.append(row)
    begin = oracle.fuse_plan(counts, ODT[dtype], thr)
    biggest = max(sum(counts[begin[b]:begin[b + 1]]) for b in range(len(begin) - 1))
    fused = [torch.empty(max(1, biggest), dtype=DT[dtype], device="cuda") for _ in range(W)]
    outs = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    v.fusion_allreduce(tens, outs, fused, op=op, ring_order=ring, threshold_bytes=thr)
    one = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    v.FusionPlan(tens, one, op=op, ring_order=ring, threshold_bytes=thr)()
    what = f"W={W} T={T} {dtype} {op} ring={ring} thr={thr}"
    for u in range(W):
        for t in range(T):
            assert to_np(one[u][t]).tobytes() == to_np(outs[u][t]).tobytes(), f"one pass vs pipeline {what} {t}"
    if ring or op in ("max", "min"):
        want = oracle.fusion_allreduce([[to_np(x) for x in tens[u]] for u in range(W)], counts, op,
                                       ODT[dtype], thr)
        for u in range(W):
            for t in range(T):
                assert_bit_exact(to_np(outs[u][t]), want[u][t], f"fusion {what} tensor {t}")


@pytest.mark.parametrize("case", range(16))
def test_random_user_ring(v, case):
    # the ring order of a permuted ring (NCCL userFromRing)
    rng = np.random.default_rng(8300 + case)
    W = int(rng.choice([2, 3, 4, 5, 8, 12, 16, 64]))
    n = int(rng.choice(NS[1:]))
    dtype = str(rng.choice(["f32", "bf16"]))
    op = str(rng.choice(["sum", "avg", "prod"]))
    ring = [int(x) for x in rng.permutation(W)]
    shifts = [int(x) for x in rng.integers(0, 4, W)] if rng.integers(2) else [0] * W
    ins = _inputs(rng, W, n, dtype, shifts, op)
    ins_np = [to_np(t) for t in ins]
    want = oracle.allreduce(ins_np, op, ODT[dtype], ring)
    rs_want = oracle.reduce_scatter(ins_np, op, ODT[dtype], ring)
    ar = v.allreduce(ins, op=op, user_from_ring=ring)
    rs = v.reduce_scatter(ins, op=op, user_from_ring=ring)
    what = f"W={W} n={n} {dtype} {op} ring={ring[:6]}"
    for u in range(W):
        assert_bit_exact(to_np(ar[u]), want[u], "AR " + what)
        assert_bit_exact(to_np(rs[u]), rs_want[u], "RS " + what)

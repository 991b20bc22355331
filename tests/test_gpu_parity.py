"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded bytes.

Ring order, max and allgather must be bit-exact; the fastest order must stay
within the tolerance derived in tests/parity.py.  Sizes span several tiles
and ragged tails; edge cases cover n = 0, n < W, W = 1, uneven segments,
misaligned pointers (shared and mixed 16-byte phases), in-place forms, guard
bands around every output, and non-default streams.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import abs_sum, assert_bit_exact, assert_close_fast, to_np

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
ODT = {"f32": oracle.F32, "bf16": oracle.BF16}


@pytest.fixture(scope="module")
def v():
    from collective_reduction_virtual_gb300 import build
    build.build()
    import collective_reduction_virtual_gb300 as vc
    return vc


def make_inputs(W, n, dtype, seed, dev="cuda", kind="normal"):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    outs = []
    for _ in range(W):
        if kind == "normal":
            x = torch.randn(n, generator=g, device=dev) * (10.0 ** torch.randint(
                -3, 4, (n,), generator=g, device=dev).float())
        else:
            x = torch.rand(n, generator=g, device=dev) * 2 - 1
        outs.append(x.to(DT[dtype]))
    return outs


SMALL_W = [1, 2, 3, 4, 5, 8, 16, 64]
SMALL_N = [0, 1, 3, 17, 4099, 65541]


@pytest.mark.parametrize("W", SMALL_W)
@pytest.mark.parametrize("n", SMALL_N)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_allreduce_small(v, W, n, dtype):
    ins = make_inputs(W, n, dtype, 1000 * W + n)
    ins_np = [to_np(t) for t in ins]
    for op in ("sum", "max", "avg"):
        want = oracle.allreduce(ins_np, op, ODT[dtype])
        for ring in (True, False):
            outs = v.allreduce(ins, op=op, ring_order=ring)
            got = [to_np(t) for t in outs]
            if ring or op == "max":
                for u in range(W):
                    assert_bit_exact(got[u], want[u], f"AR {op} ring={ring} W={W} n={n}")
            else:
                s = abs_sum(ins_np)
                for u in range(W):
                    assert_close_fast(got[u], want[u], s, W, op, f"AR {op} W={W} n={n}")
            for u in range(1, W):  # every rank holds the same bits
                assert got[u].tobytes() == got[0].tobytes()


@pytest.mark.parametrize("W", SMALL_W)
@pytest.mark.parametrize("n", SMALL_N)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_small(v, W, n, dtype):
    ins = make_inputs(W, n, dtype, 2000 * W + n)
    ins_np = [to_np(t) for t in ins]
    s = abs_sum(ins_np)
    for op in ("sum", "max", "avg"):
        want = oracle.reduce_scatter(ins_np, op, ODT[dtype])
        for ring in (True, False):
            outs = v.reduce_scatter(ins, op=op, ring_order=ring)
            for j in range(W):
                off, ln = oracle.segment(n, W, j)
                g = to_np(outs[j])
                assert g.size == ln
                if ring or op == "max":
                    assert_bit_exact(g, want[j], f"RS {op} ring={ring} W={W} n={n} seg {j}")
                else:
                    assert_close_fast(g, want[j], s[off:off + ln], W, op, f"RS {op} W={W} n={n}")


@pytest.mark.parametrize("W", SMALL_W)
@pytest.mark.parametrize("n", SMALL_N)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_allgather_small(v, W, n, dtype):
    segs = [make_inputs(1, oracle.segment(n, W, j)[1], dtype, 3000 * W + n + j)[0]
            for j in range(W)]
    want = oracle.allgather([to_np(s) for s in segs], n, ODT[dtype])
    outs = v.allgather(segs, n)
    for u in range(W):
        assert_bit_exact(to_np(outs[u]), want[u], f"AG W={W} n={n} rank {u}")


def test_ring_order_is_observable_on_gpu(v):
    # the hand-derived example: ring order gives 0 1 0 1, and the library's
    # ring mode must reproduce it exactly
    x = [torch.full((4,), val, device="cuda") for val in (1e8, 1.0, -1e8, 1.0)]
    outs = v.reduce_scatter(x, op="sum", ring_order=True)
    assert [float(o[0]) for o in outs] == [0.0, 1.0, 0.0, 1.0]
    ar = v.allreduce(x, op="sum", ring_order=True)
    assert all(o.tolist() == [0.0, 1.0, 0.0, 1.0] for o in ar)


# ------------------------------------------------------- alignment & layout

def _views(W, n, dtype, shifts, seed):
    """W tensors of n elements placed at the given element shifts inside
    larger allocations (to control 16-byte phases)."""
    base = make_inputs(W, n + 16, dtype, seed)
    return [b[s:s + n] for b, s in zip(base, shifts)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shift_kind", ["same", "mixed"])
@pytest.mark.parametrize("W", [3, 4, 8])
def test_misaligned_buffers(v, dtype, shift_kind, W):
    n = 50_001
    if shift_kind == "same":
        shifts = [1] * W
    else:
        shifts = [(u * 3) % 8 for u in range(W)]
    ins = _views(W, n, dtype, shifts, 77 + W)
    ins_np = [to_np(t) for t in ins]
    s = abs_sum(ins_np)
    obase = [torch.empty(n + 16, dtype=DT[dtype], device="cuda") for _ in range(W)]
    outs = [b[sh:sh + n] for b, sh in zip(obase, reversed(shifts))]
    for op in ("sum", "avg", "max"):
        want = oracle.allreduce(ins_np, op, ODT[dtype])
        for ring in (True, False):
            v.allreduce(ins, outs, op=op, ring_order=ring)
            for u in range(W):
                g = to_np(outs[u])
                if ring or op == "max":
                    assert_bit_exact(g, want[u], f"AR misaligned {shift_kind} {op}")
                else:
                    assert_close_fast(g, want[u], s, W, op, f"AR misaligned {shift_kind} {op}")
        rs_want = oracle.reduce_scatter(ins_np, op, ODT[dtype])
        rs_out = [b[1:1 + oracle.segment(n, W, j)[1]] for j, b in enumerate(obase)]
        v.reduce_scatter(ins, rs_out, op=op, ring_order=True)
        for j in range(W):
            assert_bit_exact(to_np(rs_out[j]), rs_want[j], f"RS misaligned {shift_kind} {op}")
    segs = [ins[j][:oracle.segment(n, W, j)[1]] for j in range(W)]
    ag_want = oracle.allgather([to_np(t) for t in segs], n, ODT[dtype])
    v.allgather(segs, n, outs)
    for u in range(W):
        assert_bit_exact(to_np(outs[u]), ag_want[u], f"AG misaligned {shift_kind}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_guard_bands_untouched(v, dtype):
    W, n, G = 5, 12_345, 64
    ins = make_inputs(W, n, dtype, 5)
    fill = torch.tensor([-1], dtype=torch.int16 if dtype == "bf16" else torch.int32)
    big = [torch.empty(n + 2 * G, dtype=DT[dtype], device="cuda") for _ in range(W)]
    for b in big:
        b.view(fill.dtype).fill_(-1)
    for kind in ("ar", "rs", "ag"):
        for b in big:
            b.view(fill.dtype).fill_(-1)
        if kind == "ar":
            outs = [b[G:G + n] for b in big]
            v.allreduce(ins, outs, op="sum")
        elif kind == "rs":
            outs = [b[G:G + oracle.segment(n, W, j)[1]] for j, b in enumerate(big)]
            v.reduce_scatter(ins, outs, op="avg", ring_order=True)
        else:
            segs = [ins[j][:oracle.segment(n, W, j)[1]] for j in range(W)]
            outs = [b[G:G + n] for b in big]
            v.allgather(segs, n, outs)
        torch.cuda.synchronize()
        for b, o in zip(big, outs):
            raw = b.view(fill.dtype).cpu()
            end = G + o.numel()
            assert bool((raw[:G] == -1).all()), f"{kind}: front guard written"
            assert bool((raw[end:] == -1).all()), f"{kind}: back guard written"


# ------------------------------------------------------------- in place

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [2, 4, 7, 8, 16])
def test_in_place(v, dtype, W):
    n = 100_003
    ins = make_inputs(W, n, dtype, 900 + W)
    ins_np = [to_np(t) for t in ins]
    want = oracle.allreduce(ins_np, "sum", ODT[dtype])
    bufs = [t.clone() for t in ins]
    v.allreduce(bufs, bufs, op="sum", ring_order=True)  # Horovod's in-place fusion allreduce
    for u in range(W):
        assert_bit_exact(to_np(bufs[u]), want[u], "AR in place")
    # NCCL in-place reduce-scatter: out[j] = in[j] + off_j
    bufs = [t.clone() for t in ins]
    outs = []
    for j in range(W):
        off, ln = oracle.segment(n, W, j)
        outs.append(bufs[j][off:off + ln])
    rs_want = oracle.reduce_scatter(ins_np, "sum", ODT[dtype])
    v.reduce_scatter(bufs, outs, op="sum", ring_order=True)
    for j in range(W):
        assert_bit_exact(to_np(outs[j]), rs_want[j], "RS in place")
    # in-place allgather: segment j already sits at its place in out[j]
    full = [torch.empty(n, dtype=DT[dtype], device="cuda") for _ in range(W)]
    segs = []
    for j in range(W):
        off, ln = oracle.segment(n, W, j)
        full[j][off:off + ln].copy_(outs[j])
        segs.append(full[j][off:off + ln])
    v.allgather(segs, n, full)
    for u in range(W):
        assert_bit_exact(to_np(full[u]), want[u], "AG in place")


def test_non_default_stream(v):
    W, n = 8, 1 << 20
    ins = make_inputs(W, n, "f32", 31)
    want = oracle.allreduce([to_np(t) for t in ins], "sum", oracle.F32)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        outs = [torch.empty_like(t) for t in ins]
        v.allreduce(ins, outs, op="sum", ring_order=True, stream=s)
    s.synchronize()
    for u in range(W):
        assert_bit_exact(to_np(outs[u]), want[u], "AR on side stream")


def test_cuda_graph_capture(v):
    # the small-message path is timed inside CUDA graphs: capture must work
    W, n = 8, 4096
    ins = make_inputs(W, n, "f32", 41)
    outs = [torch.empty_like(t) for t in ins]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        v.allreduce(ins, outs, op="sum", ring_order=True, stream=s)  # warm the caches
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        v.allreduce(ins, outs, op="sum", ring_order=True, stream=s)
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    want = oracle.allreduce([to_np(t) for t in ins], "sum", oracle.F32)
    for u in range(W):
        assert_bit_exact(to_np(outs[u]), want[u], "AR graph replay")


# ---------------------------------------------------------------- fusion

# W = 2, 4, 8, 16 copy all ranks of a tile together when the ranks' buffers
# share their 16-byte phases ("same"), rank by rank otherwise ("mixed": the
# fused buffers and the tensors of each rank at their own offsets); W = 5
# always goes rank by rank.
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W,phases", [(5, "same"), (2, "same"), (4, "same"), (8, "same"),
                                      (16, "same"), (4, "mixed"), (8, "mixed")])
def test_fuse_pack_unpack(v, dtype, W, phases):
    rng = np.random.default_rng(3)
    counts = [int(c) for c in rng.integers(0, 5000, 150 if W <= 8 else 60)] + [1, 2, 3, 0, 7]
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    if phases == "same":
        tens = [[torch.randn(c, generator=g, device="cuda").to(DT[dtype]) for c in counts]
                for _ in range(W)]
    else:  # each rank's tensors start at their own element offset
        tens = [[torch.randn(c + 7, generator=g, device="cuda").to(DT[dtype])[(u + t) % 7:(u + t) % 7 + c]
                 for t, c in enumerate(counts)] for u in range(W)]
    total = sum(counts)
    shift = (lambda u: 1) if phases == "same" else (lambda u: u % 8)
    fused = [torch.empty(total + 8, dtype=DT[dtype], device="cuda")[shift(u):shift(u) + total]
             for u in range(W)]
    v.fuse_pack(tens, fused)
    want = oracle.fuse_pack([[to_np(t) for t in tens[u]] for u in range(W)], counts, W, ODT[dtype])
    for u in range(W):
        assert_bit_exact(to_np(fused[u]), want[u], f"pack rank {u}")
    back = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    v.fuse_unpack(fused, back)
    for u in range(W):
        for t in range(len(counts)):
            assert to_np(back[u][t]).tobytes() == to_np(tens[u][t]).tobytes()


def test_fusion_allreduce_small(v):
    W = 8
    counts = [1000, 3, 4097, 250, 1, 60, 12345, 7]
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    tens = [[torch.randn(c, generator=g, device="cuda") * 1e-3 for c in counts] for _ in range(W)]
    thr = 4 * 5000
    outs = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    fused = [torch.empty(max(counts) + 5000, device="cuda") for _ in range(W)]
    v.fusion_allreduce(tens, outs, fused, op="avg", ring_order=True, threshold_bytes=thr)
    want = oracle.fusion_allreduce([[to_np(t) for t in tens[u]] for u in range(W)], counts, "avg",
                                   oracle.F32, thr)
    for u in range(W):
        for t in range(len(counts)):
            assert_bit_exact(to_np(outs[u][t]), want[u][t], f"fusion rank {u} tensor {t}")


# ------------------------------------------------- staged (TMA) variant

@pytest.mark.parametrize("W", [2, 4, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [40_000, 1_000_003, (1 << 22) + 12])
def test_staged_matches_direct_and_oracle(v, W, dtype, n):
    ins = make_inputs(W, n, dtype, 5000 * W + n)
    ins_np = [to_np(t) for t in ins]
    assert v.device_errors(clear=True) == 0
    for op in ("sum", "avg", "max"):
        want = oracle.allreduce(ins_np, op, ODT[dtype])
        for ring in (True, False):
            d = v.allreduce(ins, op=op, ring_order=ring, flags=v.FLAG_DIRECT)
            s = v.allreduce(ins, op=op, ring_order=ring, flags=v.FLAG_STAGED)
            for u in range(W):
                assert to_np(s[u]).tobytes() == to_np(d[u]).tobytes(), f"AR staged {op} {ring}"
            if ring or op == "max":
                assert_bit_exact(to_np(s[0]), want[0], f"AR staged {op}")
            rs_d = v.reduce_scatter(ins, op=op, ring_order=ring, flags=v.FLAG_DIRECT)
            rs_s = v.reduce_scatter(ins, op=op, ring_order=ring, flags=v.FLAG_STAGED)
            for j in range(W):
                assert to_np(rs_s[j]).tobytes() == to_np(rs_d[j]).tobytes(), f"RS staged {op}"
    assert v.device_errors(clear=True) == 0


def test_staged_in_place_and_phase(v):
    W, n = 8, 3_000_001
    base = make_inputs(W, n + 8, "f32", 71)
    ins = [b[2:2 + n] for b in base]  # shared non-zero 16-byte phase
    want = oracle.allreduce([to_np(t) for t in ins], "sum", oracle.F32)
    v.allreduce(ins, ins, op="sum", ring_order=True, flags=v.FLAG_STAGED)
    for u in range(W):
        assert_bit_exact(to_np(ins[u]), want[u], "staged in place")
    assert v.device_errors(clear=True) == 0


# --------------------------------------- multi-tensor allreduce (no buffer)

def _tensor_list(W, counts, dtype, seed, shift_pattern=None):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = []
    for u in range(W):
        row = []
        for i, c in enumerate(counts):
            sh = 0 if shift_pattern is None else shift_pattern(u, i)
            base = (torch.randn(c + 8, generator=g, device="cuda") *
                    (10.0 ** torch.randint(-2, 3, (c + 8,), generator=g, device="cuda").float()))
            row.append(base.to(DT[dtype])[sh:sh + c])
        out.append(row)
    return out


@pytest.mark.parametrize("W", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["aligned", "shared_shift", "mixed"])
def test_allreduce_multi_matches_pipeline_and_oracle(v, W, dtype, layout):
    counts = [1000, 3, 0, 4097, 250, 1, 60, 12345, 7, 77]
    pat = {"aligned": None, "shared_shift": lambda u, i: i % 4,
           "mixed": lambda u, i: (u + i) % 5}[layout]
    tens = _tensor_list(W, counts, dtype, 300 + W, pat)
    tot = sum(counts)
    fused = [torch.empty(tot, dtype=DT[dtype], device="cuda") for _ in range(W)]
    for op in ("sum", "avg", "max"):
        for ring in (True, False):
            direct = v.allreduce_multi(tens, op=op, ring_order=ring)
            outs = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
            v.fusion_allreduce(tens, outs, fused, op=op, ring_order=ring,
                               threshold_bytes=1 << 40)
            for u in range(W):
                for t in range(len(counts)):
                    assert to_np(direct[u][t]).tobytes() == to_np(outs[u][t]).tobytes(), \
                        f"multi vs pipeline {op} ring={ring} rank {u} tensor {t}"
            if ring or op == "max":
                want = oracle.fusion_allreduce(
                    [[to_np(t) for t in tens[u]] for u in range(W)], counts, op, ODT[dtype],
                    threshold_bytes=1 << 40)
                for u in range(W):
                    for t in range(len(counts)):
                        assert_bit_exact(to_np(direct[u][t]), want[u][t], f"multi {op} vs oracle")


def test_allreduce_multi_in_place_and_many_tensors(v):
    W = 8
    rng = np.random.default_rng(5)
    counts = [int(c) for c in rng.integers(1, 3000, 150)]  # > one launch of 64 tensors
    tens = _tensor_list(W, counts, "f32", 17)
    want = oracle.fusion_allreduce([[to_np(t) for t in tens[u]] for u in range(W)], counts, "sum",
                                   oracle.F32, threshold_bytes=1 << 40)
    v.allreduce_multi(tens, tens, op="sum", ring_order=True)
    for u in range(W):
        for t in range(len(counts)):
            assert_bit_exact(to_np(tens[u][t]), want[u][t], "multi in place")


def test_fusion_buffered_in_place_and_one_tensor_batches(v):
    # the C pipeline in place (outputs are the inputs), with batches of one
    # tensor (above the threshold: allreduced straight, no buffer) between
    # fused ones, and a fusion buffer exactly as large as the largest batch
    W = 4
    counts = [1000, 3, 9000, 250, 1, 60, 20000, 7, 7]
    thr = 4 * 5000
    tens = _tensor_list(W, counts, "f32", 41)
    want = oracle.fusion_allreduce([[to_np(t) for t in tens[u]] for u in range(W)], counts, "sum",
                                   oracle.F32, thr)
    begin = v.fuse_plan(counts, v.F32, thr)
    largest = max(sum(counts[begin[b]:begin[b + 1]]) for b in range(len(begin) - 1)
                  if begin[b + 1] - begin[b] > 1)
    fused = [torch.empty(largest, device="cuda") for _ in range(W)]
    v.fusion_allreduce(tens, tens, fused, op="sum", ring_order=True, threshold_bytes=thr)
    for u in range(W):
        for t in range(len(counts)):
            assert_bit_exact(to_np(tens[u][t]), want[u][t], f"buffered in place {u} {t}")


def test_fusion_direct_equals_pipeline_full_workload(v):
    # 200 fp32 tensors per rank, W = 8, 64 MiB batches: the one-pass path and
    # the pack -> allreduce -> unpack path give the same bits everywhere
    from collective_reduction_virtual_gb300 import inputs as I
    W = 8
    counts = [int(c) for c in I.fusion_counts()]
    tens = I.fusion_tensors(counts, W, "cuda")
    fused = [torch.empty((64 << 20) // 4, device="cuda") for _ in range(W)]
    for ring in (True, False):
        a = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
        b = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
        v.fusion_allreduce(tens, a, fused, op="avg", ring_order=ring)
        v.fusion_allreduce_direct(tens, b, op="avg", ring_order=ring)
        for u in range(W):
            assert torch.equal(torch.cat(a[u]).view(torch.int32), torch.cat(b[u]).view(torch.int32))


# ------------------------------------------------------------ min and prod

def _near_one(W, n, dtype, seed):
    """sign * 2^U(-1, 1): products of up to 64 stay far from overflow."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = []
    for _ in range(W):
        mag = torch.pow(2.0, torch.rand(n, generator=g, device="cuda") * 2 - 1)
        sgn = torch.where(torch.rand(n, generator=g, device="cuda") < 0.5, -1.0, 1.0)
        out.append((mag * sgn).to(DT[dtype]))
    return out


@pytest.mark.parametrize("W", SMALL_W)
@pytest.mark.parametrize("n", [1, 17, 4099, 65541])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_min_prod_small(v, W, n, dtype):
    for op in ("min", "prod"):
        ins = _near_one(W, n, dtype, 7000 * W + n) if op == "prod" else \
            make_inputs(W, n, dtype, 7100 * W + n)
        ins_np = [to_np(t) for t in ins]
        want = oracle.allreduce(ins_np, op, ODT[dtype])
        rs_want = oracle.reduce_scatter(ins_np, op, ODT[dtype])
        for ring in (True, False):
            got = v.allreduce(ins, op=op, ring_order=ring)
            rs = v.reduce_scatter(ins, op=op, ring_order=ring)
            for u in range(W):
                if ring or op == "min":
                    assert_bit_exact(to_np(got[u]), want[u], f"AR {op} ring={ring}")
                    assert_bit_exact(to_np(rs[u]), rs_want[u], f"RS {op} ring={ring}")
                else:
                    assert_close_fast(to_np(got[u]), want[u], None, W, op, f"AR {op}")
            if W in (2, 4, 8, 16) and n > 1000:
                st = v.allreduce(ins, op=op, ring_order=ring, flags=v.FLAG_STAGED)
                assert to_np(st[0]).tobytes() == to_np(got[0]).tobytes()
        tens = [[t] for t in ins]
        multi = v.allreduce_multi(tens, op=op, ring_order=True)
        for u in range(W):
            assert_bit_exact(to_np(multi[u][0]), want[u], f"multi {op}")


# special values for max and min: signed zeros, quiet and signalling NaNs of
# either sign, infinities, subnormals, the largest finite values
_SPECIAL_F32 = np.array([0x00000000, 0x80000000, 0x3F800000, 0xBF800000, 0x7F800000, 0xFF800000,
                         0x7FC00000, 0xFFC00000, 0x7F800001, 0x7FA00001, 0x00000001, 0x80000001,
                         0x007FFFFF, 0x7F7FFFFF, 0xFF7FFFFF, 0x40000000, 0xC0000000], dtype=np.uint32)
_SPECIAL_BF16 = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F81,
                          0x7FA1, 0x0001, 0x8001, 0x007F, 0x7F7F, 0xFF7F, 0x4000, 0xC000],
                         dtype=np.uint16)


def _special_inputs(W, n, dtype, seed, shift):
    rng = np.random.default_rng(seed)
    outs = []
    for _ in range(W):
        pool = _SPECIAL_F32 if dtype == "f32" else _SPECIAL_BF16
        bits = pool[rng.integers(0, pool.size, n + shift)]
        t = torch.from_numpy(bits.view(np.int32 if dtype == "f32" else np.int16).copy()).cuda()
        t = t.view(torch.float32 if dtype == "f32" else torch.bfloat16)
        outs.append(t[shift:])  # shift 1: a 16-byte phase other than the outputs'
    return outs


@pytest.mark.parametrize("W", [2, 3, 4, 8, 12, 16])
@pytest.mark.parametrize("n", [4099, 65541])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shift", [0, 1])
def test_max_min_special_values(v, W, n, dtype, shift):
    # every element drawn from the special values above: max and min must give
    # the oracle's bits exactly -- the canonical quiet NaN, +0 from max(+0, -0)
    # and -0 from min -- in every order, every kernel form
    ins = _special_inputs(W, n, dtype, 300 * W + n + shift, shift)
    ins_np = [to_np(t) for t in ins]
    for op in ("max", "min"):
        want = oracle.allreduce(ins_np, op, ODT[dtype])
        rs_want = oracle.reduce_scatter(ins_np, op, ODT[dtype])
        for ring in (True, False):
            got = v.allreduce(ins, op=op, ring_order=ring)
            rs = v.reduce_scatter(ins, op=op, ring_order=ring)
            for u in range(W):
                assert to_np(got[u]).tobytes() == want[u].tobytes(), f"AR {op} ring={ring} rank {u}"
                assert to_np(rs[u]).tobytes() == rs_want[u].tobytes(), f"RS {op} ring={ring} {u}"
            if W in (2, 4, 8, 16):  # the TMA-staged forms
                st = v.allreduce(ins, op=op, ring_order=ring, flags=v.FLAG_STAGED)
                rs_st = v.reduce_scatter(ins, op=op, ring_order=ring, flags=v.FLAG_STAGED)
                for u in range(W):
                    assert to_np(st[u]).tobytes() == want[u].tobytes(), f"AR staged {op} {u}"
                    assert to_np(rs_st[u]).tobytes() == rs_want[u].tobytes(), f"RS staged {op} {u}"


@pytest.mark.parametrize("W", [17, 64])
@pytest.mark.parametrize("frac", [0.01, 0.3])
def test_sparse_many_ranks(v, W, frac):
    # up to the largest rank count: per-rank states, candidate lists and
    # output folds over several groups of eight ranks (list route at 1 %,
    # band at 30 %), with and without accumulations; threshold mode too
    n = 50_003
    ins = _sparse_inputs(W, n, 70 + W)
    acc = [t * 0.3 for t in _sparse_inputs(W, n, 71 + W)]
    _check_sparse(v, ins, acc, frac, True)
    _check_sparse(v, ins, None, frac, True)
    _check_sparse(v, ins, [torch.zeros(n, device="cuda") for _ in range(W)], 1.5, False)


@pytest.mark.parametrize("W", [2, 3, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shift", [0, 1])
def test_sum_avg_prod_special_values(v, W, dtype, shift):
    # the special values under sum, avg and prod in ring order: signed zeros
    # (-0 + -0 = -0, -0 + +0 = +0), infinities and their NaNs, subnormals kept
    # (no flush to zero), overflow to infinity; NaN payloads of these ops are
    # not fixed (NaN matches NaN).  Also the one-pass multi-tensor form.
    n = 4099
    ins = _special_inputs(W, n, dtype, 500 * W + shift, shift)
    ins_np = [to_np(t) for t in ins]
    for op in ("sum", "avg", "prod"):
        want = oracle.allreduce(ins_np, op, ODT[dtype])
        rs_want = oracle.reduce_scatter(ins_np, op, ODT[dtype])
        got = v.allreduce(ins, op=op, ring_order=True)
        rs = v.reduce_scatter(ins, op=op, ring_order=True)
        multi = v.allreduce_multi([[t] for t in ins], op=op, ring_order=True)
        for u in range(W):
            assert_bit_exact(to_np(got[u]), want[u], f"AR {op} rank {u}")
            assert_bit_exact(to_np(rs[u]), rs_want[u], f"RS {op} segment {u}")
            assert_bit_exact(to_np(multi[u][0]), want[u], f"multi {op} rank {u}")


@pytest.mark.parametrize("wire", ["f16", "bf16"])
@pytest.mark.parametrize("W", [2, 3, 8])
def test_wire_special_values(v, wire, W):
    # SINGA's reduced-precision allreduce over special values, ring order:
    # every hop rounds to the wire type (fp16 overflows above 65504 and has
    # subnormals of its own; bf16 keeps fp32's range)
    n = 4099
    ins = _special_inputs(W, n, "f32", 600 * W, 0)
    ins_np = [to_np(t) for t in ins]
    for op in ("sum", "avg"):
        want = oracle.allreduce_wire(ins_np, wire, op)
        got = v.allreduce_wire(ins, wire=wire, op=op, ring_order=True)
        for u in range(W):
            assert_bit_exact(to_np(got[u]), want[u], f"wire {wire} {op} rank {u}")


@pytest.mark.parametrize("W", [2, 4])
@pytest.mark.parametrize("frac", [0.01, 0.3])
@pytest.mark.parametrize("topk", [True, False])
def test_sparse_special_values(v, W, frac, topk):
    # SINGA's sparsified allreduce over special values: without accumulations
    # x is the input itself, so NaNs of either sign take their keys' places in
    # the top-K order; with accumulations the inputs hold no NaN and the
    # accumulations are finite, so no sum makes one (the sign and payload of
    # a NaN sum are not fixed by IEEE 754, and the GPU and the host differ)
    n = 100_003
    ins = _special_inputs(W, n, "f32", 900 + W, 0)
    thr = frac if topk else 1.0
    _check_sparse(v, ins, None, thr, topk)
    no_nan = [torch.where(torch.isnan(t), torch.full_like(t, 3.0), t) for t in ins]
    acc = [t * 0.5 for t in _sparse_inputs(W, n, 901)]
    acc[0][::7] = -0.0
    acc[-1][::11] = 1e-40  # subnormal
    _check_sparse(v, no_nan, acc, thr, topk)


def test_prod_ring_order_hand_derived_on_gpu(v):
    x = [torch.full((4,), val, device="cuda") for val in (2.0 ** 100, 2.0 ** 100, 2.0 ** -100,
                                                          2.0 ** -100)]
    outs = v.reduce_scatter(x, op="prod", ring_order=True)
    assert [float(o[0]) for o in outs] == [1.0, 0.0, 1.0, float("inf")]


@pytest.mark.parametrize("n", [7, 4099, 65541])
def test_avg_scale_rounding_hand_derived_on_gpu(v, n):
    # the hand-derived avg bits for W = 3 and 5 (fl32(1/W) times the sum,
    # then the cast): integer inputs sum exactly in any order, so both
    # orders and both reduce-scatter and allreduce must give these bits
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "avg_scale_rounding.txt")
    rows = [ln.strip() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    for line in rows:
        dt, xs, bits = (p.strip() for p in line.split(";"))
        x = [torch.full((n,), float(val), device="cuda", dtype=DT[dt]) for val in xs.split()]
        want = int(bits, 16)
        view = torch.int32 if dt == "f32" else torch.int16
        mask = 0xFFFFFFFF if dt == "f32" else 0xFFFF
        for ring in (True, False):
            outs = v.allreduce(x, op="avg", ring_order=ring)
            outs += [torch.cat(v.reduce_scatter(x, op="avg", ring_order=ring))]
            for o in outs:
                got = (o.view(view).to(torch.int64) & mask).unique().tolist()
                assert got == [want], (line, ring, [hex(g) for g in got])


# Ring order on a user ring (NCCL's userFromRing): the page's 4-GPU example
# by hand, then random rings against the oracle's ring simulation.

@pytest.mark.parametrize("n", [4, 4 * 50_000])
def test_ring_permutation_hand_derived_on_gpu(v, n):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "ring_order_cancellation.txt")
    rows = [ln.strip() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    x = [torch.full((n,), val, device="cuda") for val in (1e8, 1.0, -1e8, 1.0)]
    for line in rows:
        ring_s, res_s = line.split(":")
        ring = [0, 1, 2, 3] if ring_s.strip() == "identity" else [int(q) for q in ring_s.split()]
        want = [float(q) for q in res_s.split()]
        segs = v.reduce_scatter(x, op="sum", user_from_ring=ring)
        assert [s.unique().tolist() for s in segs] == [[w] for w in want], ring_s
        ar = v.allreduce(x, op="sum", user_from_ring=ring)
        for u in range(4):
            assert [ar[u][j * n // 4: (j + 1) * n // 4].unique().tolist() for j in range(4)] == \
                [[w] for w in want], ring_s


@pytest.mark.parametrize("W", [3, 4, 5, 8, 16, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shift", [0, "mixed"])
def test_ring_permutation_matches_oracle(v, W, dtype, shift):
    n = 40_000 + W + 3  # several tiles per segment, uneven segments
    rng = np.random.default_rng(1000 + W)
    ring = [int(q) for q in rng.permutation(W)]
    base = make_inputs(W, n + 4, dtype, 77 + W)
    ins = [b[(u % 4 if shift == "mixed" else 0):][:n] for u, b in enumerate(base)]
    ins_np = [to_np(t) for t in ins]
    for op in ("sum", "avg", "prod"):
        want = oracle.reduce_scatter(ins_np, op, ODT[dtype], ring)
        segs = v.reduce_scatter(ins, op=op, user_from_ring=ring)
        for j in range(W):
            assert_bit_exact(to_np(segs[j]), want[j], f"ring RS {op} W={W} seg {j}")
        want_ar = oracle.allreduce(ins_np, op, ODT[dtype], ring)
        outs = v.allreduce(ins, op=op, user_from_ring=ring)
        for u in range(W):
            assert_bit_exact(to_np(outs[u]), want_ar[u], f"ring AR {op} W={W} rank {u}")


def test_ring_permutation_in_place(v):
    W, n = 8, 100_003
    ring = [3, 7, 0, 5, 1, 6, 2, 4]
    bufs = make_inputs(W, n, "f32", 5)
    want = oracle.allreduce([to_np(t) for t in bufs], "sum", oracle.F32, ring)
    v.allreduce(bufs, bufs, op="sum", user_from_ring=ring)
    for u in range(W):
        assert_bit_exact(to_np(bufs[u]), want[u], f"ring AR in place {u}")


# ------------------------------------------------------------ allgatherv

@pytest.mark.parametrize("W", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_allgatherv(v, W, dtype):
    rng = np.random.default_rng(W)
    counts = [int(c) for c in rng.integers(0, 20000, W)]
    counts[0] = 0 if W > 1 else counts[0]
    pieces = [make_inputs(1, c, dtype, 8000 + j)[0] for j, c in enumerate(counts)]
    want = oracle.allgatherv([to_np(p) for p in pieces], ODT[dtype])
    outs = v.allgatherv(pieces)
    for u in range(W):
        assert_bit_exact(to_np(outs[u]), want[u], f"AGV rank {u}")
    # in place: each piece already sits at its offset in its own output
    full = [torch.empty(sum(counts), dtype=DT[dtype], device="cuda") for _ in range(W)]
    offs = np.cumsum([0] + counts)
    views = []
    for j in range(W):
        full[j][offs[j]:offs[j + 1]].copy_(pieces[j])
        views.append(full[j][offs[j]:offs[j + 1]])
    v.allgatherv(views, full)
    for u in range(W):
        assert_bit_exact(to_np(full[u]), want[u], "AGV in place")


@pytest.mark.parametrize("W", [3, 8, 16])
@pytest.mark.parametrize("ring", [True, False])
def test_fusion_allreduce_entry_many_batches(v, W, ring):
    # many small batches: pieces of several batches share launches, and the
    # piece table (not the pointer table) decides where a launch ends
    rng = np.random.default_rng(W)
    counts = [int(c) for c in rng.integers(1, 2500, 150)]
    thr = 4 * 3000
    tens = _tensor_list(W, counts, "f32", 900 + W)
    a = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    fused = [torch.empty(max(counts) + 3000, device="cuda") for _ in range(W)]
    v.fusion_allreduce(tens, a, fused, op="avg", ring_order=ring, threshold_bytes=thr)
    b = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    plan = v.FusionPlan(tens, b, op="avg", ring_order=ring, threshold_bytes=thr)
    plan()
    assert plan.nbatches == len(v.fuse_plan(counts, v.F32, thr)) - 1
    for u in range(W):
        assert torch.equal(torch.cat(a[u]).view(torch.int32), torch.cat(b[u]).view(torch.int32))
    if ring:
        want = oracle.fusion_allreduce([[to_np(t) for t in tens[u]] for u in range(W)], counts,
                                       "avg", oracle.F32, thr)
        for u in (0, W - 1):
            for t in range(len(counts)):
                assert_bit_exact(to_np(b[u][t]), want[u][t], "fusion entry vs oracle")


# ------------------------------------------------- pinned host buffers

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pinned_host_buffers(v, dtype):
    # the kernels read and write pinned host memory directly (unified
    # addressing); the bits equal the device-buffer path
    W, n = 8, 300_007
    ins = make_inputs(W, n, dtype, 61)
    h_in = [t.cpu().pin_memory() for t in ins]
    h_out = [torch.empty(n, dtype=DT[dtype], pin_memory=True) for _ in range(W)]
    for op in ("sum", "avg", "max"):
        for ring in (True, False):
            d = v.allreduce(ins, op=op, ring_order=ring)
            v.allreduce(h_in, h_out, op=op, ring_order=ring)
            torch.cuda.synchronize()
            for u in range(W):
                assert to_np(h_out[u]).tobytes() == to_np(d[u]).tobytes()
    segs = [torch.empty(v.segment(n, W, j)[1], dtype=DT[dtype], pin_memory=True) for j in range(W)]
    v.reduce_scatter(h_in, segs, op="sum", ring_order=True)
    torch.cuda.synchronize()
    want = oracle.reduce_scatter([to_np(t) for t in ins], "sum", ODT[dtype])
    for j in range(W):
        assert_bit_exact(to_np(segs[j]), want[j], "RS on host buffers")
    v.allgather(segs, n, h_out)
    torch.cuda.synchronize()
    ring = v.allreduce(ins, op="sum", ring_order=True)
    for u in range(W):
        assert to_np(h_out[u]).tobytes() == to_np(ring[u]).tobytes()


def test_staged_request_on_host_buffers_runs_the_direct_kernels(v):
    # the TMA bulk copies of the staged forms run only on device memory; with
    # pinned host buffers a staged request gives the direct kernels' bits
    W, n = 8, 300_007
    ins = make_inputs(W, n, "f32", 62)
    h_in = [t.cpu().pin_memory() for t in ins]
    h_out = [torch.empty(n, pin_memory=True) for _ in range(W)]
    d = v.allreduce(ins, op="sum", flags=v.FLAG_DIRECT)
    v.allreduce(h_in, h_out, op="sum", flags=v.FLAG_STAGED)
    torch.cuda.synchronize()
    for u in range(W):
        assert to_np(h_out[u]).tobytes() == to_np(d[u]).tobytes()
    segs = [torch.empty(v.segment(n, W, j)[1], pin_memory=True) for j in range(W)]
    v.reduce_scatter(h_in, segs, op="sum", ring_order=True, flags=v.FLAG_STAGED)
    ag = [torch.empty(n, pin_memory=True) for _ in range(W)]
    v.allgather(segs, n, ag, flags=v.FLAG_STAGED)
    torch.cuda.synchronize()
    ring = v.allreduce(ins, op="sum", ring_order=True)
    for u in range(W):
        assert to_np(ag[u]).tobytes() == to_np(ring[u]).tobytes()
    assert v.device_errors(clear=True) == 0


@pytest.mark.parametrize("W", [2, 3, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [100_003, (1 << 22) + 6, 3 << 22])
def test_allgather_tma_matches_direct(v, W, dtype, n):
    segs = [make_inputs(1, oracle.segment(n, W, j)[1], dtype, 9000 + W + j)[0] for j in range(W)]
    d = v.allgather(segs, n, flags=v.FLAG_DIRECT)
    assert v.device_errors(clear=True) == 0
    t = v.allgather(segs, n, flags=v.FLAG_STAGED)
    assert v.device_errors(clear=True) == 0
    for u in range(W):
        assert to_np(t[u]).tobytes() == to_np(d[u]).tobytes(), f"rank {u}"
    if n < 200_000:
        want = oracle.allgather([to_np(s) for s in segs], n, ODT[dtype])
        for u in range(W):
            assert_bit_exact(to_np(t[u]), want[u], "AG TMA vs oracle")
    # shared non-zero phase: views one element into larger buffers
    base = [torch.empty(n + 8, dtype=DT[dtype], device="cuda") for _ in range(W)]
    outs = [b[1:1 + n] for b in base]
    sbase = [torch.empty(s.numel() + 8, dtype=DT[dtype], device="cuda") for s in segs]
    off = [oracle.segment(n, W, j)[0] for j in range(W)]
    # segment j must share the outputs' phase: element off_j at offset 1 + off_j
    sv = []
    for j, (sb, s) in enumerate(zip(sbase, segs)):
        sh = (1 + off[j]) % (4 if dtype == "f32" else 8)
        sb[sh:sh + s.numel()].copy_(s)
        sv.append(sb[sh:sh + s.numel()])
    v.allgather(sv, n, outs, flags=v.FLAG_STAGED)
    for u in range(W):
        assert to_np(outs[u]).tobytes() == to_np(d[u]).tobytes(), f"phase rank {u}"


# ------------------------------------------- reduced-precision wire allreduce

@pytest.mark.parametrize("wire", ["f16", "bf16"])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("n", [1, 17, 4099, 100_003])
def test_allreduce_wire(v, wire, W, n):
    g = torch.Generator(device="cuda")
    g.manual_seed(W * 1000 + n)
    ins = [torch.randn(n, generator=g, device="cuda") *
           (10.0 ** torch.randint(-6, 3, (n,), generator=g, device="cuda").float())
           for _ in range(W)]
    ins_np = [to_np(t) for t in ins]
    u = 2.0 ** -11 if wire == "f16" else 2.0 ** -8
    for op in ("sum", "avg"):
        want = oracle.allreduce_wire(ins_np, wire, op)
        ring = v.allreduce_wire(ins, wire=wire, op=op, ring_order=True)
        fast = v.allreduce_wire(ins, wire=wire, op=op)
        for r in range(W):
            assert_bit_exact(to_np(ring[r]), want[r], f"wire {wire} {op} ring")
            # fastest order: both orders start from the same rounded inputs
            # and each is W-1 hop roundings from their exact sum; a rounding
            # errs by at most u_w |partial| + eta, where eta is half the wire
            # type's subnormal spacing (2^-25 for fp16; bf16 has fp32's
            # range, where 2^-25 is ample) and |partial| <= s = sum |x_r|
            # (divided by W for avg, whose hop errors the scale divides too);
            # avg's scale multiply and its second rounding to the wire type
            # add two more terms.  So each order is within (W+1)(u_w s + eta)
            # of the exact sum and the two within twice that.
            s = abs_sum([(to_np(t)) for t in ins]) / (W if op == "avg" else 1)
            bound = 2 * (W + 1) * (u * s + 2.0 ** -25)
            d = np.abs(to_np(fast[r]).astype(np.float64) - want[r].astype(np.float64))
            ok = (d <= bound) | (np.isnan(to_np(fast[r])) & np.isnan(want[r]))
            assert ok.all(), f"wire {wire} {op} fast: max excess {(d - bound).max()}"


def test_allreduce_wire_hop_rounding_on_gpu(v):
    for wire, xs, want in (("f16", (2048.0, 1.0, 1.0), [2050.0, 2048.0, 2048.0]),
                           ("bf16", (256.0, 1.0, 1.0), [258.0, 256.0, 256.0])):
        x = [torch.full((3,), val, device="cuda") for val in xs]
        out = v.allreduce_wire(x, wire=wire, op="sum", ring_order=True)
        assert all(o.tolist() == want for o in out), wire


def test_allreduce_wire_misaligned(v):
    W, n = 4, 50_001
    base = [torch.randn(n + 8, device="cuda") for _ in range(W)]
    ins = [b[(u * 3) % 4: (u * 3) % 4 + n] for u, b in enumerate(base)]
    want = oracle.allreduce_wire([to_np(t) for t in ins], "f16", "sum")
    got = v.allreduce_wire(ins, wire="f16", op="sum", ring_order=True)
    for r in range(W):
        assert_bit_exact(to_np(got[r]), want[r], "wire misaligned")


# ----------------------------------------------- sparsified allreduce (SINGA)

def _sparse_inputs(W, n, seed, ties=False):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    xs = []
    for _ in range(W):
        x = torch.randn(n, generator=g, device="cuda")
        if ties:
            x = torch.round(x * 4) / 4  # many equal values across the top-K cut
        xs.append(x)
    return xs


def _check_sparse(v, ins, acc, thr, topk, workspace_bytes=None, outs=None):
    W = len(ins)
    ins_np = [to_np(t) for t in ins]
    acc_np = [to_np(a).copy() for a in acc] if acc is not None else None
    want, want_nnz = oracle.sparse_allreduce(ins_np, thr, topk, acc_np)
    nnz = torch.empty(W, dtype=torch.int64, device="cuda")
    ws = None
    if workspace_bytes is not None:
        ws = torch.empty(workspace_bytes, dtype=torch.uint8, device="cuda")
    outs = v.sparse_allreduce(ins, outs, accum=acc, threshold=thr, topk=topk, nnz=nnz,
                              workspace=ws)
    torch.cuda.synchronize()
    for u in range(W):
        assert_bit_exact(to_np(outs[u]), want[u], f"sparse topk={topk} out {u}")
        if acc is not None:
            assert_bit_exact(to_np(acc[u]), acc_np[u], f"sparse topk={topk} accum {u}")
    assert nnz.cpu().tolist() == list(want_nnz)


@pytest.mark.parametrize("W", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("n", [1, 17, 4097, 100_003])
@pytest.mark.parametrize("with_acc", [False, True])
def test_sparse_threshold(v, W, n, with_acc):
    ins = _sparse_inputs(W, n, 40 * W + n)
    acc = [t * 0.3 for t in _sparse_inputs(W, n, 41 * W + n)] if with_acc else None
    _check_sparse(v, ins, acc, 0.8, False)


@pytest.mark.parametrize("W", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 17, 4097, 100_003])
@pytest.mark.parametrize("frac", [0.0, 0.001, 0.05, 0.5, 1.0])
def test_sparse_topk(v, W, n, frac):
    ins = _sparse_inputs(W, n, 50 * W + n)
    acc = [t * 0.3 for t in _sparse_inputs(W, n, 51 * W + n)]
    _check_sparse(v, ins, acc, frac, True)


@pytest.mark.parametrize("frac", [0.001, 0.01, 0.05, 0.3, 0.77])
def test_sparse_topk_ties_straddle_the_cut(v, frac):
    W, n = 4, 50_001
    ins = _sparse_inputs(W, n, 77, ties=True)
    _check_sparse(v, ins, None, frac, True)
    _check_sparse(v, ins, [torch.zeros(n, device="cuda") for _ in range(W)], frac, True)


def test_sparse_misaligned_and_in_place(v):
    W, n = 3, 30_001
    base = _sparse_inputs(W, n + 4, 9)
    ins = [b[u % 4: u % 4 + n] for u, b in enumerate(base)]  # mixed 16-byte phases
    _check_sparse(v, ins, None, 0.9, False)
    _check_sparse(v, ins, None, 0.02, True)
    bufs = [t.clone() for t in _sparse_inputs(W, n, 10)]
    want, _ = oracle.sparse_allreduce([to_np(t) for t in bufs], 0.05, True)
    v.sparse_allreduce(bufs, bufs, threshold=0.05, topk=True)
    for u in range(W):
        assert_bit_exact(to_np(bufs[u]), want[u], "sparse in place")


# With accumulations and output from the lists, the candidate pass writes the
# residual of entries above the sample's settled bin itself; the output pass
# undoes it for any that are not kept, and so does a restore pass when the
# result does not come from the lists.  These cover the candidate pass's
# three layouts (shared 16-byte phase, a head and tail per tile, mixed phases)
# and a settled bin that the data contradict.

@pytest.mark.parametrize("shift", [0, 1, "mixed"])
@pytest.mark.parametrize("frac", [0.01, 0.02])
def test_sparse_topk_settled_residuals_layouts(v, shift, frac):
    W, n = 3, 128 * 4096 + 11
    base = _sparse_inputs(W, n + 4, 300 + W)
    abase = [t * 0.3 for t in _sparse_inputs(W, n + 4, 301 + W)]
    obase = [torch.empty(n + 4, device="cuda") for _ in range(W)]
    # shift 0 / 1: every buffer at that element offset (16-byte phase 0, or a
    # head and tail per tile); mixed: inputs, accumulations and outputs at
    # different phases (the element-wise candidate pass)
    ph = {"in": lambda u: u % 4, "acc": lambda u: (u + 1) % 4, "out": lambda u: 0} \
        if shift == "mixed" else {k: (lambda u: shift) for k in ("in", "acc", "out")}
    ins = [b[ph["in"](u): ph["in"](u) + n] for u, b in enumerate(base)]
    acc = [a[ph["acc"](u): ph["acc"](u) + n] for u, a in enumerate(abase)]
    outs = [o[ph["out"](u): ph["out"](u) + n] for u, o in enumerate(obase)]
    _check_sparse(v, ins, acc, frac, True, outs=outs)
    _check_sparse(v, ins, acc, frac, True, outs=outs)  # a second step on the new residuals


# Without accumulations the candidate pass takes two tiles per CTA (one list
# reservation for both): odd and even tile counts, a head and tail in every
# tile, and mixed phases (the element-wise form) must all give the oracle's
# bits, on the list route (small K) and with the two-sided band.
@pytest.mark.parametrize("shift", [0, 1, 3, "mixed"])
@pytest.mark.parametrize("n", [129 * 4096 + 11, 128 * 4096 - 1, 4096 + 5])
@pytest.mark.parametrize("frac", [0.01, 0.3])
def test_sparse_topk_no_accumulation_layouts(v, shift, n, frac):
    W = 8
    base = _sparse_inputs(W, n + 4, 310 + n % 97)
    obase = [torch.empty(n + 4, device="cuda") for _ in range(W)]
    pin = (lambda u: u % 4) if shift == "mixed" else (lambda u: shift)
    ins = [b[pin(u): pin(u) + n] for u, b in enumerate(base)]
    outs = [o[pin(u): pin(u) + n] for u, o in enumerate(obase)]
    _check_sparse(v, ins, None, frac, True, outs=outs)


def test_sparse_topk_settled_bin_contradicted(v):
    # the sampled tiles (every 16th of 4096 entries) hold smaller values than
    # the rest, so the sample places the settled bin too low (about twice K
    # entries lie above it) while the lower bound still holds the K-th key:
    # the settled entries that are not kept must get their x back
    W, n = 2, 64 * 4096
    ins = _sparse_inputs(W, n, 17)
    for t in ins:
        tiles = t.view(-1, 4096)
        tiles[::16] *= 0.75
    acc = [torch.zeros(n, device="cuda") for _ in range(W)]
    _check_sparse(v, ins, acc, 0.01, True)
    _check_sparse(v, ins, acc, 0.02, True)


def test_sparse_topk_larger(v):
    W, n = 8, 1 << 21
    ins = _sparse_inputs(W, n, 123)
    acc = [torch.zeros(n, device="cuda") for _ in range(W)]
    _check_sparse(v, ins, acc, 0.01, True)
    _check_sparse(v, ins, acc, 0.01, True)  # second step: the error feedback is nonzero now


def test_sparse_topk_sample_bound_redo(v):
    # the sample pass reads every 16th tile of 4096 entries; large values only
    # in those tiles make its lower bound far too high for the whole array,
    # so the first-digit pass must be redone over all bins on the device
    W, n = 2, 64 * 4096
    ins = _sparse_inputs(W, n, 5)
    for t in ins:
        tiles = t.view(-1, 4096)
        tiles[::16] = tiles[::16].abs() + 100.0
    _check_sparse(v, ins, None, 0.01, True)
    _check_sparse(v, ins, [torch.zeros(n, device="cuda") for _ in range(W)], 0.2, True)
    _check_sparse(v, ins, None, 0.4, True)  # the band (K >= n/4) misses as well


@pytest.mark.parametrize("frac", [0.001, 0.01, 0.1])
def test_sparse_topk_layered_buffer(v, frac):
    # a fused gradient buffer: tensors of log-uniform sizes, each at its own
    # scale (10^U(-4, -2)), so the sampled tiles see a mixture of layers
    from collective_reduction_virtual_gb300 import inputs as I
    W, n = 4, (1 << 22) + 5
    counts = I.fusion_counts(T=200, lo=256, hi=262144)
    rng = np.random.default_rng(9)
    scales = 10.0 ** rng.uniform(-4, -2, counts.size)
    ins = _sparse_inputs(W, n, 91)
    for t in ins:
        off = 0
        for c, sc in zip(counts, scales):
            if off >= n:
                break
            t[off:off + int(c)] *= float(sc)
            off += int(c)
    acc = [torch.zeros(n, device="cuda") for _ in range(W)]
    _check_sparse(v, ins, acc, frac, True)
    _check_sparse(v, ins, acc, frac, True)  # the error feedback is nonzero now
    _check_sparse(v, ins, None, frac, True)


@pytest.mark.parametrize("scale", [0.85, 0.97, 0.997, 1.003, 1.03, 1.15])
@pytest.mark.parametrize("frac", [0.05, 0.1, 0.3])
def test_sparse_topk_band_refined_bounds_contradicted(v, scale, frac):
    # the two-sided band (lists too small for 3K entries), refined to 22-bit
    # bounds by the second sample pass: the sampled tiles (every 16th of 4096
    # entries, four tiles here, so the band's margin is about 14 % of K's
    # share) are scaled so that the band sits below or above the K-th key of
    # the whole array (0.85, 1.15: too many entries above the band, or the
    # K-th key below it, and the rank falls back) or near its edges (the
    # bounds still hold)
    W, n = 2, 64 * 4096
    ins = _sparse_inputs(W, n, 23)
    for t in ins:
        tiles = t.view(-1, 4096)
        tiles[::16] *= scale
    _check_sparse(v, ins, None, frac, True)
    _check_sparse(v, ins, [t * 0.1 for t in _sparse_inputs(W, n, 24)], frac, True)


# The top-K select runs over candidate lists when the workspace has room for
# them (the entries above a sampled bound), else over the whole array; a rank
# whose list overflows or misses the K-th key falls back on the device.  Every
# route must give the oracle's bits.

@pytest.mark.parametrize("frac", [0.001, 0.01, 0.05])
def test_sparse_topk_minimum_workspace(v, frac):
    W, n = 4, 300_007
    ins = _sparse_inputs(W, n, 61)
    acc = [t * 0.3 for t in _sparse_inputs(W, n, 62)]
    least = v.sparse_workspace_min_bytes(W, n)
    assert least < v.sparse_workspace_bytes(W, n)
    _check_sparse(v, ins, acc, frac, True, workspace_bytes=least)


def test_sparse_topk_candidate_list_overflows(v):
    # the sampled tiles (every 16th of 4096 entries) hold tiny values, so the
    # sampled bound admits about half of every other tile: far more than the
    # lists hold
    W, n = 2, 64 * 4096 + 5
    ins = _sparse_inputs(W, n, 8)
    for t in ins:
        tiles = t[: 64 * 4096].view(-1, 4096)
        tiles[::16] *= 1e-6
    _check_sparse(v, ins, None, 0.01, True)
    _check_sparse(v, ins, [torch.zeros(n, device="cuda") for _ in range(W)], 0.03, True)
    # K >= n/4: the band's upper bound sits among the tiny sampled values, so
    # far more than K entries lie above it
    _check_sparse(v, ins, None, 0.3, True)


def test_sparse_topk_mixed_routes_in_one_call(v):
    # rank 0 overflows its list, rank 1 misses the K-th key (large values only
    # in the sampled tiles), ranks 2 and 3 stay on their lists, ranks 3 with
    # ties across the cut
    W, n = 4, 128 * 4096
    ins = _sparse_inputs(W, n, 12)
    ins[0].view(-1, 4096)[::16] *= 1e-6
    t1 = ins[1].view(-1, 4096)
    t1[::16] = t1[::16].abs() + 100.0
    ins[3] = torch.round(ins[3] * 4) / 4
    _check_sparse(v, ins, None, 0.01, True)
    # a workspace between the minimum and the recommended size: shorter lists
    mid = (v.sparse_workspace_min_bytes(W, n) + v.sparse_workspace_bytes(W, n)) // 2
    _check_sparse(v, ins, [torch.zeros(n, device="cuda") for _ in range(W)], 0.01, True,
                  workspace_bytes=mid)
    # K >= n/4: a band with an upper bound on the ranks whose sample holds
    _check_sparse(v, ins, None, 0.3, True)
    _check_sparse(v, ins, None, 0.6, True, workspace_bytes=mid)


# K beyond what the lists hold above a wide lower bound (3K > n/8 + 4096):
# the sample sets a two-sided band, entries above it are only counted
@pytest.mark.parametrize("frac", [0.05, 0.1, 0.25, 0.3, 0.5, 0.9, 0.999])
def test_sparse_topk_large_k_band(v, frac):
    W, n = 4, 256 * 4096 + 3
    ins = _sparse_inputs(W, n, 70)
    acc = [t * 0.3 for t in _sparse_inputs(W, n, 71)]
    _check_sparse(v, ins, acc, frac, True)
    ins = [torch.round(t * 8) / 8 for t in ins]  # ties at the K-th key
    _check_sparse(v, ins, None, frac, True)


@pytest.mark.parametrize("extra,W", [(1, 2), (6, 2), (255, 2), (300, 2), (6, 8), (300, 8)])
@pytest.mark.parametrize("with_acc", [False, True])
def test_sparse_topk_few_ties_at_the_cut(v, extra, W, with_acc):
    # `extra` entries below the K-th largest value are raised to it, so that
    # keys equal to the K-th one straddle the cut: up to 256 of them are
    # collected and ranked by index, more take the digit passes (every rank
    # at once with W = 8)
    n, frac = 64 * 4096 + 7, 0.01
    K = int(np.ceil(np.float32(frac) * np.float32(n)))
    ins = _sparse_inputs(W, n, 900 + extra + W)
    g = torch.Generator(device="cuda")
    g.manual_seed(extra + W)
    for t in ins:
        kth = torch.topk(t, K).values[-1]
        below = torch.nonzero(t < kth).flatten()
        pick = below[torch.randperm(below.numel(), generator=g, device="cuda")[:extra]]
        t[pick] = kth
    acc = [torch.zeros(n, device="cuda") for _ in range(W)] if with_acc else None
    _check_sparse(v, ins, acc, frac, True)


def test_sparse_topk_all_equal_values(v):
    # every entry ties: the K kept are the K lowest indices
    W, n = 3, 100_000
    ins = [torch.full((n,), 0.5, device="cuda") for _ in range(W)]
    _check_sparse(v, ins, None, 0.01, True)
    ins = [torch.zeros(n, device="cuda") for _ in range(W)]
    _check_sparse(v, ins, None, 0.02, True)
    # -0 + -0 keeps the sign: the kept -0 entries leave a residual of
    # -0 - (0 + -0) = -0
    ins = [torch.full((n,), -0.0, device="cuda") for _ in range(W)]
    _check_sparse(v, ins, [torch.full((n,), -0.0, device="cuda") for _ in range(W)], 0.02, True)


@pytest.mark.parametrize("frac,skew", [(0.01, False), (0.3, False), (0.01, True)])
def test_sparse_topk_in_a_cuda_graph(v, frac, skew):
    # every route decision is taken on the device, so a captured call replays
    # correctly on new inputs, falling back or not as the data demand; the
    # replays must match the oracle, residuals included
    W, n = 4, 64 * 4096 + 3
    ins = _sparse_inputs(W, n, 90)
    acc = [torch.zeros(n, device="cuda") for _ in range(W)]
    outs = [torch.empty(n, device="cuda") for _ in range(W)]
    nnz = torch.empty(W, dtype=torch.int64, device="cuda")
    ws = torch.empty(v.sparse_workspace_bytes(W, n), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        v.sparse_allreduce(ins, outs, acc, frac, True, nnz, ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        v.sparse_allreduce(ins, outs, acc, frac, True, nnz, ws, stream=s)
    for step in range(2):
        new = _sparse_inputs(W, n, 91 + step)
        if skew and step == 1:  # large values only in the sampled tiles: a fallback
            for t in new:
                tl = t[: 64 * 4096].view(-1, 4096)
                tl[::16] = tl[::16].abs() + 100.0
        for t, x in zip(ins, new):
            t.copy_(x)
        acc_np = [to_np(a).copy() for a in acc]
        want, want_nnz = oracle.sparse_allreduce([to_np(t) for t in ins], frac, True, acc_np)
        g.replay()
        torch.cuda.synchronize()
        for u in range(W):
            assert_bit_exact(to_np(outs[u]), want[u], f"graph replay {step} out {u}")
            assert_bit_exact(to_np(acc[u]), acc_np[u], f"graph replay {step} accum {u}")
        assert nnz.cpu().tolist() == list(want_nnz)


# Inputs at mixed 16-byte phases, outputs sharing one: the realigning vector
# kernel (each input read as the two aligned blocks around a vector and
# funnel-shifted).  Ring order bit-exact; the fast order is the same left
# fold as the element-wise kernel, checked to the reordering bound.
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("n", [1031, 200_003])
def test_realigned_inputs(v, dtype, W, n):
    V = 4 if dtype == "f32" else 8
    shifts = [(u * 5 + 1) % 16 for u in range(W)]
    ins = _views(W, n, dtype, shifts, 300 + W + n)
    ins_np = [to_np(t) for t in ins]
    s = abs_sum(ins_np)
    outs = [torch.empty(n, dtype=DT[dtype], device="cuda") for _ in range(W)]  # one phase
    for op in ("sum", "avg", "max", "min", "prod"):
        want = oracle.allreduce(ins_np, op, ODT[dtype])
        for ring in (True, False):
            v.allreduce(ins, outs, op=op, ring_order=ring)
            for u in range(W):
                g = to_np(outs[u])
                if ring or op in ("max", "min"):
                    assert_bit_exact(g, want[u], f"AR realigned {op} ring={ring}")
                else:
                    assert_close_fast(g, want[u], s, W, op, f"AR realigned {op}")
        # reduce-scatter outputs placed so that out[j] - off_j shares one phase
        rs_want = oracle.reduce_scatter(ins_np, op, ODT[dtype])
        rbase = [torch.empty(n + 16, dtype=DT[dtype], device="cuda") for _ in range(W)]
        rs_out = []
        for j in range(W):
            off, ln = oracle.segment(n, W, j)
            k = (off + 3) % V  # (k - off) % V == 3 for every j
            rs_out.append(rbase[j][k:k + ln])
        v.reduce_scatter(ins, rs_out, op=op, ring_order=True)
        for j in range(W):
            assert_bit_exact(to_np(rs_out[j]), rs_want[j], f"RS realigned {op}")


# Large enough that the launch uses full-size tiles (several vectors per
# thread per rank) for every rank count, so a kernel that covered only part
# of a tile would show; odd n gives uneven segments (realigned vectors for
# the reduce-scatter) and W outside {2, 4, 8, 16} the runtime-W kernels.
@pytest.mark.parametrize("W", [3, 6, 8, 12])
@pytest.mark.parametrize("n", [3 * (1 << 20), 3 * (1 << 20) + 5])
def test_full_tiles_runtime_w_and_uneven(v, W, n):
    ins = make_inputs(W, n, "f32", 500 + W + n)
    ins_np = [to_np(t) for t in ins]
    want = oracle.reduce_scatter(ins_np, "sum", oracle.F32)
    outs = v.reduce_scatter(ins, op="sum", ring_order=True)
    for j in range(W):
        assert_bit_exact(to_np(outs[j]), want[j], f"RS full tiles W={W} n={n}")
    want = oracle.allreduce(ins_np, "sum", oracle.F32)
    outs = v.allreduce(ins, op="sum", ring_order=True)
    for u in (0, W - 1):
        assert_bit_exact(to_np(outs[u]), want[u], f"AR full tiles W={W} n={n}")
    segs = [ins[j][:oracle.segment(n, W, j)[1]].clone() for j in range(W)]
    ag_want = oracle.allgather([to_np(s) for s in segs], n, oracle.F32)
    ag = v.allgather(segs, n)
    for u in (0, W - 1):
        assert_bit_exact(to_np(ag[u]), ag_want[u], f"AG full tiles W={W} n={n}")


def test_collectives_and_fusion_in_a_cuda_graph(v):
    # these calls captured in a CUDA graph on a side stream (no host sync, no
    # allocation inside), replayed after the inputs change in place, against
    # the same calls made directly
    W, n = 4, 70_001
    ins = make_inputs(W, n, "f32", 9100)
    segs = [torch.empty(oracle.segment(n, W, j)[1], device="cuda") for j in range(W)]
    ar = [torch.empty(n, device="cuda") for _ in range(W)]
    ar_st = [torch.empty(n, device="cuda") for _ in range(W)]
    ag = [torch.empty(n, device="cuda") for _ in range(W)]
    wire = [torch.empty(n, device="cuda") for _ in range(W)]
    rs_ring = [torch.empty_like(s) for s in segs]
    counts = [5000, 1, 0, 12345, 777]
    pieces = [t[:c] for t, c in zip(ins, [100, 2000, 0, 70_001])]
    agv = [torch.empty(sum(p.numel() for p in pieces), device="cuda") for _ in range(W)]
    tens = [[torch.randn(c, device="cuda") for c in counts] for _ in range(W)]
    t_one = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    t_buf = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    fused = [torch.empty(sum(counts), device="cuda") for _ in range(W)]
    one_plan = v.FusionPlan(tens, t_one, op="avg", threshold_bytes=4 * 6000)
    buf_plan = v.FusionBufferPlan(tens, t_buf, fused, op="avg", threshold_bytes=4 * 6000)
    ring = [2, 0, 3, 1]

    def calls(s):
        v.reduce_scatter(ins, segs, op="sum", ring_order=True, stream=s)
        v.allgather(segs, n, ag, stream=s)
        v.allreduce(ins, ar, op="max", stream=s)
        v.allreduce(ins, ar_st, op="avg", flags=v.FLAG_STAGED, stream=s)
        v.allreduce_wire(ins, wire, wire="bf16", op="sum", ring_order=True, stream=s)
        v.reduce_scatter(ins, rs_ring, op="sum", user_from_ring=ring, stream=s)
        v.allgatherv(pieces, agv, stream=s)
        one_plan(s)
        buf_plan(s)

    def results():
        return [t.clone() for t in segs + ag + ar + ar_st + wire + rs_ring + agv] + \
            [t.clone() for u in range(W) for t in t_one[u] + t_buf[u]]

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls(s)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(s)
    for step in range(2):
        for t in ins:
            t.mul_(-1.5).add_(0.25)
        for row in tens:
            for t in row:
                t.mul_(0.5).add_(1.0)
        g.replay()
        torch.cuda.synchronize()
        got = results()
        calls(torch.cuda.current_stream())
        torch.cuda.synchronize()
        want = results()
        for a, b in zip(got, want):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"graph replay {step}"

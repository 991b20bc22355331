"""Pins for the CPU oracle: what the pages and the mathematics fix, checked
against the oracle without any GPU.  Each test names what it pins.

Pins used (none retypes the oracle's own formulas):
  * the 4-GPU schedule table printed on the NCCL reduce_scatter.cu page;
  * hand-derived order-sensitive sums (tests/golden/ring_order_cancellation.txt);
  * exact integer sums (integer-valued floats add exactly in any order);
  * exact rational sums within the textbook reordering bound gamma_{W-1};
  * numpy.maximum.reduce for max on NaN-free data, hand cases for +-0 and NaN;
  * torch's CPU bf16 conversion and hand-derived ties for the bf16 cast;
  * the identities of the "Distributed primitives" notes (AllReduce =
    ReduceScatter + AllGather, every node holds the same aggregate);
  * NCCL's single-GPU copy and empty-message cases;
  * Horovod's fusion batching rule on hand-derived lists, numpy.concatenate
    for the packed layout.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(20261202 + seed)


def _golden_lines(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- schedule

def test_ring_schedule_matches_nccl_page_table():
    rows = _golden_lines("nccl_ring_schedule_4gpu.txt")
    table = np.array([[int(v) for v in r.split()[1:]] for r in rows])
    got = oracle.ring_schedule(4, [1, 2, 0, 3])
    assert np.array_equal(got, table)


@pytest.mark.parametrize("W", [1, 2, 3, 5, 8, 16])
def test_ring_schedule_structure(W):
    # The page's description of the table: the last row is userFromRing, each
    # earlier row is the next one shifted left by one, and each GPU's column
    # visits every block exactly once.
    perm = list(_rng(W).permutation(W))
    tab = oracle.ring_schedule(W, perm)
    assert list(tab[W - 1]) == perm
    for s in range(W - 1):
        assert list(tab[s]) == list(np.roll(tab[s + 1], -1))
    for p in range(W):
        assert sorted(tab[:, p]) == list(range(W))


# ----------------------------------------------------------- segmentation

def test_segments_golden():
    for line in _golden_lines("segments_uneven.txt"):
        head, tail = line.split(":")
        n, W = (int(v) for v in head.split())
        vals = [int(v) for v in tail.split()]
        for j in range(W):
            assert oracle.segment(n, W, j) == (vals[2 * j], vals[2 * j + 1]), (n, W, j)


@pytest.mark.parametrize("n,W", [(0, 1), (1, 7), (1000, 3), (1 << 20, 4), (12345, 16), (5, 64)])
def test_segments_cover_contiguously(n, W):
    end = 0
    lens = []
    for j in range(W):
        off, ln = oracle.segment(n, W, j)
        assert off == end
        end += ln
        lens.append(ln)
    assert end == n
    assert max(lens) - min(lens) <= 1
    assert lens == sorted(lens, reverse=True)


# ------------------------------------------------------- fold order (pins)

def test_ring_order_hand_derived():
    x = [np.full(4, v, np.float32) for v in (1e8, 1.0, -1e8, 1.0)]
    for line in _golden_lines("ring_order_cancellation.txt"):
        ring_s, res_s = line.split(":")
        ring = None if ring_s.strip() == "identity" else [int(v) for v in ring_s.split()]
        want = [float(v) for v in res_s.split()]
        segs = oracle.reduce_scatter(x, "sum", oracle.F32, ring)
        assert [float(s[0]) for s in segs] == want, ring_s
        ar = oracle.allreduce(x, "sum", oracle.F32, ring)
        for u in range(4):
            assert list(ar[u]) == want


def _stepwise_ring_fold(vals, j, ring):
    # Independent re-fold of one element of block j: follow the block through
    # the ring positions after its owner, widening to float32 and adding one
    # rank at a time with numpy scalars (fp32 IEEE adds).
    W = len(vals)
    k = ring.index(j)
    acc = np.float32(vals[ring[(k + 1) % W]])
    for t in range(2, W + 1):
        acc = np.float32(acc + np.float32(vals[ring[(k + t) % W]]))
    return acc


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("n", [1, 2, 5, 16])
def test_brute_force_tiny(W, n):
    rng = _rng(100 * W + n)
    ring = list(rng.permutation(W))
    # wide dynamic range so that different orders really give different bits
    ins = [(rng.standard_normal(n) * 10.0 ** rng.integers(-3, 9, n)).astype(np.float32)
           for _ in range(W)]
    segs = oracle.reduce_scatter(ins, "sum", oracle.F32, ring)
    for j in range(W):
        off, ln = oracle.segment(n, W, j)
        for k in range(ln):
            want = _stepwise_ring_fold([ins[u][off + k] for u in range(W)], j, ring)
            assert segs[j][k].tobytes() == want.tobytes()


def test_order_is_actually_observable():
    # Same multiset of values, different start rank: the results differ, so
    # the tests above really pin the order and not just the multiset.
    x = [np.full(4, v, np.float32) for v in (1e8, 1.0, -1e8, 1.0)]
    segs = oracle.reduce_scatter(x, "sum")
    assert len({float(s[0]) for s in segs}) > 1


# ------------------------------------------------------------- sum values

@pytest.mark.parametrize("W", [1, 2, 3, 4, 7, 8, 16])
def test_integer_valued_sums_exact(W):
    rng = _rng(W)
    n = 1000 + W
    ins = [rng.integers(-1024, 1025, n).astype(np.float32) for _ in range(W)]
    want = np.sum(np.stack([a.astype(np.int64) for a in ins]), axis=0)
    ar = oracle.allreduce(ins, "sum")
    for u in range(W):
        assert np.array_equal(ar[u].astype(np.int64), want)


@pytest.mark.parametrize("W", [2, 4, 8, 16])
def test_sum_within_reordering_bound_of_exact(W):
    rng = _rng(7 * W)
    n = 300
    ins = [rng.uniform(-1, 1, n).astype(np.float32) for _ in range(W)]
    ar = oracle.allreduce(ins, "sum")[0]
    u = Fraction(1, 1 << 24)
    gamma = (W - 1) * u / (1 - (W - 1) * u)
    for i in range(n):
        exact = sum(Fraction(float(a[i])) for a in ins)
        mag = sum(abs(Fraction(float(a[i]))) for a in ins)
        assert abs(Fraction(float(ar[i])) - exact) <= gamma * mag


@pytest.mark.parametrize("k", [0, 1, 2, 3, 4])
def test_avg_power_of_two_exact(k):
    W = 1 << k
    rng = _rng(k)
    ins = [(rng.integers(-512, 513, 333) * W).astype(np.float32) for _ in range(W)]
    want = np.sum(np.stack([a.astype(np.int64) for a in ins]), axis=0) // W
    for got in oracle.allreduce(ins, "avg"):
        assert np.array_equal(got.astype(np.int64), want)
    assert np.array_equal(np.concatenate(oracle.reduce_scatter(ins, "avg")).astype(np.int64), want)


@pytest.mark.parametrize("W", [3, 5, 6])
def test_avg_close_to_exact_mean(W):
    rng = _rng(W + 40)
    ins = [rng.uniform(-1, 1, 200).astype(np.float32) for _ in range(W)]
    got = oracle.allreduce(ins, "avg")[0]
    u = Fraction(1, 1 << 24)
    gamma = (W + 1) * u / (1 - (W + 1) * u)  # W-1 adds, 1/W rounding, 1 multiply
    for i in range(200):
        exact = sum(Fraction(float(a[i])) for a in ins) / W
        mag = sum(abs(Fraction(float(a[i]))) for a in ins) / W
        assert abs(Fraction(float(got[i])) - exact) <= gamma * mag


def test_avg_scale_rounding_hand_derived():
    # avg multiplies the ring sum by fl32(1/W) once and casts after that:
    # for W = 3 and 5 this differs in the last bit from dividing by W, and
    # for bf16 output from casting the sum before the scale
    for line in _golden_lines("avg_scale_rounding.txt"):
        dt, xs, bits = (p.strip() for p in line.split(";"))
        xs = [float(v) for v in xs.split()]
        W, n = len(xs), 7
        if dt == "f32":
            dtype = oracle.F32
            ins = [np.full(n, v, np.float32) for v in xs]
        else:
            # the inputs are exact in bf16: the high half of their fp32 bits
            dtype = oracle.BF16
            ins = [np.full(n, np.float32(v).view(np.uint32) >> 16, np.uint16) for v in xs]
        want = int(bits, 16)
        ring = list(range(W))[::-1]
        for ufr in (None, ring):
            outs = oracle.allreduce(ins, "avg", dtype, ufr)
            outs += [np.concatenate(oracle.reduce_scatter(ins, "avg", dtype, ufr))]
            for o in outs:
                got = o.view(np.uint32 if dtype == oracle.F32 else np.uint16)
                assert [int(g) for g in got] == [want] * n, (line, ufr)


# ------------------------------------------------------------------- max

@pytest.mark.parametrize("W", [2, 3, 4, 8, 16])
def test_max_matches_numpy(W):
    rng = _rng(W + 99)
    n = 777
    ins = [rng.standard_normal(n).astype(np.float32) for _ in range(W)]
    want = np.maximum.reduce(ins)
    for got in oracle.allreduce(ins, "max"):
        assert np.array_equal(got, want)


def test_max_signed_zero_and_nan():
    pz, nz, nan = np.float32(0.0), np.float32(-0.0), np.float32(np.nan)
    ins = [np.array([pz, nz, nz, 1.0, nan], np.float32),
           np.array([nz, pz, nz, nan, 1.0], np.float32)]
    got = oracle.allreduce(ins, "max")[0]
    bits = got.view(np.uint32)
    assert bits[0] == 0x00000000 and bits[1] == 0x00000000  # +0 wins either order
    assert bits[2] == 0x80000000  # max(-0, -0) = -0
    assert bits[3] == 0x7FC00000 and bits[4] == 0x7FC00000  # canonical quiet NaN


# ------------------------------------------------------------------ bf16

def test_bf16_rne_golden():
    for line in _golden_lines("bf16_rne.txt"):
        fb, hb = line.split()
        f = np.array([int(fb, 16)], np.uint32).view(np.float32)
        assert oracle.bf16_from_f32(f)[0] == int(hb, 16), line


def test_bf16_matches_torch_cpu_conversion():
    torch = pytest.importorskip("torch")
    rng = _rng(5)
    bits = rng.integers(0, 1 << 32, 200_000, dtype=np.uint64).astype(np.uint32)
    # add exact ties and near-ties around many exponents
    hi = rng.integers(0, 1 << 16, 20_000, dtype=np.uint64).astype(np.uint32) << 16
    bits = np.concatenate([bits, hi | 0x8000, hi | 0x7FFF, hi | 0x8001])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_f32(f)
    assert np.array_equal(got, want)


def test_bf16_nan_stays_nan():
    f = np.array([0x7FC00000, 0xFFC00001, 0x7F800001, 0x7FBFFFFF], np.uint32).view(np.float32)
    h = oracle.bf16_from_f32(f).astype(np.uint32)
    assert all(((v & 0x7F80) == 0x7F80) and (v & 0x7F) != 0 and (v & 0x40) for v in h)


def test_bf16_allreduce_accumulates_in_fp32():
    # 256 + 1 + 1 is 258 in fp32, and 258 is a bf16 value; rounding to bf16
    # after every hop would lose the ones (256 + 1 -> 256 in bf16).
    def b(v):
        return oracle.bf16_from_f32(np.full(4, v, np.float32))
    ins = [b(256.0), b(1.0), b(1.0)]
    out = oracle.allreduce(ins, "sum", oracle.BF16)
    assert all(np.array_equal(o, b(258.0)) for o in out)


# ------------------------------------------------- RS / AG / AR identities

@pytest.mark.parametrize("W,n", [(2, 9), (3, 10), (4, 4096 + 3), (8, 1001), (16, 50)])
@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16])
@pytest.mark.parametrize("op", ["sum", "max", "avg"])
def test_allgather_of_reduce_scatter_is_allreduce(W, n, dtype, op):
    rng = _rng(W * n)
    vals = [rng.standard_normal(n).astype(np.float32) for _ in range(W)]
    ins = vals if dtype == oracle.F32 else [oracle.bf16_from_f32(v) for v in vals]
    ring = list(rng.permutation(W))
    rs = oracle.reduce_scatter(ins, op, dtype, ring)
    ag = oracle.allgather(rs, n, dtype, ring)
    ar = oracle.allreduce(ins, op, dtype, ring)
    for u in range(W):
        assert ag[u].tobytes() == ar[u].tobytes()
        assert ar[u].tobytes() == ar[0].tobytes()  # every rank holds the same
    assert np.concatenate(rs).tobytes() == ar[0].tobytes()


@pytest.mark.parametrize("W", [1, 2, 5, 8])
def test_allgather_is_concatenation(W):
    rng = _rng(W)
    n = 37
    segs = [rng.standard_normal(oracle.segment(n, W, j)[1]).astype(np.float32) for j in range(W)]
    want = np.concatenate(segs)
    for out in oracle.allgather(segs, n, oracle.F32, list(rng.permutation(W))):
        assert out.tobytes() == want.tobytes()


def test_single_rank_is_copy():
    rng = _rng(1)
    x = rng.standard_normal(100).astype(np.float32)
    x[3] = np.nan
    for op in ("sum", "max", "avg"):
        assert oracle.reduce_scatter([x], op)[0].tobytes() == x.tobytes()
        assert oracle.allreduce([x], op)[0].tobytes() == x.tobytes()


def test_empty_message_is_noop():
    ins = [np.empty(0, np.float32) for _ in range(4)]
    assert all(s.size == 0 for s in oracle.reduce_scatter(ins))
    assert all(s.size == 0 for s in oracle.allreduce(ins))


def test_invalid_arguments_rejected():
    x = [np.zeros(4, np.float32)] * 2
    with pytest.raises(ValueError):
        oracle.reduce_scatter(x, 7)
    with pytest.raises(ValueError):
        oracle.allreduce(x, "sum", oracle.F32, [0, 0])
    with pytest.raises(ValueError):
        oracle.segment(10, 0, 0)


@pytest.mark.parametrize("W,n", [(4, 1 << 12), (8, 1000), (3, 17), (16, 4099)])
@pytest.mark.parametrize("op", ["sum", "max", "avg"])
@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16])
def test_sampled_equals_full(W, n, op, dtype):
    rng = _rng(W + n)
    vals = [rng.standard_normal(n).astype(np.float32) for _ in range(W)]
    ins = vals if dtype == oracle.F32 else [oracle.bf16_from_f32(v) for v in vals]
    full = oracle.allreduce(ins, op, dtype)[0]
    idx = np.concatenate([[0, n - 1], rng.integers(0, n, 200)])
    samp = np.stack([np.asarray(a)[idx] for a in ins], axis=1)
    got = oracle.allreduce_sampled(samp, idx, n, op, dtype)
    assert got.tobytes() == full[idx].tobytes()


# ---------------------------------------------------------------- fusion

def test_fuse_plan_golden():
    for line in _golden_lines("horovod_fusion_batches.txt"):
        thr, sizes, begin = (p.strip() for p in line.split(";"))
        counts = [int(v) // 4 for v in sizes.split()]
        assert oracle.fuse_plan(counts, oracle.F32, int(thr)) == [int(v) for v in begin.split()]


def test_fuse_plan_greedy_properties():
    rng = _rng(3)
    counts = np.round(np.exp(rng.uniform(np.log(1024), np.log(4194304), 200))).astype(np.int64)
    thr = 64 << 20
    begin = oracle.fuse_plan(counts, oracle.F32, thr)
    assert begin[0] == 0 and begin[-1] == 200
    for b in range(len(begin) - 1):
        size = int(counts[begin[b]:begin[b + 1]].sum()) * 4
        assert size <= thr or begin[b + 1] - begin[b] == 1
        if begin[b + 1] < 200:  # greedy: the next tensor would not have fit
            assert size + int(counts[begin[b + 1]]) * 4 > thr


def test_pack_is_concatenation_and_unpack_inverts():
    rng = _rng(11)
    W, counts = 3, [5, 1, 17, 2, 8]
    tensors = [[rng.standard_normal(c).astype(np.float32) for c in counts] for _ in range(W)]
    fused = oracle.fuse_pack(tensors, counts, W)
    for u in range(W):
        assert fused[u].tobytes() == np.concatenate(tensors[u]).tobytes()
    back = oracle.fuse_unpack(fused, counts)
    for u in range(W):
        for t in range(len(counts)):
            assert back[u][t].tobytes() == tensors[u][t].tobytes()


def test_fusion_allreduce_integer_mean_exact():
    rng = _rng(12)
    W = 8
    counts = [1000, 3, 4097, 250, 1, 60]
    tensors = [[(rng.integers(-100, 101, c) * 8).astype(np.float32) for c in counts]
               for _ in range(W)]
    outs = oracle.fusion_allreduce(tensors, counts, "avg", oracle.F32, threshold_bytes=4 * 4100)
    for t, c in enumerate(counts):
        want = sum(tensors[u][t].astype(np.int64) for u in range(W)) // W
        for u in range(W):
            assert np.array_equal(outs[u][t].astype(np.int64), want)


def test_fusion_allreduce_is_batchwise_allreduce_of_concatenation():
    # The fused allreduce segments the whole batch, so its bits are those of
    # an allreduce of the concatenated tensors of each batch.
    rng = _rng(13)
    W = 4
    counts = [7, 300, 41, 1000, 5]
    thr = 4 * 400
    tensors = [[rng.standard_normal(c).astype(np.float32) for c in counts] for _ in range(W)]
    outs = oracle.fusion_allreduce(tensors, counts, "avg", oracle.F32, thr)
    begin = oracle.fuse_plan(counts, oracle.F32, thr)
    for b in range(len(begin) - 1):
        ts = range(begin[b], begin[b + 1])
        cat = [np.concatenate([tensors[u][t] for t in ts]) for u in range(W)]
        ar = oracle.allreduce(cat, "avg")
        for u in range(W):
            assert np.concatenate([outs[u][t] for t in ts]).tobytes() == ar[u].tobytes()


# ------------------------------------------------------------ min and prod

@pytest.mark.parametrize("W", [2, 3, 4, 8, 16])
def test_min_matches_numpy(W):
    rng = _rng(W + 199)
    ins = [rng.standard_normal(555).astype(np.float32) for _ in range(W)]
    want = np.minimum.reduce(ins)
    for got in oracle.allreduce(ins, "min"):
        assert np.array_equal(got, want)


def test_min_signed_zero_and_nan():
    pz, nz, nan = np.float32(0.0), np.float32(-0.0), np.float32(np.nan)
    ins = [np.array([pz, nz, pz, 1.0, nan], np.float32),
           np.array([nz, pz, pz, nan, 1.0], np.float32)]
    bits = oracle.allreduce(ins, "min")[0].view(np.uint32)
    assert bits[0] == 0x80000000 and bits[1] == 0x80000000  # -0 wins either order
    assert bits[2] == 0x00000000
    assert bits[3] == 0x7FC00000 and bits[4] == 0x7FC00000


def test_prod_ring_order_hand_derived():
    line = _golden_lines("ring_order_prod.txt")[0]
    want = [float(v) for v in line.split()]
    x = [np.full(4, v, np.float32) for v in (2.0 ** 100, 2.0 ** 100, 2.0 ** -100, 2.0 ** -100)]
    got = [float(s[0]) for s in oracle.reduce_scatter(x, "prod")]
    assert got == want


@pytest.mark.parametrize("W", [2, 3, 5, 8])
def test_prod_of_small_integers_exact(W):
    rng = _rng(W + 300)
    ins = [rng.choice(np.array([-2, -1, 1, 2, 3], np.float32), 400) for _ in range(W)]
    want = np.prod(np.stack([a.astype(np.int64) for a in ins]), axis=0)
    for got in oracle.allreduce(ins, "prod"):
        assert np.array_equal(got.astype(np.int64), want)


# ------------------------------------------------------------ allgatherv

@pytest.mark.parametrize("W", [1, 2, 3, 7])
def test_allgatherv_is_concatenation(W):
    rng = _rng(W + 400)
    pieces = [rng.standard_normal(int(rng.integers(0, 50))).astype(np.float32) for _ in range(W)]
    want = np.concatenate(pieces)
    for out in oracle.allgatherv(pieces, oracle.F32, list(rng.permutation(W))):
        assert out.tobytes() == want.tobytes()


def test_allgatherv_with_even_sizes_is_allgather():
    rng = _rng(401)
    n, W = 40, 4
    segs = [rng.standard_normal(oracle.segment(n, W, j)[1]).astype(np.float32) for j in range(W)]
    a = oracle.allgatherv(segs)
    b = oracle.allgather(segs, n)
    assert all(x.tobytes() == y.tobytes() for x, y in zip(a, b))


# ---------------------------------------- fp16 and the reduced-precision wire

def test_f16_rne_golden():
    for line in _golden_lines("f16_rne.txt"):
        fb, hb = line.split()[:2]
        f = np.array([int(fb, 16)], np.uint32).view(np.float32)
        assert oracle.f16_from_f32(f)[0] == int(hb, 16), line


def test_f16_matches_numpy_conversion():
    rng = _rng(77)
    bits = rng.integers(0, 1 << 32, 100_000, dtype=np.uint64).astype(np.uint32)
    # concentrate on the binary16 range, subnormals and the overflow edge
    mags = np.concatenate([rng.uniform(-30, 17, 100_000), rng.uniform(-26, -13, 50_000)])
    vals = (np.sign(rng.standard_normal(mags.size)) * 2.0 ** mags).astype(np.float32)
    hi = rng.integers(0, 1 << 19, 20_000, dtype=np.uint64).astype(np.uint32) << 13
    ties = (hi | 0x1000) + (0x70 << 23)
    f = np.concatenate([bits.view(np.float32), vals, ties.view(np.float32)])
    f = f[~np.isnan(f)]
    with np.errstate(over="ignore"):
        want = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f16_from_f32(f), want)


def test_f16_nan_stays_nan():
    # IEEE narrowing keeps a NaN a NaN (quiet), whatever its payload -- also
    # a signaling one whose payload lies only in the 13 bits binary16 drops.
    # (Passed one by one the values become Python floats, which quiets them;
    # the wire allreduce narrows the buffer's own bit patterns.)
    f = np.array([0x7FC00000, 0xFFC00001, 0x7F800001, 0x7FBFFFFF, 0xFF801FFF],
                 np.uint32).view(np.float32)
    h = oracle.f16_from_f32(f).astype(np.uint32)
    assert all(((v & 0x7C00) == 0x7C00) and (v & 0x3FF) != 0 and (v & 0x200) for v in h)
    for wire in ("f16", "bf16"):
        out = oracle.allreduce_wire([f.copy()], wire, "sum")[0]  # one rank: a round trip
        assert np.all(np.isnan(out)), wire


def test_f16_widening_matches_numpy_for_all_patterns():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f32_from_f16(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_wire_hop_rounding_hand_derived():
    for line in _golden_lines("wire_hop_rounding.txt"):
        wire, xs, res, *rest = (p.strip() for p in line.split(";"))
        op = rest[0] if rest else "sum"
        x = [np.full(3, float(v), np.float32) for v in xs.split()]
        want = [float(v) for v in res.split()]
        got = oracle.allreduce_wire(x, wire, op)
        for u in range(3):
            assert list(got[u]) == want, (wire, op)


@pytest.mark.parametrize("wire", ["f16", "bf16"])
@pytest.mark.parametrize("W", [2, 3, 8])
def test_wire_integer_sums_exact(wire, W):
    # integers up to 256 are exact in both wire types and every partial sum
    # here stays below 256
    rng = _rng(W + 500)
    ins = [rng.integers(-16, 17, 300).astype(np.float32) for _ in range(W)]
    want = np.sum(np.stack([a.astype(np.int64) for a in ins]), axis=0)
    for out in oracle.allreduce_wire(ins, wire, "sum"):
        assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("wire", ["f16", "bf16"])
def test_wire_single_rank_is_round_trip(wire):
    rng = _rng(501)
    x = rng.standard_normal(1000).astype(np.float32)
    conv = oracle.f16_from_f32 if wire == "f16" else oracle.bf16_from_f32
    back = oracle.f32_from_f16 if wire == "f16" else \
        (lambda h: (h.astype(np.uint32) << 16).view(np.float32))
    got = oracle.allreduce_wire([x], wire, "sum")[0]
    assert got.tobytes() == back(conv(x)).tobytes()


def test_wire_within_hop_rounding_bound():
    # each of the W-1 hops rounds relatively by at most u_wire, plus the
    # input conversion: |wire result - exact| <= ((W-1) + 1) u_w sum|x| (+ tiny)
    rng = _rng(502)
    W = 8
    ins = [rng.standard_normal(2000).astype(np.float32) for _ in range(W)]
    exact = np.sum(np.stack(ins).astype(np.float64), axis=0)
    mag = np.sum(np.abs(np.stack(ins).astype(np.float64)), axis=0)
    for wire, u in (("f16", 2.0 ** -11), ("bf16", 2.0 ** -8)):
        got = oracle.allreduce_wire(ins, wire, "sum")[0].astype(np.float64)
        gam = W * u / (1 - W * u)
        assert np.all(np.abs(got - exact) <= gam * mag + 2.0 ** -24)


# ------------------------------------------------- sparsified allreduce

def test_sparse_allreduce_hand_derived():
    x = [np.array([3, -1, 0.5, 2], np.float32), np.array([1, 4, -2, 0.1], np.float32)]
    for line in _golden_lines("singa_sparse_allreduce.txt"):
        mode, thr, res, r0, r1 = (p.strip() for p in line.split(";"))
        acc = [np.zeros(4, np.float32), np.zeros(4, np.float32)]
        outs, nnz = oracle.sparse_allreduce(x, float(thr), mode == "topk", acc)
        want = np.array([float(v) for v in res.split()], np.float32)
        assert all(np.array_equal(o, want) for o in outs), mode
        assert np.array_equal(acc[0], np.array([float(v) for v in r0.split()], np.float32))
        assert np.array_equal(acc[1], np.array([float(v) for v in r1.split()], np.float32))
    x = [np.array([v], np.float32) for v in (1.0, 1e8, -1e8)]
    assert float(oracle.sparse_allreduce(x, 0.5)[0][0][0]) == 0.0


def _golden_cases(name):
    """Blocks of a "case <name>" golden file as dicts of lists of fp32 arrays."""
    def val(tok):
        if tok.startswith("0x"):
            return np.array([int(tok, 16)], np.uint32).view(np.float32)[0]
        return np.float32(float(tok))
    cases, cur = [], None
    for line in _golden_lines(name):
        key, *toks = line.split()
        if key == "case":
            cur = {"name": toks[0]}
            cases.append(cur)
        elif key in ("threshold",):
            cur[key] = float(toks[0])
        elif key == "nnz":
            cur[key] = [int(t) for t in toks]
        else:
            cur.setdefault(key, []).append(np.array([val(t) for t in toks], np.float32))
    return cases


def test_sparse_topk_ties_and_signed_zero_hand_derived():
    # ties across the cut keep the lower indices; a kept -0 leaves a -0
    # residual (the sent values are added into zeros first) and adds +0
    for c in _golden_cases("singa_topk_ties_signed_zero.txt"):
        acc = [a.copy() for a in c["acc"]]
        outs, nnz = oracle.sparse_allreduce(c["in"], c["threshold"], True, acc)
        for o in outs:
            assert o.tobytes() == c["result"][0].tobytes(), c["name"]
        for a, want in zip(acc, c["residual"]):
            assert a.tobytes() == want.tobytes(), c["name"]
        assert list(nnz) == c["nnz"], c["name"]


def _keys(a):
    u = a.view(np.uint32).astype(np.uint64)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)


def _dense_reference(xs, kept):
    # zeros, then each rank's kept values in rank order (fp32 adds)
    res = np.zeros(xs[0].size, np.float32)
    for x, k in zip(xs, kept):
        res = np.where(k, (res + x).astype(np.float32), res)
    return res


@pytest.mark.parametrize("W", [1, 2, 3, 8])
@pytest.mark.parametrize("with_acc", [False, True])
def test_sparse_threshold_matches_dense_definition(W, with_acc):
    rng = _rng(600 + W)
    n = 5000
    xs = [(rng.standard_normal(n) * 10.0 ** rng.integers(-2, 2, n)).astype(np.float32)
          for _ in range(W)]
    acc = [(rng.standard_normal(n) * 0.1).astype(np.float32) for _ in range(W)] if with_acc \
        else None
    acc0 = [a.copy() for a in acc] if with_acc else None
    thr = 0.7
    outs, nnz = oracle.sparse_allreduce(xs, thr, False, acc)
    eff = [(x + a).astype(np.float32) for x, a in zip(xs, acc0)] if with_acc else xs
    kept = [(np.abs(e) > thr) & (e != 0) for e in eff]
    want = _dense_reference(eff, kept)
    for o in outs:
        assert o.tobytes() == want.tobytes()
    assert list(nnz) == [int(k.sum()) for k in kept]
    if with_acc:
        for a, e, k in zip(acc, eff, kept):
            assert np.array_equal(a, np.where(k, np.float32(0), e))


@pytest.mark.parametrize("W", [1, 2, 5])
@pytest.mark.parametrize("frac", [0.0, 0.001, 0.05, 0.5, 1.0])
def test_sparse_topk_matches_sorted_selection(W, frac):
    rng = _rng(700 + W)
    n = 3001
    xs = [rng.standard_normal(n).astype(np.float32) for _ in range(W)]
    xs[0][::7] = 0.25  # ties across the selection boundary for some fractions
    acc = [np.zeros(n, np.float32) for _ in range(W)]
    outs, nnz = oracle.sparse_allreduce(xs, frac, True, acc)
    K = min(n, int(np.ceil(np.float32(frac) * np.float32(n))))
    kept = []
    for x in xs:
        order = np.lexsort((np.arange(n), -_keys(x).astype(np.int64)))  # value desc, index asc
        k = np.zeros(n, bool)
        k[order[:K]] = True
        kept.append(k)
    want = _dense_reference(xs, kept)
    for o in outs:
        assert o.tobytes() == want.tobytes()
    assert list(nnz) == [K] * W
    for a, x, k in zip(acc, xs, kept):
        assert np.array_equal(a, np.where(k, np.float32(0), x))


def test_sparse_topk_count_rounding():
    # K = ceil(threshold * n) in fp32, as the page computes it: 0.1f * 10
    # rounds to exactly 1 in fp32 (K = 1), where double gives 1.0000000149
    # (K = 2)
    for n, thr, K in ((10, 0.25, 3), (1000, 0.01, 10), (7, 1.0, 7), (100, 0.0, 0), (3, 0.34, 2),
                      (10, 0.1, 1)):
        xs = [np.arange(n, dtype=np.float32)]
        _, nnz = oracle.sparse_allreduce(xs, thr, True)
        assert nnz[0] == K, (n, thr)

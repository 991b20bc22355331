"""The no-allocation sparsified allreduce, for callers that must not allocate
device memory themselves (a framework whose pool owns the device, a callback
that must not block on cudaMalloc, a loop that sets every resource up front).

It is called through the C ABI and must give exactly what the entry point
with a caller-provided workspace gives, on two calls in a row: the fixed
working memory inside the library keeps the previous call's contents, so the
second call checks that everything that must start at zero is cleared.
This file is collected last on purpose.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v():
    from collective_reduction_virtual_gb300 import build
    build.build()
    import collective_reduction_virtual_gb300 as vc
    return vc


def _ptrs(ts):
    return [t.data_ptr() for t in ts]


# What the fixed 1 MiB leaves beyond the minimum is candidate-list room:
# - n = 2^20 + 3: about 15K entries per rank, too few for K = 1 % (3K = 31K),
#   so the select passes read the whole array;
# - n = 2^18 + 5, K = 1 %: 3K = 7.9K entries fit, so the candidate lists and
#   the output from the lists are used;
# - n = 62.6 M: the minimum nearly fills the array and leaves 56 entries per
#   rank; K = 16 (3K = 48) still asks for the lists, which the sampled bound
#   can overflow, sending a rank back to the whole-array passes.
@pytest.mark.parametrize("topk,frac,n", [(True, 0.01, (1 << 20) + 3), (True, 0.3, (1 << 20) + 3),
                                         (False, 0.9, (1 << 20) + 3),
                                         (True, 0.01, (1 << 18) + 5),
                                         (True, 2.5e-7, 62_600_000)])
def test_noalloc_matches_workspace_entry_two_calls_in_a_row(v, topk, frac, n):
    W = 8
    g = torch.Generator(device="cuda")
    g.manual_seed(2026)
    ins = [torch.randn(n, generator=g, device="cuda") for _ in range(W)]
    acc_a = [torch.randn(n, generator=g, device="cuda") * 0.1 for _ in range(W)]
    acc_b = [a.clone() for a in acc_a]
    out_a = [torch.empty(n, device="cuda") for _ in range(W)]
    out_b = [torch.empty(n, device="cuda") for _ in range(W)]
    nnz_a = torch.empty(W, dtype=torch.int64, device="cuda")
    nnz_b = torch.empty(W, dtype=torch.int64, device="cuda")
    # the minimum fits the fixed memory; the caller's workspace is the
    # recommended size, so for top-K the two entries may take different select
    # paths (candidate lists or whole-array passes) and must still agree
    assert v.vcoll_sparse_workspace_min_bytes(W, n, topk) <= v.SPARSE_NOALLOC_BYTES
    ws_bytes = v.vcoll_sparse_workspace_bytes(W, n, topk)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        rc = v.vcoll_sparse_allreduce_noalloc(_ptrs(ins), _ptrs(out_a), _ptrs(acc_a), W, n, frac,
                                              topk, nnz_a.data_ptr(), stream)
        assert rc == v.OK, v.last_error()
        rc = v.vcoll_sparse_allreduce(_ptrs(ins), _ptrs(out_b), _ptrs(acc_b), W, n, frac, topk,
                                      nnz_b.data_ptr(), ws.data_ptr(), ws_bytes, stream)
        assert rc == v.OK, v.last_error()
        torch.cuda.synchronize()
        # the sparsified allreduce is bit-exact in every test of this library
        for u in range(W):
            assert torch.equal(out_a[u].view(torch.int32), out_b[u].view(torch.int32)), (call, u)
            assert torch.equal(acc_a[u].view(torch.int32), acc_b[u].view(torch.int32)), (call, u)
        assert torch.equal(nnz_a, nnz_b), call


def test_noalloc_rejects_sizes_beyond_its_fixed_memory(v):
    # 64 ranks of 2^24 elements need far more than the fixed 1 MiB; the call
    # fails on the host before touching the device
    W, n = 64, 1 << 24
    assert v.vcoll_sparse_workspace_min_bytes(W, n, True) > v.SPARSE_NOALLOC_BYTES
    fake = [0x100000 * (u + 1) for u in range(W)]
    rc = v.vcoll_sparse_allreduce_noalloc(fake, fake, None, W, n, 0.01, True)
    assert rc == v.ERR_INVALID_ARG
    assert "working memory" in v.last_error()

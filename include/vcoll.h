/*
 * vcoll.h -- C ABI of the virtual-rank collective library for one GB300 GPU.
 *
 * A "virtual rank" is one device buffer.  W ranks live in the HBM of the
 * current CUDA device; the collectives combine them element by element inside
 * single kernel launches.  There is no second GPU, peer access or NCCL.
 *
 * Common conventions for every entry point below
 * ------------------------------------------------
 *  - Pointer arrays (`in`, `out`, `tensors`, `fused`) are HOST arrays of
 *    DEVICE pointers on the current device.  Pinned host memory
 *    (cudaHostAlloc / cudaHostRegister) is accepted too: with unified
 *    addressing its host pointer is a device pointer, and the kernels then
 *    read and write it directly over the CPU-GPU link, which is faster than
 *    staging copies in and out.  Each device pointer must be
 *    aligned to the element size.  Any 16-byte phase works.  Reduce-scatter,
 *    allreduce and allgather use 16-byte vectors whenever their outputs share
 *    a phase (each reduce-scatter output on a grid of its own), realigning
 *    inputs at other phases on the fly; the other entry points when all their
 *    buffers share one.  Otherwise an element-wise path gives the same bits,
 *    more slowly.
 *  - `n` counts elements per rank (int64).  Segment j of an n-element buffer
 *    is [off_j, off_j + len_j) with q = n / W, r = n % W,
 *    off_j = j*q + min(j, r), len_j = q + (j < r): contiguous, the first r
 *    segments one element longer (vcoll_segment computes it).  When W divides
 *    n this is NCCL's layout (block j at j * recvcount).
 *  - Ownership: the caller owns every buffer; the library allocates no device
 *    memory and keeps no pointer after the call returns.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Work is enqueued asynchronously on it; nothing
 *    synchronises the host.
 *  - Errors: every call returns a vcoll_status_t.  Argument errors are found
 *    on the host before anything is enqueued.  vcoll_last_error() returns a
 *    thread-local message for the last failure on the calling thread.
 *  - Types: VCOLL_F32 and VCOLL_BF16.  Arithmetic is fp32 for both; bf16
 *    inputs are widened exactly and outputs rounded to nearest even once (a
 *    NaN keeps its sign and top payload bits and is made quiet: the
 *    canonical fp32 NaN becomes 0x7FC0).  Subnormals are kept (no flush to
 *    zero).
 *  - Ops: VCOLL_SUM, VCOLL_MAX, VCOLL_AVG (sum times fl32(1/W), applied once
 *    to the finished sum), VCOLL_MIN, VCOLL_PROD (one fp32 multiply per hop).
 *    max: a NaN operand gives the canonical quiet NaN; +0 wins over -0;
 *    otherwise the larger value.  min: the mirror image (-0 wins over +0).
 *  - Order: with VCOLL_FLAG_RING_ORDER each element of segment j is folded
 *    in ring order -- starting at rank (j+1) mod W, accumulator first, ending
 *    at rank j -- which reproduces the early NCCL ring bit for bit.  Without
 *    it the library uses its fastest order (a pairwise tree for W in
 *    {4, 8, 16}); results then differ from ring order only by float
 *    reassociation.  max and min are the same in every order.
 *  - Special cases: n == 0 returns VCOLL_OK without enqueuing anything;
 *    W == 1 is a device-to-device copy (nothing when in and out coincide).
 *
 * Sources: early NCCL "src/reduce_scatter.cu" (pytorch mirror) for the ring
 * schedule (GetBlock, ReduceScatterKernel) and the error conventions
 * (ncclInvalidType / ncclInvalidOperation, recvcount == 0, nDev == 1);
 * "Distributed primitives" notes for all-reduce / all-gather /
 * reduce-scatter semantics and ring allreduce = reduce-scatter + allgather;
 * Horovod "horovod/common/operations.cc" (PerformOperation, fusion batching in
 * BackgroundThreadLoop) and Apache SINGA "src/io/communicator.cc"
 * (Communicator::fusedSynch) for tensor fusion; MLX PR #3901 ("Add scatter
 * reduce for JACCL") for the latency-bound path at <= 32 KB and the in-place
 * read-before-write rule.
 */
#ifndef VCOLL_H_
#define VCOLL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VCOLL_MAX_RANKS 64

typedef enum {
  VCOLL_F32 = 0,
  VCOLL_BF16 = 1,
  VCOLL_F16 = 2 /* IEEE binary16: only as the wire type of vcoll_allreduce_wire */
} vcoll_dtype_t;

typedef enum {
  VCOLL_SUM = 0,
  VCOLL_MAX = 1,
  VCOLL_AVG = 2,
  VCOLL_MIN = 3, /* NCCL FuncMin */
  VCOLL_PROD = 4 /* NCCL FuncProd */
} vcoll_op_t;

typedef enum {
  VCOLL_OK = 0,
  VCOLL_ERR_INVALID_ARG = 1,  /* null pointer, W out of [1, 64], n < 0, misaligned
                                 pointer, or an overlap other than the allowed
                                 in-place forms */
  VCOLL_ERR_INVALID_TYPE = 2, /* dtype not a vcoll_dtype_t (ncclInvalidType) */
  VCOLL_ERR_INVALID_OP = 3,   /* op not a vcoll_op_t (ncclInvalidOperation) */
  VCOLL_ERR_UNSUPPORTED = 4,  /* a valid request this build does not handle */
  VCOLL_ERR_CUDA = 5          /* a CUDA runtime call or launch failed */
} vcoll_status_t;

/* Fold each segment in ring order (bit-exact with the NCCL ring). */
#define VCOLL_FLAG_RING_ORDER 0x1u
/* Force the variant that stages the W input tiles through shared memory with
 * bulk asynchronous copies (TMA), or the variant that loads straight into
 * registers.  Without either flag the library picks by message size.  Both
 * give identical bits.  The staged variant runs on device memory only: when
 * any buffer is pinned host or managed memory (cudaPointerGetAttributes), a
 * staged request runs the direct kernels. */
#define VCOLL_FLAG_STAGED 0x2u
#define VCOLL_FLAG_DIRECT 0x4u

/*
 * Reduce-scatter ("Distributed primitives", section 3; NCCL
 * ncclReduceScatter).  in[u]: n elements of rank u.  out[j]: receives the
 * len_j elements of segment j of the element-wise reduction of all W inputs.
 * In place: out[j] == (char*)in[j] + off_j * elemsize (NCCL's convention) or
 * any out/in pair with the same element mapping; other overlaps are
 * rejected.
 */
int vcoll_reduce_scatter(const void* const* in, void* const* out, int W, int64_t n, int dtype,
                         int op, unsigned flags, void* stream);

/*
 * Allgather ("Distributed primitives", section 2; ring allreduce's second
 * half).  in[j]: the len_j elements of segment j.  out[u]: receives all n
 * elements (segment j at off_j) on every rank u.  op is checked but unused.
 * In place: in[j] == (char*)out[u] + off_j * elemsize for some u.
 */
int vcoll_allgather(const void* const* in, void* const* out, int W, int64_t n, int dtype, int op,
                    unsigned flags, void* stream);

/*
 * Allgather with per-rank sizes (Horovod's allgatherv path: every rank's
 * tensor, first dimensions possibly different, concatenated in rank order on
 * every rank).  in[j]: counts[j] elements (counts: host array of W).
 * out[u]: receives counts[0] + ... + counts[W-1] elements, piece j at
 * counts[0] + ... + counts[j-1].  In place: in[j] == (char*)out[u] + that
 * offset * elemsize.
 */
int vcoll_allgatherv(const void* const* in, const int64_t* counts, void* const* out, int W,
                     int dtype, void* stream);

/*
 * Allreduce ("Distributed primitives", section 1 and ring allreduce =
 * reduce-scatter + allgather; Horovod / SINGA ncclAllReduce call sites).
 * in[u]: n elements; out[u]: n elements, all W outputs receive the same
 * result.  One kernel pass reads the W inputs once and writes the W outputs
 * from registers; its bits equal reduce-scatter followed by allgather.
 * In place: out[u] == in[u] (Horovod's in-place fusion-buffer allreduce).
 */
int vcoll_allreduce(const void* const* in, void* const* out, int W, int64_t n, int dtype, int op,
                    unsigned flags, void* stream);

/*
 * Ring order on a user ring (early NCCL src/reduce_scatter.cu: GetBlock maps
 * a ring position and step to a block through comm->userFromRing, and the
 * schedule comment of ncclReduceScatterWithTypeAndFunc works a 4-GPU ring
 * userFromRing = {1, 2, 0, 3}).  user_from_ring[p] is the rank at ring
 * position p, a permutation of 0 .. W-1 (host array of W ints; NULL: the
 * identity ring, the same as VCOLL_FLAG_RING_ORDER).  Segment j is folded
 * the way the ring reduce-scatter folds block j: it starts with the rank at
 * the ring position after rank j's, takes the following positions' ranks in
 * ring order (accumulator first), and ends at rank j.  The result is written
 * as by vcoll_reduce_scatter / vcoll_allreduce (an allreduce holds the
 * reduce-scatter's segments in every output: its allgather is a bit copy).
 * Arguments, aliasing and errors as vcoll_reduce_scatter / vcoll_allreduce;
 * a user_from_ring that is not a permutation gives VCOLL_ERR_INVALID_ARG.
 * max and min give the same bits in every order.
 */
int vcoll_reduce_scatter_ring(const void* const* in, void* const* out, int W, int64_t n,
                              int dtype, int op, const int* user_from_ring, void* stream);
int vcoll_allreduce_ring(const void* const* in, void* const* out, int W, int64_t n, int dtype,
                         int op, const int* user_from_ring, void* stream);

/*
 * Reduced-precision ("wire") allreduce, Apache SINGA Communicator::synchHalf /
 * fusedSynchHalf: fp32 inputs are converted to the 16-bit wire type (wire =
 * VCOLL_F16 as SINGA's float2half, or VCOLL_BF16), allreduced in that type by
 * the NCCL ring, whose buffers hold wire values so every hop rounds to the
 * wire type, and converted back to fp32 (half2float).  One pass: each
 * element is rounded, folded with a rounding after every op (ring order with
 * VCOLL_FLAG_RING_ORDER, else a pairwise tree), and the widened result is
 * written to the W fp32 outputs.  in[u], out[u]: n fp32 elements.  op: sum or
 * avg (the rounded sum times fl32(1/W), rounded again); max/min/prod give
 * VCOLL_ERR_UNSUPPORTED.  W == 1 is the round trip through the wire type.
 */
int vcoll_allreduce_wire(const void* const* in, void* const* out, int W, int64_t n, int wire, int op,
                         unsigned flags, void* stream);

/*
 * Tensor-fusion batching (Horovod BackgroundThreadLoop): greedy in tensor
 * order; a batch starts with the next tensor (even one above the threshold)
 * and takes the following tensors while the fused byte size stays
 * <= threshold_bytes.  counts[T] (host) are element counts; batch_begin
 * (host, T + 1 ints) receives the first tensor of each batch followed by T;
 * *nbatches the number of batches.  Host only, no GPU work.
 */
int vcoll_fuse_plan(const int64_t* counts, int T, int dtype, int64_t threshold_bytes,
                    int* batch_begin, int* nbatches);

/*
 * Fusion pack (Horovod PerformOperation "memcpy in fusion buffer"; SINGA
 * fusedSynch): fused[u] receives tensors[u*T + t] for t = 0..T-1 back to back,
 * no padding (tensor t at element offset counts[0] + ... + counts[t-1]).
 * tensors: host array of W*T device pointers, rank-major.  counts: host.
 * One kernel launch per up to 64 tensors (fewer when W*T would exceed 1024);
 * no buffer may overlap another.
 */
int vcoll_fuse_pack(const void* const* tensors, const int64_t* counts, int T, void* const* fused,
                    int W, int dtype, void* stream);

/* Fusion unpack: the inverse of vcoll_fuse_pack. */
int vcoll_fuse_unpack(const void* const* fused, const int64_t* counts, int T,
                      void* const* tensors, int W, int dtype, void* stream);

/*
 * Multi-tensor allreduce: Horovod's tensor fusion (PerformOperation: pack into
 * the fusion buffer, ncclAllReduce it in place, unpack; SINGA fusedSynch)
 * without the fusion buffer.  For each rank u the T tensors in[u*T + t] form
 * one virtual buffer of n = counts[0] + ... + counts[T-1] elements (tensor t at
 * offset counts[0] + ... + counts[t-1]); the allreduce of the W virtual
 * buffers is written to out[u*T + t].  The result has the bits of
 * vcoll_fuse_pack -> vcoll_allreduce (in place, same flags) ->
 * vcoll_fuse_unpack of the same batch, but every byte moves once (2*W*n*elemsize
 * instead of 6*W*n*elemsize).  Call it once per batch of vcoll_fuse_plan.
 * in, out: host arrays of W*T device pointers, rank-major; counts: host.  In
 * place: out[e] == in[e].  One launch per up to 64 tensors (fewer when W*T
 * would exceed 768).
 */
int vcoll_allreduce_multi(const void* const* in, void* const* out, const int64_t* counts, int T,
                          int W, int dtype, int op, unsigned flags, void* stream);

/*
 * Tensor-fusion allreduce, planned and executed in one call: the Horovod
 * batches of vcoll_fuse_plan(counts, T, dtype, threshold_bytes) are each
 * allreduced as in vcoll_allreduce_multi (each batch segmented on its own,
 * exactly as its fusion buffer would be), with the pieces of all batches
 * sharing kernel launches.  *nbatches (may be NULL) receives the batch count.
 * Same arguments and aliasing rules as vcoll_allreduce_multi; the bits equal
 * pack -> vcoll_allreduce -> unpack per batch.
 */
int vcoll_fusion_allreduce(const void* const* in, void* const* out, const int64_t* counts, int T,
                           int W, int dtype, int op, unsigned flags, int64_t threshold_bytes,
                           int* nbatches, void* stream);

/*
 * Tensor fusion through fusion buffers, Horovod operations.cc PerformOperation
 * (the NCCL allreduce path): the tensors are planned into the batches of
 * vcoll_fuse_plan(counts, T, dtype, threshold_bytes); for each batch of two or
 * more tensors every rank's tensors are copied back to back into that rank's
 * fusion buffer fused[u] (MEMCPY_IN_FUSION_BUFFER), the W buffers are
 * allreduced in place (NCCL_ALLREDUCE), and the results are copied out to
 * the output tensors (MEMCPY_OUT_FUSION_BUFFER); a batch of one tensor is
 * allreduced straight from its input to its output, as Horovod does with a
 * single entry.  The same fusion buffers serve every batch, in order, on
 * `stream`: the whole pipeline (3 launches per fused batch) runs from one
 * call.  The bits equal vcoll_fusion_allreduce's.
 * in, out: host arrays of W*T device pointers, rank-major; out[e] may equal
 * in[e] (in place), no other tensor may overlap another.  counts: host, T
 * element counts.  fused: host array of W device pointers, each to
 * fused_bytes bytes that overlap no tensor; every batch of two or more
 * tensors must fit (VCOLL_ERR_INVALID_ARG otherwise, before anything is
 * enqueued).  *nbatches (may be NULL) receives the batch count.  Other
 * arguments and errors as vcoll_allreduce.
 */
int vcoll_fusion_allreduce_buffered(const void* const* in, void* const* out,
                                    const int64_t* counts, int T, void* const* fused,
                                    int64_t fused_bytes, int W, int dtype, int op, unsigned flags,
                                    int64_t threshold_bytes, int* nbatches, void* stream);

/*
 * Sparsified allreduce with error feedback (Apache SINGA
 * Communicator::valSparsAllReduce, topK == false, and topKSparsAllReduce,
 * topK == true), fp32.  Per rank u: x = in[u] (+ accum[u] when accum is not
 * NULL).  threshold mode: the entries with |x| > threshold survive (and
 * x != 0); top-K mode: the K = ceil(threshold * n) entries (threshold in
 * [0, 1], computed in fp32 as SINGA does) with the largest values survive,
 * ties broken toward the lower index; values are ordered by their bits (-0
 * just below +0, NaNs beyond the infinities by sign -- with accum, where a
 * NaN comes from the sum in + accum its sign is the GPU's, which IEEE 754
 * leaves open).  With accum, accum[u] becomes x minus
 * the sent values: x elsewhere; where an entry survived, x - x in threshold
 * mode and x - (0 + x) in top-K mode (the sent values are scattered into
 * zeros first): zero for a finite x (-0 for a kept -0 in top-K mode), NaN for
 * an infinite one.  Every out[u]
 * receives the sum of all ranks' survivors, added into zeros rank by rank --
 * what the allgathered sparse lists scattered with cusparseSaxpyi give.
 * nnz (device, W int64, may be NULL) receives each rank's survivor count.
 * workspace: device memory of workspace_bytes bytes, 16-byte aligned, owned
 * by the caller, not kept after the call; calls that share a workspace must
 * not overlap.  Threshold mode needs none.  Top-K needs at least
 * vcoll_sparse_workspace_min_bytes(W, n, 1) (about n/1024 bytes + 8 KiB per
 * rank; smaller gives VCOLL_ERR_INVALID_ARG); vcoll_sparse_workspace_bytes(W,
 * n, 1) (about n bytes + 40 KiB per rank) adds room for candidate lists, which lets the
 * select passes after the first read only the entries above a sampled bound
 * instead of the whole array, and for small K lets the output come from the
 * lists (the same results, about three times as fast at K = 1 % of n; a size
 * in between gives smaller lists, and a rank whose list does not fit falls
 * back to the passes over the whole array).
 * In place: out[u] == in[u].
 */
size_t vcoll_sparse_workspace_bytes(int W, int64_t n, int topk);
size_t vcoll_sparse_workspace_min_bytes(int W, int64_t n, int topk);
int vcoll_sparse_allreduce(const void* const* in, void* const* out, void* const* accum, int W,
                           int64_t n, float threshold, int topk, int64_t* nnz, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * vcoll_sparse_allreduce without a caller workspace, for code that may not
 * allocate device memory (a framework that owns the whole device through its
 * own pool, a callback that must not block on cudaMalloc, a loop that must
 * have every resource in place before it starts).  The top-K working memory
 * is a fixed array inside the library, 1 MiB (VCOLL_SPARSE_NOALLOC_BYTES) on
 * every GPU that loads it, held until the process exits;
 * the call allocates nothing.  Arguments and results are those of
 * vcoll_sparse_allreduce; sizes whose minimum working memory would not fit
 * (vcoll_sparse_workspace_min_bytes(W, n, 1) > the maximum, about n <= 120 Mi
 * elements at W = 8) return VCOLL_ERR_INVALID_ARG with an explanation, and
 * what the array holds beyond that minimum is candidate-list room (enough
 * for the fast path up to a few million entries over all ranks at K = 1 %).  The
 * threshold mode needs no working memory and passes straight through.
 * The first top-K call on a device looks up the array's device address with
 * cudaGetSymbolAddress (again after the device's context changes, as after
 * cudaDeviceReset); make that first call before capturing a stream.
 * All calls share the one array and it keeps the last call's contents (the
 * call clears what must start at zero), so calls that may run at the same
 * time on the GPU -- on different streams, or from different threads --
 * race on it: order them on one stream.
 * The pages have no counterpart of this entry point.
 */
#define VCOLL_SPARSE_NOALLOC_BYTES (1u << 20)
int vcoll_sparse_allreduce_noalloc(const void* const* in, void* const* out, void* const* accum,
                                   int W, int64_t n, float threshold, int topk, int64_t* nnz,
                                   void* stream);

/* Device-side error bits, OR-ed into one word per device by the kernels.
 * The staged kernels bound every wait on their shared-memory barriers (2 s of
 * wall-clock time); a wait that gives up records VCOLL_DEVICE_ERR_TIMEOUT and
 * the kernel returns early (its outputs are then incomplete). */
#define VCOLL_DEVICE_ERR_TIMEOUT 0x1u

/* Reads the current device's error word into *flags (and resets it when
 * clear != 0).  Synchronous: waits for all work on the device to finish. */
int vcoll_device_errors(unsigned* flags, int clear);

/* Diagnostics for the bounded waits: launches one thread that waits on a
 * shared-memory barrier nothing ever arrives at; the wait gives up after
 * limit_us microseconds (1 .. 10^6) and records VCOLL_DEVICE_ERR_TIMEOUT in
 * the device error word, and the kernel returns -- the device stays usable.
 * Read the word with vcoll_device_errors.  Asynchronous on `stream`. */
int vcoll_selftest_wait_timeout(unsigned limit_us, void* stream);

/* Segment j of an n-element buffer over W ranks (host only). */
int vcoll_segment(int64_t n, int W, int j, int64_t* off, int64_t* len);

/* Static description of a status code. */
const char* vcoll_status_string(int status);

/* Thread-local detail of the last failing call on this thread ("" if none). */
const char* vcoll_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int vcoll_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VCOLL_H_ */

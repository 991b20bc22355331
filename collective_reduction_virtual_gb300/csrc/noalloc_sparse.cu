// vcoll_sparse_allreduce_noalloc: the sparsified allreduce for callers that
// cannot allocate device memory.
//
// Who cannot allocate: code that runs where cudaMalloc is off limits -- inside
// a framework whose memory pool owns the whole device and forbids outside
// allocations, in a plugin or callback that must not grow the process's
// footprint or must not synchronise (cudaMalloc and cudaFree can block the
// whole device), or in a real-time loop that has to have every resource in
// place before it starts.  Such callers still own their input and output
// buffers, but have no way to hand the top-K selection its working memory.
//
// This entry point keeps that working memory in a fixed array compiled into
// the library (kNoAllocScratchBytes, 1 MiB), so the call itself allocates
// nothing.  Every GPU that loads the library holds the array until the
// process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "vcoll_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = VCOLL_SPARSE_NOALLOC_BYTES;

// The working memory.  In host code this name is only a stand-in for the
// device array: its device address must be looked up per device (below) and
// never taken from the name itself.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The address is looked up once per device and context.  A device's context
// can be replaced within one process (cudaDeviceReset, or a caller that makes
// its own context current), and the new context loads the library's module
// afresh, so the array may then sit at another address: the cache keeps the
// id of the context it was resolved in and resolves again when the current
// one differs.  The context functions come from the driver through the
// runtime's entry-point query, so the library does not link libcuda.
constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;  // 0: not resolved
  void* addr;
};
std::mutex g_mu;
ScratchSlot g_slot[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
std::once_flag g_driver_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The id of the context current on this thread, or 0 when none is current or
// the driver does not provide the query.
unsigned long long current_context_id() {
  std::call_once(g_driver_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = (CtxGetCurrentFn)f;
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = (CtxGetIdFn)f;
  });
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Looks up the array's device address on the current device, with that
// device current: once per device and context (every call, if the context
// cannot be identified).
int scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return vcoll::report_error(VCOLL_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return vcoll::report_error(VCOLL_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  unsigned long long id = current_context_id();
  if (id && g_slot[dev].ctx_id == id) {
    *addr = g_slot[dev].addr;
    return VCOLL_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the fixed scratch failed: %s",
             cudaGetErrorString(e));
    return vcoll::report_error(VCOLL_ERR_CUDA, msg);
  }
  // the lookup makes the runtime's context current if none was
  if (!id) id = current_context_id();
  g_slot[dev].ctx_id = id;
  g_slot[dev].addr = p;
  *addr = p;
  return VCOLL_OK;
}

}  // namespace

extern "C" int vcoll_sparse_allreduce_noalloc(const void* const* in, void* const* out,
                                              void* const* accum, int W, int64_t n,
                                              float threshold, int topk, int64_t* nnz,
                                              void* stream) {
  if (!topk)  // the threshold mode needs no working memory at all
    return vcoll_sparse_allreduce(in, out, accum, W, n, threshold, topk, nnz, nullptr, 0, stream);
  // the minimum working memory; what the array holds beyond it becomes
  // candidate-list room (a list that does not fit sends the select passes
  // over the whole array instead)
  const size_t need =
      (W >= 1 && W <= VCOLL_MAX_RANKS && n >= 0) ? vcoll::topk_workspace_min_bytes(W, n) : 0;
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "top-K over W=%d ranks of n=%lld elements needs %zu bytes of working memory; the "
             "fixed scratch holds %zu (use vcoll_sparse_allreduce with your own workspace)",
             W, (long long)n, need, kNoAllocScratchBytes);
    return vcoll::report_error(VCOLL_ERR_INVALID_ARG, msg);
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  // vcoll_sparse_allreduce clears the histograms at the start of every call;
  // the rest of the working memory is written before it is read
  return vcoll_sparse_allreduce(in, out, accum, W, n, threshold, topk, nnz, scratch,
                                kNoAllocScratchBytes, stream);
}

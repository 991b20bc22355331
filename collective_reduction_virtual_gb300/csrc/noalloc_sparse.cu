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

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address per device, set up once

// Looks up the array's device address on the current device (once per
// device, with that device current).
int scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return vcoll::report_error(VCOLL_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return vcoll::report_error(VCOLL_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the fixed scratch failed: %s",
               cudaGetErrorString(e));
      return vcoll::report_error(VCOLL_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
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

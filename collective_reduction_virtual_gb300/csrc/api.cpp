// Host side of the C ABI declared in include/vcoll.h: argument validation,
// segment / alignment / aliasing analysis, kernel selection and launch.
//
// Error conventions follow the early NCCL page (ncclReduceScatter: an unknown
// datatype is ncclInvalidType, an unknown op ncclInvalidOperation, an empty
// message succeeds without work, a single GPU is a plain device copy) and
// Horovod's Status-with-message reporting (operations.cc): every failure
// returns a code and leaves a thread-local message.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "vcoll_internal.h"

using namespace vcoll;

namespace {

thread_local char g_err[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(VCOLL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int elem_size(int dtype) {
  if (dtype == VCOLL_F32) return 4;
  if (dtype == VCOLL_BF16) return 2;
  return 0;
}

// ------------------------------------------------------------ device info

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];  // 0 = not queried yet

struct OccEntry {
  int dev;
  const void* fn;
  int threads;
  size_t smem;
  int blocks;
};
std::vector<OccEntry> g_occ;

int current_device(int* dev, int* sms) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return fail(VCOLL_ERR_UNSUPPORTED, "device %d", *dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[*dev] == 0) {
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, *dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_sms[*dev] = v;
  }
  *sms = g_sms[*dev];
  return VCOLL_OK;
}

// Lets fn take `bytes` of dynamic shared memory on the current device (once
// per device and kernel).
int allow_dynamic_smem(const void* fn, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static std::vector<std::pair<int, const void*>> done;
  std::lock_guard<std::mutex> lk(g_mu);
  for (const auto& d : done)
    if (d.first == dev && d.second == fn) return VCOLL_OK;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  done.push_back({dev, fn});
  return VCOLL_OK;
}

int resident_blocks(int dev, const void* fn, int threads, size_t smem, int* blocks) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (const OccEntry& o : g_occ)
    if (o.dev == dev && o.fn == fn && o.threads == threads && o.smem == smem) {
      *blocks = o.blocks;
      return VCOLL_OK;
    }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  }
  int b = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (b < 1) b = 1;
  g_occ.push_back({dev, fn, threads, smem, b});
  *blocks = b;
  return VCOLL_OK;
}

// ------------------------------------------------------- buffer analysis

void segment_of(int64_t n, int W, int j, int64_t* off, int64_t* len) {
  const int64_t q = n / W, r = n % W;
  *off = (int64_t)j * q + (j < r ? j : r);
  *len = q + (j < r ? 1 : 0);
}

// One buffer of a call: bytes [addr, addr + nbytes) hold the elements
// [lo, lo + nbytes / es) of the index space, so element i sits at
// base + i * es with base = addr - lo * es (mod 2^64).
struct Buf {
  uint64_t addr;
  uint64_t nbytes;
  uint64_t base;
  bool out;
};

// Outputs must not overlap each other; an input may overlap an output only
// when both map every element index to the same address (then the thread
// that owns the index reads it before writing it).  Returns VCOLL_OK or
// INVALID_ARG.  *vec / *phase: whether all buffers share one 16-byte phase.
int check_aliasing(const std::vector<Buf>& bufs) {
  // sorted by start address, each buffer only meets the ones that start
  // before it ends
  std::vector<const Buf*> v;
  v.reserve(bufs.size());
  for (const Buf& b : bufs)
    if (b.nbytes) v.push_back(&b);
  std::sort(v.begin(), v.end(), [](const Buf* a, const Buf* b) { return a->addr < b->addr; });
  for (size_t i = 0; i < v.size(); ++i) {
    const uint64_t end = v[i]->addr + v[i]->nbytes;
    for (size_t k = i + 1; k < v.size() && v[k]->addr < end; ++k) {
      const Buf& a = *v[i];
      const Buf& b = *v[k];
      if (a.out && b.out) return fail(VCOLL_ERR_INVALID_ARG, "two output buffers overlap");
      if (a.out != b.out && a.base != b.base)
        return fail(VCOLL_ERR_INVALID_ARG,
                    "an input overlaps an output at a different element offset "
                    "(only exact in-place aliasing is allowed)");
    }
  }
  return VCOLL_OK;
}

int analyse(const std::vector<Buf>& bufs, int es, int* vec, int* phase) {
  int rc = check_aliasing(bufs);
  if (rc) return rc;
  uint64_t ph = bufs.empty() ? 0 : (bufs[0].base & 15);
  int same = 1;
  for (const Buf& b : bufs)
    if ((b.base & 15) != ph) same = 0;
  *vec = same;
  *phase = same ? (int)(ph / es) : 0;
  return VCOLL_OK;
}

// No two of the given byte ranges may overlap (sort + sweep).
int check_disjoint(std::vector<Buf> bufs) {
  std::sort(bufs.begin(), bufs.end(), [](const Buf& a, const Buf& b) { return a.addr < b.addr; });
  uint64_t end = 0;
  bool any = false;
  for (const Buf& b : bufs) {
    if (!b.nbytes) continue;
    if (any && b.addr < end) return fail(VCOLL_ERR_INVALID_ARG, "two buffers overlap");
    end = std::max(end, b.addr + b.nbytes);
    any = true;
  }
  return VCOLL_OK;
}

int check_ptrs(const void* const* p, int W, const char* what, int es, const int64_t* lens) {
  if (!p) return fail(VCOLL_ERR_INVALID_ARG, "%s array is NULL", what);
  for (int u = 0; u < W; ++u) {
    if (lens[u] == 0) continue;
    if (!p[u]) return fail(VCOLL_ERR_INVALID_ARG, "%s[%d] is NULL", what, u);
    if ((uint64_t)p[u] % es)
      return fail(VCOLL_ERR_INVALID_ARG, "%s[%d] is not aligned to the element size", what, u);
  }
  return VCOLL_OK;
}

int check_common(int W, int64_t n, int dtype, int op) {
  if (W < 1 || W > VCOLL_MAX_RANKS)
    return fail(VCOLL_ERR_INVALID_ARG, "W = %d outside [1, %d]", W, VCOLL_MAX_RANKS);
  if (n < 0) return fail(VCOLL_ERR_INVALID_ARG, "n = %lld < 0", (long long)n);
  if (!elem_size(dtype)) return fail(VCOLL_ERR_INVALID_TYPE, "unknown dtype %d", dtype);
  if (op != VCOLL_SUM && op != VCOLL_MAX && op != VCOLL_AVG && op != VCOLL_MIN &&
      op != VCOLL_PROD)
    return fail(VCOLL_ERR_INVALID_OP, "unknown op %d", op);
  return VCOLL_OK;
}

constexpr int64_t kSmallBytes = 32 * 1024;  // latency-bound path (MLX PR #3901: <= 32 KB)

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tile size (elements) for a one-CTA-per-tile launch over nseg segments of
// about n / nseg elements: the kernel's full tile (threads x unroll x V) for
// large messages, smaller tiles -- down to one vector per thread -- while
// that gives fewer than about two CTAs per SM, so that mid-size messages
// spread over the GPU instead of a handful of CTAs (measured on GB300: a
// target of four per SM made 2-8 MiB messages slower, one per SM left
// 64 KiB-1 MiB messages about 1 us slower).  The kernels bound every
// tile by its own end, so any multiple of threads x V works.
int64_t adaptive_tile(int64_t n, int nseg, int threads, int V, int unroll) {
  const int64_t unit = (int64_t)threads * V;
  const int64_t full = unit * unroll;
  int dev = 0, sms = 0;
  if (current_device(&dev, &sms) != VCOLL_OK || sms <= 0) {
    g_err[0] = 0;  // not fatal here: the launch reports device errors
    return full;
  }
  const int64_t want = std::max<int64_t>(1, ceil_div(2LL * sms, nseg));  // tiles per segment
  const int64_t per = ceil_div(ceil_div(n, nseg), want);
  return std::min(full, std::max(unit, ceil_div(per, unit) * unit));
}

// Tiles per segment: enough for the longest aligned body, at least one (tile
// 0 also does the unaligned head and tail).
int64_t tiles_per_segment(int64_t n, int W, int nseg, int V, int phase, int64_t tile_elems) {
  int64_t tps = 1;
  for (int j = 0; j < nseg; ++j) {
    int64_t a, len;
    if (nseg == 1) {
      a = 0;
      len = n;
    } else {
      segment_of(n, W, j, &a, &len);
    }
    const int64_t b = a + len;
    int64_t up = a + ((V - ((a + phase) % V)) % V);
    const int64_t av = std::min(up, b);
    const int64_t dn = b - ((b + phase) % V);
    const int64_t bv = std::max(dn, av);
    tps = std::max(tps, ceil_div(bv - av, tile_elems));
  }
  return tps;
}

// persistent: as many CTAs as fit on the GPU at once, each looping over
// tiles (the pipelined kernels need it to keep their stages full); otherwise
// one CTA per tile.  Measured on the W=8 fp32 allreduce: one CTA per tile
// reaches 7.0 TB/s where the persistent grid-stride loop reaches 6.35 TB/s --
// the hardware scheduler keeps the CTAs in flight on a compact window of
// addresses, while persistent CTAs drift apart over the buffers.
// cudaLaunchKernel with programmatic stream serialization: the kernel's
// blocks may be scheduled while the previous kernel in the stream finishes;
// each waits (griddepcontrol, pdl_enter) for it to complete before touching
// memory, so only launch latency is hidden, never an ordering
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, size_t smem,
                       cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

int launch(const void* fn, int64_t num_tiles, int threads, size_t smem, bool persistent,
           void* params, void* stream) {
  int64_t grid = num_tiles;
  if (persistent) {
    int dev = 0, sms = 0, blocks = 0;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    rc = resident_blocks(dev, fn, threads, smem, &blocks);
    if (rc) return rc;
    grid = std::min<int64_t>(num_tiles, (int64_t)sms * blocks);
  }
  grid = std::max<int64_t>(1, std::min<int64_t>(grid, 0x7FFFFFFF));
  void* args[] = {params};
  cudaError_t e = launch_pdl(fn, dim3((unsigned)grid), dim3(threads), args, smem,
                             (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return VCOLL_OK;
}

int copy_d2d(void* dst, const void* src, int64_t bytes, void* stream) {
  if (dst == src || bytes == 0) return VCOLL_OK;
  cudaError_t e = cudaMemcpyAsync(dst, src, (size_t)bytes, cudaMemcpyDeviceToDevice,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  return VCOLL_OK;
}

// Launch sequence of the sparsified allreduce (shared by the entry points
// that differ only in where the top-K workspace lives; workspace_bytes is at
// least topk_workspace_min_bytes).
int sparse_launch(SparseParams& prm, int topk, void* workspace, size_t workspace_bytes,
                  void* stream) {
  int dev = 0, sms = 0;
  int rc = current_device(&dev, &sms);
  if (rc) return rc;
  const int W = prm.W;
  cudaStream_t st = (cudaStream_t)stream;
  if (topk) {
    const TopkLayout L = topk_layout(W, prm.n);
    char* ws = (char*)workspace;
    prm.hist = (uint32_t*)ws;
    prm.state = (TopkState*)(ws + L.state);
    prm.cand_n = (unsigned long long*)(ws + L.cand_n);
    prm.tilecnt = (uint32_t*)(ws + L.tilecnt);
    // candidate lists in what is left (a multiple of 4 entries per rank keeps
    // the index list 16-byte aligned)
    const size_t lists = L.cands + L.chunk_bytes;
    const size_t spare = workspace_bytes > lists ? workspace_bytes - lists : 0;
    int64_t cap = (int64_t)(spare / ((size_t)W * 8));
    cap = std::min<int64_t>(cap, topk_cand_cap_default(prm.n)) & ~(int64_t)3;
    prm.cand_cap = cap;
    prm.chunk = (uint32_t*)(ws + L.cands);
    prm.cand_key = (uint32_t*)(ws + lists);
    prm.cand_idx = prm.cand_key + (size_t)W * (size_t)cap;
    // worth it when the list can hold what the sample typically admits:
    // 2K-4K entries above a wide lower bound for K < n/4, else a two-sided
    // band (the K-th key's bin and a few percent of n around it)
    const bool wide = 4 * prm.K < prm.n && cap >= 3 * prm.K;
    prm.band = wide ? 0 : 1;
    prm.use_cand = prm.K > 0 && prm.K < prm.n && (wide || 10 * cap >= prm.n);
    // with a wide lower bound the lists hold every kept entry (unless a rank
    // falls back), so the result can be built from them
    prm.list_out = prm.use_cand && !prm.band;
  }
  if (topk && prm.K > 0) {
    // histograms, states and candidate counts start at zero
    cudaError_t e = cudaMemsetAsync(workspace, 0, topk_layout(W, prm.n).tilecnt, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    // data passes: one CTA per tile (per sampled tile for the sample); passes
    // that usually find nothing to do for their rank (the whole-array ones
    // beside the candidate path) and the candidate passes: a few CTAs per SM
    const int64_t gx = std::max<int64_t>(
        1, std::min<int64_t>(prm.tiles_per_rank, ceil_div((int64_t)sms * 4, W)));
    const unsigned tiles = (unsigned)std::min<int64_t>(prm.tiles_per_rank, 0x7FFFFFFF);
    void* args[] = {&prm};
    const dim3 few((unsigned)gx, (unsigned)W), sgrid((unsigned)W);
    // the sample: every 16th tile, up to every 128th for large arrays (at
    // least 128 tiles, half a million entries, per rank; every 128th rather
    // than every 64th took 10 us off a call at W = 8, 2^26 per rank)
    prm.sample_stride = (int)std::min<int64_t>(128, std::max<int64_t>(16, prm.tiles_per_rank / 128));
    const dim3 every(tiles, (unsigned)W),
        sample((unsigned)ceil_div(tiles, prm.sample_stride), (unsigned)W);
    const dim3 full_grid = prm.use_cand ? few : every;
    auto run = [&](const void* k, dim3 grid, unsigned threads) -> int {
      cudaError_t e2 = launch_pdl(k, grid, dim3(threads), args, 0, st);
      return e2 == cudaSuccess ? VCOLL_OK : cuda_fail(e2, "top-K pass launch");
    };
    // sample pass and lower bound
    if ((rc = run(topk_sample_kernel(), sample, 256)) || (rc = run(topk_select_low_kernel(), sgrid, 1024)))
      return rc;
    // on the candidate path: the second digit over the same sample narrows
    // the settled bound (list route with accumulations: the candidate pass
    // writes those residuals), the lower bound and the band's upper bound to
    // 22-bit prefixes
    if (prm.use_cand &&
        ((rc = run(topk_sample2_kernel(), sample, 256)) ||
         (rc = run(topk_select_refine_kernel(), sgrid, 1024))))
      return rc;
    if (prm.use_cand) {
      // one pass collects the candidates, the first digit from the lists
      // (a CTA loops over two tiles with accumulations, four without: its
      // setup is paid once for them; measured at W = 8, 2^26 per rank)
      const dim3 fgrid((unsigned)ceil_div((int64_t)tiles, prm.has_acc ? 2 : 4), (unsigned)W);
      if ((rc = run(topk_filter_kernel(prm.has_acc, prm.band), fgrid, 256))) return rc;
      // the candidate pass stored x = in + acc in acc: later passes read acc
      prm.x_in_acc = prm.has_acc;
      if ((rc = run(topk_cand_hist_kernel(0), few, 256)) ||
          (rc = run(topk_select_kernel(0), sgrid, 1024)))
        return rc;
      // off the list route (decided by that selection), x comes back where
      // the candidate pass stored settled residuals
      if (prm.list_out && prm.has_acc && (rc = run(topk_restore_kernel(), few, 256))) return rc;
    } else {
      // the first digit from the bound up
      if ((rc = run(topk_hist_kernel(0), every, 256)) ||
          (rc = run(topk_select_kernel(0), sgrid, 1024)))
        return rc;
    }
    // ranks whose bound failed (or whose list did) redo it over all bins
    if ((rc = run(topk_redo_hist_kernel(), full_grid, 256)) ||
        (rc = run(topk_redo_select_kernel(), sgrid, 1024)))
      return rc;
    // second and third digits: the whole array for ranks on the full path,
    // the lists for the others
    for (int pass = 1; pass <= 2; ++pass) {
      if ((rc = run(topk_hist_kernel(pass), full_grid, 256))) return rc;
      if (prm.use_cand && (rc = run(topk_cand_hist_kernel(pass), few, 256))) return rc;
      if ((rc = run(topk_select_kernel(pass), sgrid, 1024))) return rc;
    }
    // keys equal to the K-th one straddling the cut: tile counts and a scan
    // on the full path, three index digits on the candidate path
    if ((rc = run(topk_tie_count_kernel(), full_grid, 256)) ||
        (rc = run(topk_tie_find_kernel(), sgrid, 1024)))
      return rc;
    // on the candidate path one pass collects the equal keys' indices and
    // picks the boundary (the last CTA of each rank); ranks with more equal
    // keys than it holds take three index-digit passes
    if (prm.use_cand) {
      if ((rc = run(topk_ties_kernel(), few, 256))) return rc;
      for (int pass = 3; pass <= 5; ++pass)
        if ((rc = run(topk_cand_hist_kernel(pass), few, 256)) ||
            (rc = run(topk_index_select_kernel(pass), sgrid, 1024)))
          return rc;
    }
  }
  const void* fn = sparse_apply_kernel(topk);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(prm.num_tiles, 0x7FFFFFFF));
  // on the list route the dense pass works only for a call where a rank fell
  // back (it returns at once otherwise): a few CTAs per SM, looping over the
  // tiles, keep its launch cheap (one CTA per tile cost 19 us to return)
  const int64_t agrid = prm.list_out ? std::min<int64_t>(grid, (int64_t)sms * 8) : grid;
  void* args[] = {&prm};
  cudaError_t e = launch_pdl(fn, dim3((unsigned)agrid), dim3(256), args, 0, st);
  if (e != cudaSuccess) return cuda_fail(e, "sparse apply launch");
  if (topk && prm.list_out) {  // the result from the lists (decided on the device)
    e = launch_pdl(topk_list_out_kernel(), dim3((unsigned)grid), dim3(256), args, 0, st);
    if (e != cudaSuccess) return cuda_fail(e, "top-K output launch");
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse allreduce");
  return VCOLL_OK;
}

// The TMA bulk copies of the staged forms run only on device memory: when a
// buffer is elsewhere (pinned host memory, managed memory) a staged request
// runs the direct kernels, which give the same bits.
bool all_device_memory(const void* const* p, int W) {
  for (int u = 0; u < W; ++u) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p[u]) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    if (a.type != cudaMemoryTypeDevice) return false;
  }
  return true;
}

// wire >= 0: the reduced-precision allreduce (fp32 buffers, arithmetic rounded
// to the 16-bit wire type every hop); -1: the plain collectives.
int reduce_common(int kind, const void* const* in, void* const* out, int W, int64_t n, int dtype,
                  int op, unsigned flags, void* stream, int wire = -1,
                  const int* user_from_ring = nullptr) {
  g_err[0] = 0;
  int rc = check_common(W, n, dtype, op);
  if (rc) return rc;
  if ((flags & VCOLL_FLAG_STAGED) && (flags & VCOLL_FLAG_DIRECT))
    return fail(VCOLL_ERR_INVALID_ARG, "VCOLL_FLAG_STAGED and VCOLL_FLAG_DIRECT both set");
  if (flags & ~(VCOLL_FLAG_RING_ORDER | VCOLL_FLAG_STAGED | VCOLL_FLAG_DIRECT))
    return fail(VCOLL_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  const int es = elem_size(dtype);
  int64_t in_len[VCOLL_MAX_RANKS], out_len[VCOLL_MAX_RANKS], seg_off[VCOLL_MAX_RANKS];
  for (int u = 0; u < W; ++u) {
    segment_of(n, W, u, &seg_off[u], &out_len[u]);
    in_len[u] = n;
    if (kind == KIND_AR) out_len[u] = n;
  }
  if ((rc = check_ptrs(in, W, "in", es, in_len))) return rc;
  if ((rc = check_ptrs((const void* const*)out, W, "out", es, out_len))) return rc;
  if (n == 0) return VCOLL_OK;
  if ((flags & VCOLL_FLAG_STAGED) &&
      !(all_device_memory(in, W) && all_device_memory((const void* const*)out, W)))
    flags &= ~VCOLL_FLAG_STAGED;

  std::vector<Buf> bufs;
  for (int u = 0; u < W; ++u) {
    bufs.push_back({(uint64_t)in[u], (uint64_t)(n * es), (uint64_t)in[u], false});
    const uint64_t lo = kind == KIND_AR ? 0 : (uint64_t)seg_off[u];
    bufs.push_back({(uint64_t)out[u], (uint64_t)(out_len[u] * es),
                    (uint64_t)out[u] - lo * (uint64_t)es, true});
  }
  int vec, phase;
  if ((rc = analyse(bufs, es, &vec, &phase))) return rc;

  // ring order: the kernels fold segment j from input ring_start[j] on.  The
  // identity ring starts at rank j + 1; a user ring (NCCL's userFromRing:
  // user_from_ring[p] is the rank at ring position p) reorders the inputs by
  // ring position and starts segment j at the position after rank j's, so
  // the fold runs around the ring and ends at rank j
  const void* ring_in[VCOLL_MAX_RANKS];
  uint8_t ring_start[VCOLL_MAX_RANKS];
  for (int j = 0; j < W; ++j) {
    ring_in[j] = in[j];
    ring_start[j] = (uint8_t)((j + 1) % W);
  }
  if (user_from_ring) {
    int pos[VCOLL_MAX_RANKS];
    for (int u = 0; u < W; ++u) pos[u] = -1;
    for (int q = 0; q < W; ++q) {
      const int u = user_from_ring[q];
      if (u < 0 || u >= W || pos[u] >= 0)
        return fail(VCOLL_ERR_INVALID_ARG, "user_from_ring is not a permutation of 0..%d", W - 1);
      pos[u] = q;
    }
    for (int q = 0; q < W; ++q) ring_in[q] = in[user_from_ring[q]];
    for (int j = 0; j < W; ++j) ring_start[j] = (uint8_t)((pos[j] + 1) % W);
    in = ring_in;
  }

  if (wire >= 0) {
    // every rank count, W = 1 included, goes through the kernel: even a single
    // rank's values are rounded to the wire type and back
    const bool ring = (flags & VCOLL_FLAG_RING_ORDER) && W > 2;
    const int W_t = (W == 2 || W == 4 || W == 8 || W == 16) ? W : 0;
    ReduceParams prm;
    memset(&prm, 0, sizeof(prm));
    for (int u = 0; u < W; ++u) {
      prm.in[u] = in[u];
      prm.out[u] = out[u];
    }
    prm.n = n;
    prm.q = n / W;
    prm.r = n % W;
    prm.W = W;
    prm.nseg = ring ? W : 1;
    prm.phase = vec ? phase : -1;
    prm.ring = ring ? 1 : 0;
    memcpy(prm.ring_start, ring_start, sizeof(prm.ring_start));
    prm.scale = op == VCOLL_AVG ? 1.0f / (float)W : 1.0f;
    prm.do_scale = op == VCOLL_AVG ? 1 : 0;
    const bool small = n * es <= kSmallBytes;
    const int threads = small ? 128 : 256;
    prm.tile_elems = vec ? adaptive_tile(n, prm.nseg, threads, 4, 2) : (int64_t)threads * 4;
    prm.tiles_per_seg = vec ? tiles_per_segment(n, W, prm.nseg, 4, phase, prm.tile_elems)
                            : tiles_per_segment(n, W, prm.nseg, 1, 0, prm.tile_elems);
    prm.num_tiles = prm.tiles_per_seg * prm.nseg;
    return launch(wire_kernel(wire, W_t, ring ? 1 : 0), prm.num_tiles, threads, 0, false, &prm,
                  stream);
  }

  if (W == 1) return copy_d2d(out[0], in[0], n * es, stream);

  const bool ring = (flags & VCOLL_FLAG_RING_ORDER) && op != VCOLL_MAX && op != VCOLL_MIN && W > 2;
  const int W_t = (W == 2 || W == 4 || W == 8 || W == 16) ? W : 0;
  const int nseg = (kind == KIND_RS || ring) ? W : 1;
  const bool small = n * es <= kSmallBytes;
  const int threads = small ? 128 : 256;
  // inputs at other phases than the outputs: realigned vectors on the
  // outputs' grid -- the allreduce's outputs must share a phase; each
  // reduce-scatter segment follows its own output (uneven segments included)
  bool realign = false;
  if (!vec) {
    realign = true;
    if (kind == KIND_AR)
      for (int u = 1; u < W; ++u)
        if (((uint64_t)out[u] & 15) != ((uint64_t)out[0] & 15)) realign = false;
    if (realign && kind == KIND_AR) phase = (int)(((uint64_t)out[0] & 15) / es);
  }
  // aligned buffers with W in 3..7: the realigning kernel (all shifts zero)
  // is compiled for those W, the plain vector kernels only for 2, 4, 8, 16
  if (vec && W >= 3 && W <= 7 && W != 4 && !(flags & VCOLL_FLAG_STAGED)) realign = true;
  const bool vec_like = vec || realign;
  const int V = vec_like ? 16 / es : 1;

  // The staged (TMA bulk copy) variant needs the 16-byte vector layout and a
  // compile-time W; everything else runs the direct kernels (same bits).
  const bool staged = (flags & VCOLL_FLAG_STAGED) && vec && W_t != 0 && !small;
  const void* fn;
  if (staged)
    fn = dtype == VCOLL_F32 ? staged_kernel_f32(op, kind, W_t, ring)
                            : staged_kernel_bf16(op, kind, W_t, ring);
  else if (realign)  // compiled in for every W up to 8
    fn = dtype == VCOLL_F32 ? reduce_kernel_f32_realign(op, kind, W, ring)
                            : reduce_kernel_bf16_realign(op, kind, W, ring);
  else
    fn = dtype == VCOLL_F32 ? reduce_kernel_f32(op, kind, W_t, ring, vec)
                            : reduce_kernel_bf16(op, kind, W_t, ring, vec);
  ReduceParams prm;
  memset(&prm, 0, sizeof(prm));
  for (int u = 0; u < W; ++u) {
    prm.in[u] = in[u];
    prm.out[u] = out[u];
  }
  prm.n = n;
  prm.q = n / W;
  prm.r = n % W;
  prm.W = W;
  prm.nseg = nseg;
  prm.phase = phase;
  prm.ring = ring ? 1 : 0;
  memcpy(prm.ring_start, ring_start, sizeof(prm.ring_start));
  prm.scale = op == VCOLL_AVG ? 1.0f / (float)W : 1.0f;
  prm.do_scale = op == VCOLL_AVG ? 1 : 0;
  if (realign)
    for (int u = 0; u < W; ++u) {
      prm.in_phase[u] = (uint8_t)((uint64_t)in[u] & 15);
      const uint64_t ob = kind == KIND_AR ? (uint64_t)out[0]
                                          : (uint64_t)out[u] - (uint64_t)seg_off[u] * es;
      prm.out_phase[u] = (uint8_t)(ob & 15);
    }
  if (realign && W <= 8)  // the compiled-W kernels read the shifts from a table
    for (int j = 0; j < W; ++j)
      for (int u = 0; u < W; ++u)
        prm.wshift[j * 8 + u] = (uint8_t)((prm.in_phase[u] - prm.out_phase[j]) & 15);
  if (staged)
    prm.tile_elems = staged_slice_bytes(W_t) / es;
  else if (realign)  // two vectors per thread (the compile-time-W kernel loops over any tile)
    prm.tile_elems = adaptive_tile(n, nseg, threads, V, 2);
  else
    prm.tile_elems = vec ? adaptive_tile(n, nseg, threads, V, unroll_for(W_t)) : (int64_t)threads * 4;
  prm.tiles_per_seg = tiles_per_segment(n, W, nseg, V, phase, prm.tile_elems);
  if (realign && kind == KIND_RS)  // segments on grids of their own phases
    for (int ph = 0; ph < V; ++ph)
      prm.tiles_per_seg =
          std::max(prm.tiles_per_seg, tiles_per_segment(n, W, nseg, V, ph, prm.tile_elems));
  prm.num_tiles = prm.tiles_per_seg * nseg;
  if (staged)
    return launch(fn, prm.num_tiles, kStagedThreads, (size_t)staged_smem_bytes(W_t), true, &prm,
                  stream);
  return launch(fn, prm.num_tiles, threads, 0, false, &prm, stream);
}

}  // namespace

// ======================================================================
extern "C" {

int vcoll_reduce_scatter(const void* const* in, void* const* out, int W, int64_t n, int dtype,
                         int op, unsigned flags, void* stream) {
  return reduce_common(KIND_RS, in, out, W, n, dtype, op, flags, stream);
}

int vcoll_allreduce(const void* const* in, void* const* out, int W, int64_t n, int dtype, int op,
                    unsigned flags, void* stream) {
  return reduce_common(KIND_AR, in, out, W, n, dtype, op, flags, stream);
}

int vcoll_reduce_scatter_ring(const void* const* in, void* const* out, int W, int64_t n,
                              int dtype, int op, const int* user_from_ring, void* stream) {
  return reduce_common(KIND_RS, in, out, W, n, dtype, op, VCOLL_FLAG_RING_ORDER, stream, -1,
                       user_from_ring);
}

int vcoll_allreduce_ring(const void* const* in, void* const* out, int W, int64_t n, int dtype,
                         int op, const int* user_from_ring, void* stream) {
  return reduce_common(KIND_AR, in, out, W, n, dtype, op, VCOLL_FLAG_RING_ORDER, stream, -1,
                       user_from_ring);
}

int vcoll_allreduce_wire(const void* const* in, void* const* out, int W, int64_t n, int wire, int op,
                         unsigned flags, void* stream) {
  g_err[0] = 0;
  if (wire != VCOLL_F16 && wire != VCOLL_BF16)
    return fail(VCOLL_ERR_INVALID_TYPE, "wire type %d is neither VCOLL_F16 nor VCOLL_BF16", wire);
  if (op != VCOLL_SUM && op != VCOLL_AVG) {
    if (op == VCOLL_MAX || op == VCOLL_MIN || op == VCOLL_PROD)
      return fail(VCOLL_ERR_UNSUPPORTED, "the wire allreduce supports sum and avg");
    return fail(VCOLL_ERR_INVALID_OP, "unknown op %d", op);
  }
  if (flags & (VCOLL_FLAG_STAGED | VCOLL_FLAG_DIRECT)) flags &= VCOLL_FLAG_RING_ORDER;
  return reduce_common(KIND_AR, in, out, W, n, VCOLL_F32, op, flags, stream, wire);
}

// Allgather of W pieces, piece j landing at [disp[j], disp[j+1]) of every
// output (shared by allgather and allgatherv).
static int gather_common(const void* const* in, void* const* out, int W, const int64_t* disp,
                         int dtype, unsigned flags, void* stream) {
  const int es = elem_size(dtype);
  const int64_t n = disp[W];
  int64_t in_len[VCOLL_MAX_RANKS], out_len[VCOLL_MAX_RANKS];
  for (int u = 0; u < W; ++u) {
    in_len[u] = disp[u + 1] - disp[u];
    out_len[u] = n;
  }
  int rc;
  if ((rc = check_ptrs(in, W, "in", es, in_len))) return rc;
  if ((rc = check_ptrs((const void* const*)out, W, "out", es, out_len))) return rc;
  if (n == 0) return VCOLL_OK;
  std::vector<Buf> bufs;
  for (int u = 0; u < W; ++u) {
    if (in_len[u])
      bufs.push_back({(uint64_t)in[u], (uint64_t)(in_len[u] * es),
                      (uint64_t)in[u] - (uint64_t)disp[u] * es, false});
    bufs.push_back({(uint64_t)out[u], (uint64_t)(n * es), (uint64_t)out[u], true});
  }
  int vec, phase;
  if ((rc = analyse(bufs, es, &vec, &phase))) return rc;
  if (W == 1) return copy_d2d(out[0], in[0], n * es, stream);

  const bool small = n * es <= kSmallBytes;
  const int threads = small ? 128 : 256;
  // pieces at other phases than the outputs, which share one: the vector
  // kernel realigns them
  bool realign = false;
  if (!vec) {
    realign = true;
    for (int u = 1; u < W; ++u)
      if (((uint64_t)out[u] & 15) != ((uint64_t)out[0] & 15)) realign = false;
    if (realign) phase = (int)(((uint64_t)out[0] & 15) / es);
  }
  const int V = (vec || realign) ? 16 / es : 1;
  GatherParams prm;
  memset(&prm, 0, sizeof(prm));
  for (int u = 0; u < W; ++u) {
    prm.in[u] = in[u];
    prm.out[u] = out[u];
    if (realign)
      prm.ishift[u] = (uint8_t)(((uint64_t)in[u] - (uint64_t)disp[u] * es - (uint64_t)out[0]) & 15);
  }
  for (int u = 0; u <= W; ++u) prm.disp[u] = disp[u];
  prm.W = W;
  prm.phase = phase;
  prm.tile_elems = adaptive_tile(n, W, threads, V, 4);
  auto gather_tiles = [&](int64_t tile) {  // tiles per segment
    int64_t t = 1;
    for (int j = 0; j < W; ++j) {
      const int64_t a = disp[j], b = disp[j + 1];
      const int64_t up = a + ((V - ((a + phase) % V)) % V);
      const int64_t av = std::min(up, b);
      const int64_t bv = std::max(b - ((b + phase) % V), av);
      t = std::max(t, ceil_div(bv - av, tile));
    }
    return t;
  };
  int64_t tps = gather_tiles(prm.tile_elems);
  // Launches of about 512 CTAs ran 25-30 % slower than half or twice as
  // many at every W measured on GB300 (2-16; 2-8 MiB per rank, L2-resident
  // or not): such a launch takes tiles half the size instead
  const int64_t unit = (int64_t)threads * V;
  if (tps * W >= 400 && tps * W <= 640 && prm.tile_elems >= 2 * unit) {
    prm.tile_elems = ceil_div(prm.tile_elems / 2, unit) * unit;
    tps = gather_tiles(prm.tile_elems);
  }
  prm.tiles_per_seg = tps;
  prm.num_tiles = tps * W;
  // TMA variant only when asked for: with one CTA per tile the direct kernel
  // is ahead at every W measured (2-16)
  const bool tma = (flags & VCOLL_FLAG_STAGED) != 0 && all_device_memory(in, W) &&
                   all_device_memory((const void* const*)out, W);
  if (tma && vec && !small) {
    // TMA variant: bulk loads into shared memory, W bulk stores per tile
    prm.tile_elems = kGatherTmaTileBytes / es;
    tps = 1;
    for (int j = 0; j < W; ++j) {
      const int64_t a = disp[j], b = disp[j + 1];
      const int64_t up = a + ((V - ((a + phase) % V)) % V);
      const int64_t av = std::min(up, b);
      const int64_t bv = std::max(b - ((b + phase) % V), av);
      tps = std::max(tps, ceil_div(bv - av, prm.tile_elems));
    }
    prm.tiles_per_seg = tps;
    prm.num_tiles = tps * W;
    return launch(gather_tma_kernel(es), prm.num_tiles, kGatherTmaThreads,
                  (size_t)kGatherTmaStages * kGatherTmaTileBytes + 64, true, &prm, stream);
  }
  // The realigned variant reads each shifted vector as two aligned blocks,
  // the second usually still in L1 from the neighbouring lane's first; with
  // fewer CTAs per SM more of them stay there.  Shared memory the kernel does
  // not use holds it to two CTAs per SM: 11 % faster than the register-bound
  // five (W = 8, n = 2^26 + 2: 5836 -> 6500 GB/s).
  size_t smem = 0;
  if (realign && !small) {
    smem = kGatherRealignSmem;
    if ((rc = allow_dynamic_smem(gather_kernel(es, 2), smem))) return rc;
  }
  return launch(gather_kernel(es, vec ? 1 : realign ? 2 : 0), prm.num_tiles, threads, smem,
                false, &prm, stream);
}

int vcoll_allgather(const void* const* in, void* const* out, int W, int64_t n, int dtype, int op,
                    unsigned flags, void* stream) {
  g_err[0] = 0;
  int rc = check_common(W, n, dtype, op);
  if (rc) return rc;
  if (flags & ~(VCOLL_FLAG_RING_ORDER | VCOLL_FLAG_STAGED | VCOLL_FLAG_DIRECT))
    return fail(VCOLL_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  int64_t disp[VCOLL_MAX_RANKS + 1];
  for (int u = 0; u < W; ++u) {
    int64_t len;
    segment_of(n, W, u, &disp[u], &len);
  }
  disp[W] = n;
  return gather_common(in, out, W, disp, dtype, flags, stream);
}

int vcoll_allgatherv(const void* const* in, const int64_t* counts, void* const* out, int W,
                     int dtype, void* stream) {
  g_err[0] = 0;
  int rc = check_common(W, 0, dtype, VCOLL_SUM);
  if (rc) return rc;
  if (!counts) return fail(VCOLL_ERR_INVALID_ARG, "counts is NULL");
  int64_t disp[VCOLL_MAX_RANKS + 1];
  disp[0] = 0;
  for (int u = 0; u < W; ++u) {
    if (counts[u] < 0) return fail(VCOLL_ERR_INVALID_ARG, "counts[%d] < 0", u);
    disp[u + 1] = disp[u] + counts[u];
  }
  return gather_common(in, out, W, disp, dtype, 0, stream);
}

int vcoll_fuse_plan(const int64_t* counts, int T, int dtype, int64_t threshold_bytes,
                    int* batch_begin, int* nbatches) {
  g_err[0] = 0;
  const int es = elem_size(dtype);
  if (!es) return fail(VCOLL_ERR_INVALID_TYPE, "unknown dtype %d", dtype);
  if (T < 0 || (T > 0 && !counts) || !batch_begin || !nbatches || threshold_bytes < 0)
    return fail(VCOLL_ERR_INVALID_ARG, "invalid fuse_plan arguments");
  for (int t = 0; t < T; ++t)
    if (counts[t] < 0) return fail(VCOLL_ERR_INVALID_ARG, "counts[%d] < 0", t);
  int nb = 0;
  int t = 0;
  while (t < T) {
    batch_begin[nb++] = t;
    int64_t bytes = counts[t] * es;
    for (++t; t < T && bytes + counts[t] * es <= threshold_bytes; ++t) bytes += counts[t] * es;
  }
  batch_begin[nb] = T;
  *nbatches = nb;
  return VCOLL_OK;
}

static int fuse_common(const void* const* tensors, const int64_t* counts, int T,
                       const void* const* fused, int W, int dtype, int unpack, void* stream) {
  g_err[0] = 0;
  const int es = elem_size(dtype);
  if (!es) return fail(VCOLL_ERR_INVALID_TYPE, "unknown dtype %d", dtype);
  if (W < 1 || W > VCOLL_MAX_RANKS)
    return fail(VCOLL_ERR_INVALID_ARG, "W = %d outside [1, %d]", W, VCOLL_MAX_RANKS);
  if (T < 0 || (T > 0 && (!counts || !tensors)) || !fused)
    return fail(VCOLL_ERR_INVALID_ARG, "invalid fuse arguments");
  int64_t total = 0;
  for (int t = 0; t < T; ++t) {
    if (counts[t] < 0) return fail(VCOLL_ERR_INVALID_ARG, "counts[%d] < 0", t);
    total += counts[t];
  }
  std::vector<Buf> bufs;
  for (int u = 0; u < W; ++u) {
    if (total && !fused[u]) return fail(VCOLL_ERR_INVALID_ARG, "fused[%d] is NULL", u);
    if ((uint64_t)fused[u] % es)
      return fail(VCOLL_ERR_INVALID_ARG, "fused[%d] is not aligned to the element size", u);
    bufs.push_back({(uint64_t)fused[u], (uint64_t)(total * es), 0, true});
    for (int t = 0; t < T; ++t) {
      const void* p = tensors[(int64_t)u * T + t];
      if (!counts[t]) continue;
      if (!p) return fail(VCOLL_ERR_INVALID_ARG, "tensors[%d] is NULL", u * T + t);
      if ((uint64_t)p % es)
        return fail(VCOLL_ERR_INVALID_ARG, "tensors[%d] is not aligned to the element size",
                    u * T + t);
      bufs.push_back({(uint64_t)p, (uint64_t)(counts[t] * es), 1, true});
    }
  }
  int rc = check_disjoint(bufs);
  if (rc) return rc;
  if (total == 0) return VCOLL_OK;

  const int chunk = std::min(kFuseMaxTensors, kFuseMaxCopies / W);
  const int threads = 256;
  const int64_t tile_elems = (int64_t)threads * 4 * (16 / es);
  int64_t offset = 0;
  for (int t0 = 0; t0 < T; t0 += chunk) {
    const int nt = std::min(chunk, T - t0);
    FuseParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.T = nt;
    prm.W = W;
    prm.unpack = unpack;
    prm.tile_elems = tile_elems;
    int64_t tiles = 0;
    for (int t = 0; t < nt; ++t) {
      prm.count[t] = counts[t0 + t];
      prm.offset[t] = offset;
      prm.tile_begin[t] = tiles;
      tiles += ceil_div(counts[t0 + t], tile_elems);
      offset += counts[t0 + t];
    }
    prm.tile_begin[nt] = tiles;
    for (int u = 0; u < W; ++u) {
      prm.fused[u] = (void*)fused[u];
      for (int t = 0; t < nt; ++t) prm.tensor[t * W + u] = (void*)tensors[(int64_t)u * T + t0 + t];
    }
    if (tiles == 0) continue;
    // one CTA per (tile, rank)
    void* args[] = {&prm};
    cudaError_t e = launch_pdl(fuse_flat_kernel(es), dim3((unsigned)tiles, (unsigned)W),
                               dim3(threads), args, 0, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "fusion copy launch");
  }
  return VCOLL_OK;
}

int vcoll_fuse_pack(const void* const* tensors, const int64_t* counts, int T, void* const* fused,
                    int W, int dtype, void* stream) {
  return fuse_common(tensors, counts, T, (const void* const*)fused, W, dtype, 0, stream);
}

int vcoll_fuse_unpack(const void* const* fused, const int64_t* counts, int T,
                      void* const* tensors, int W, int dtype, void* stream) {
  return fuse_common((const void* const*)tensors, counts, T, fused, W, dtype, 1, stream);
}

// Multi-tensor allreduce over consecutive batches of tensors: batch b is
// tensors [batch_begin[b], batch_begin[b+1]), whose per-rank concatenation is
// one virtual buffer segmented on its own (as its fusion buffer would be).
// Pieces of different batches share launches; each carries its fold start.
static int multi_run(const void* const* in, void* const* out, const int64_t* counts, int T, int W,
                     int dtype, int op, unsigned flags, const std::vector<int>& batch_begin,
                     void* stream) {
  int rc = check_common(W, 0, dtype, op);
  if (rc) return rc;
  if (flags & ~(VCOLL_FLAG_RING_ORDER | VCOLL_FLAG_STAGED | VCOLL_FLAG_DIRECT))
    return fail(VCOLL_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  if (T < 0 || (T > 0 && (!counts || !in || !out)))
    return fail(VCOLL_ERR_INVALID_ARG, "invalid multi-tensor arguments");
  const int es = elem_size(dtype);
  // per tensor: its offset inside its batch's virtual buffer, and that size
  std::vector<int64_t> boff(T), bn(T);
  int64_t total = 0;
  for (size_t b = 0; b + 1 < batch_begin.size(); ++b) {
    int64_t o = 0;
    for (int t = batch_begin[b]; t < batch_begin[b + 1]; ++t) {
      if (counts[t] < 0) return fail(VCOLL_ERR_INVALID_ARG, "counts[%d] < 0", t);
      boff[t] = o;
      o += counts[t];
    }
    for (int t = batch_begin[b]; t < batch_begin[b + 1]; ++t) bn[t] = o;
    total += o;
  }
  std::vector<Buf> bufs;
  bufs.reserve(2 * (size_t)W * T);
  int64_t bbase = 0;  // distinct fused index space per batch for the aliasing check
  for (size_t b = 0; b + 1 < batch_begin.size(); ++b) {
    for (int u = 0; u < W; ++u)
      for (int t = batch_begin[b]; t < batch_begin[b + 1]; ++t) {
        if (!counts[t]) continue;
        const int64_t e = (int64_t)u * T + t;
        if (!in[e] || !out[e])
          return fail(VCOLL_ERR_INVALID_ARG, "tensor %d of rank %d is NULL", t, u);
        if ((uint64_t)in[e] % es || (uint64_t)out[e] % es)
          return fail(VCOLL_ERR_INVALID_ARG, "tensor %d of rank %d is not element-aligned", t, u);
        const uint64_t sh = (uint64_t)(bbase + boff[t]) * es;
        bufs.push_back({(uint64_t)in[e], (uint64_t)(counts[t] * es), (uint64_t)in[e] - sh, false});
        bufs.push_back({(uint64_t)out[e], (uint64_t)(counts[t] * es), (uint64_t)out[e] - sh, true});
      }
    bbase += bn[batch_begin[b]] + 1;
  }
  if ((rc = check_aliasing(bufs))) return rc;
  if (total == 0) return VCOLL_OK;
  if (W == 1) {
    for (int t = 0; t < T; ++t)
      if ((rc = copy_d2d(out[t], in[t], counts[t] * es, stream))) return rc;
    return VCOLL_OK;
  }

  const bool ring = (flags & VCOLL_FLAG_RING_ORDER) && op != VCOLL_MAX && op != VCOLL_MIN && W > 2;
  const int W_t = (W == 2 || W == 4 || W == 8 || W == 16) ? W : 0;
  const void* fn = dtype == VCOLL_F32 ? multi_kernel_f32(op, W_t, ring)
                                      : multi_kernel_bf16(op, W_t, ring);
  const int threads = 256;
  const int V = 16 / es;
  const int64_t tile_elems = (int64_t)threads * unroll_for(W_t) * V;
  const int max_t = std::min(kMultiMaxTensors, kMultiMaxPtrs / W);

  // pieces of one tensor: pieces of a batch segment, each with its fold start
  struct Cut {
    int64_t k0, len;
    int start;
  };
  auto cuts_of = [&](int tg, std::vector<Cut>& cuts) {
    cuts.clear();
    const int64_t n = bn[tg];
    int64_t k = 0;
    while (k < counts[tg]) {
      const int64_t i = boff[tg] + k;
      int j = 0;
      int64_t seg_end = n;
      if (ring) {
        const int64_t q = n / W, r = n % W;
        const int64_t big = r * (q + 1);
        j = i < big ? (int)(i / (q + 1)) : (int)(r + (i - big) / q);
        int64_t so, sl;
        segment_of(n, W, j, &so, &sl);
        seg_end = so + sl;
      }
      const int64_t len = std::min(counts[tg] - k, seg_end - i);
      cuts.push_back({k, len, ring ? (j + 1) % W : 0});
      k += len;
    }
  };

  static_assert(kMultiMaxPieces >= VCOLL_MAX_RANKS, "a tensor has at most W pieces");
  std::vector<Cut> cuts;
  MultiParams prm;
  int t0 = 0;
  while (t0 < T) {
    memset(&prm, 0, sizeof(prm));
    prm.W = W;
    prm.scale = op == VCOLL_AVG ? 1.0f / (float)W : 1.0f;
    prm.do_scale = op == VCOLL_AVG ? 1 : 0;
    prm.tile_elems = tile_elems;
    int nt = 0, np = 0;
    int64_t tiles = 0;
    // take tensors while both the pointer table and the piece table have room
    while (t0 + nt < T && nt < max_t) {
      const int tg = t0 + nt;
      cuts_of(tg, cuts);
      if (np + (int)cuts.size() > kMultiMaxPieces) break;
      for (const Cut& c : cuts) {
        MultiPiece& pc = prm.piece[np++];
        pc.k0 = c.k0;
        pc.len = c.len;
        pc.tile_begin = tiles;
        pc.t = nt;
        pc.start = c.start;
        // one 16-byte phase for every rank's input and output at element k0?
        int ph = -1;
        bool same = true;
        for (int u = 0; u < W && same; ++u) {
          const uint64_t a = (uint64_t)in[(int64_t)u * T + tg] + (uint64_t)c.k0 * es;
          const uint64_t o = (uint64_t)out[(int64_t)u * T + tg] + (uint64_t)c.k0 * es;
          const int pa = (int)(a & 15), pb = (int)(o & 15);
          if (ph < 0) ph = pa;
          same = (pa == ph) && (pb == ph);
        }
        pc.phase = same ? ph / es : -1;
        tiles += std::max<int64_t>(1, ceil_div(c.len, tile_elems));
      }
      ++nt;
    }
    // pointer tables of the nt tensors taken, tensor-major (t * W + u)
    prm.T = nt;
    for (int u = 0; u < W; ++u)
      for (int t = 0; t < nt; ++t) {
        prm.in[t * W + u] = in[(int64_t)u * T + t0 + t];
        prm.out[t * W + u] = out[(int64_t)u * T + t0 + t];
      }
    prm.npieces = np;
    prm.num_tiles = tiles;
    if (np > 0 && (rc = launch(fn, tiles, threads, 0, false, &prm, stream)))
      return rc;
    t0 += nt;
  }
  return VCOLL_OK;
}

int vcoll_allreduce_multi(const void* const* in, void* const* out, const int64_t* counts, int T,
                          int W, int dtype, int op, unsigned flags, void* stream) {
  g_err[0] = 0;
  if (T < 0) return fail(VCOLL_ERR_INVALID_ARG, "T = %d < 0", T);
  std::vector<int> begin = {0, T};
  return multi_run(in, out, counts, T, W, dtype, op, flags, begin, stream);
}

int vcoll_fusion_allreduce(const void* const* in, void* const* out, const int64_t* counts, int T,
                           int W, int dtype, int op, unsigned flags, int64_t threshold_bytes,
                           int* nbatches, void* stream) {
  g_err[0] = 0;
  if (T < 0) return fail(VCOLL_ERR_INVALID_ARG, "T = %d < 0", T);
  std::vector<int> begin(T + 1);
  int nb = 0;
  int rc = vcoll_fuse_plan(counts, T, dtype, threshold_bytes, begin.data(), &nb);
  if (rc) return rc;
  begin.resize(nb + 1);
  if (nbatches) *nbatches = nb;
  return multi_run(in, out, counts, T, W, dtype, op, flags, begin, stream);
}

int vcoll_fusion_allreduce_buffered(const void* const* in, void* const* out,
                                    const int64_t* counts, int T, void* const* fused,
                                    int64_t fused_bytes, int W, int dtype, int op, unsigned flags,
                                    int64_t threshold_bytes, int* nbatches, void* stream) {
  g_err[0] = 0;
  int rc = check_common(W, 0, dtype, op);
  if (rc) return rc;
  if (flags & ~(VCOLL_FLAG_RING_ORDER | VCOLL_FLAG_STAGED | VCOLL_FLAG_DIRECT))
    return fail(VCOLL_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  if (T < 0) return fail(VCOLL_ERR_INVALID_ARG, "T = %d < 0", T);
  if (T > 0 && (!counts || !in || !out))
    return fail(VCOLL_ERR_INVALID_ARG, "invalid fusion arguments");
  if (!fused || fused_bytes < 0) return fail(VCOLL_ERR_INVALID_ARG, "invalid fusion buffers");
  const int es = elem_size(dtype);
  std::vector<int> begin(T + 1);
  int nb = 0;
  if ((rc = vcoll_fuse_plan(counts, T, dtype, threshold_bytes, begin.data(), &nb))) return rc;
  // every check before the first launch: a call that fails enqueues nothing
  for (int u = 0; u < W; ++u) {
    if (!fused[u]) return fail(VCOLL_ERR_INVALID_ARG, "fused[%d] is NULL", u);
    for (int t = 0; t < T; ++t) {
      const int64_t e = (int64_t)u * T + t;
      if (counts[t] && (!in[e] || !out[e]))
        return fail(VCOLL_ERR_INVALID_ARG, "tensor %d of rank %d is NULL", t, u);
    }
  }
  for (int b = 0; b < nb; ++b) {
    if (begin[b + 1] - begin[b] < 2) continue;
    int64_t bytes = 0;
    for (int t = begin[b]; t < begin[b + 1]; ++t) bytes += counts[t] * es;
    if (bytes > fused_bytes)
      return fail(VCOLL_ERR_INVALID_ARG,
                  "batch %d of the plan needs %lld bytes of fusion buffer, fused_bytes = %lld", b,
                  (long long)bytes, (long long)fused_bytes);
  }
  if (nbatches) *nbatches = nb;
  std::vector<const void*> bin((size_t)W * (T > 0 ? T : 1)), bout((size_t)W * (T > 0 ? T : 1));
  for (int b = 0; b < nb; ++b) {
    const int t0 = begin[b], nt = begin[b + 1] - begin[b];
    // the batch's tensors, rank-major
    for (int u = 0; u < W; ++u)
      for (int t = 0; t < nt; ++t) {
        bin[(size_t)u * nt + t] = in[(int64_t)u * T + t0 + t];
        bout[(size_t)u * nt + t] = out[(int64_t)u * T + t0 + t];
      }
    if (nt == 1) {  // one tensor: allreduced straight from its input to its output
      if ((rc = reduce_common(KIND_AR, bin.data(), (void* const*)bout.data(), W, counts[t0], dtype,
                              op, flags, stream)))
        return rc;
      continue;
    }
    int64_t n = 0;
    for (int t = t0; t < t0 + nt; ++t) n += counts[t];
    if ((rc = fuse_common(bin.data(), counts + t0, nt, (const void* const*)fused, W, dtype, 0,
                          stream)) ||
        (rc = reduce_common(KIND_AR, (const void* const*)fused, fused, W, n, dtype, op, flags,
                            stream)) ||
        (rc = fuse_common(bout.data(), counts + t0, nt, (const void* const*)fused, W, dtype, 1,
                          stream)))
      return rc;
  }
  return VCOLL_OK;
}

size_t vcoll_sparse_workspace_bytes(int W, int64_t n, int topk) {
  if (W < 1 || W > VCOLL_MAX_RANKS || n < 0 || !topk) return 0;
  return topk_workspace_bytes(W, n);
}

size_t vcoll_sparse_workspace_min_bytes(int W, int64_t n, int topk) {
  if (W < 1 || W > VCOLL_MAX_RANKS || n < 0 || !topk) return 0;
  return topk_workspace_min_bytes(W, n);
}

int vcoll_sparse_allreduce(const void* const* in, void* const* out, void* const* accum, int W,
                           int64_t n, float threshold, int topk, int64_t* nnz, void* workspace,
                           size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  int rc = check_common(W, n, VCOLL_F32, VCOLL_SUM);
  if (rc) return rc;
  if (topk && !(threshold >= 0.0f && threshold <= 1.0f))
    return fail(VCOLL_ERR_INVALID_ARG, "top-K fraction %g outside [0, 1]", (double)threshold);
  if (topk && n >= (int64_t)1 << 32)
    return fail(VCOLL_ERR_UNSUPPORTED, "top-K needs n < 2^32 elements per rank");
  int64_t lens[VCOLL_MAX_RANKS];
  for (int u = 0; u < W; ++u) lens[u] = n;
  if ((rc = check_ptrs(in, W, "in", 4, lens))) return rc;
  if ((rc = check_ptrs((const void* const*)out, W, "out", 4, lens))) return rc;
  if (accum && (rc = check_ptrs((const void* const*)accum, W, "accum", 4, lens))) return rc;
  // the survivor counts are outputs: zero them first (also when n == 0)
  if (nnz) {
    if ((uint64_t)nnz % 8) return fail(VCOLL_ERR_INVALID_ARG, "nnz is not 8-byte aligned");
    cudaError_t e = cudaMemsetAsync(nnz, 0, sizeof(int64_t) * W, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  }
  if (n == 0) return VCOLL_OK;
  std::vector<Buf> bufs;
  for (int u = 0; u < W; ++u) {
    bufs.push_back({(uint64_t)in[u], (uint64_t)(n * 4), (uint64_t)in[u], false});
    bufs.push_back({(uint64_t)out[u], (uint64_t)(n * 4), (uint64_t)out[u], true});
    if (accum) bufs.push_back({(uint64_t)accum[u], (uint64_t)(n * 4), (uint64_t)accum[u], true});
  }
  int vec, phase;
  if ((rc = analyse(bufs, 4, &vec, &phase))) return rc;

  int64_t K = 0;
  if (topk) {
    // K = ceil(threshold * num) in fp32, as SINGA computes nnzMax
    const float kf = ceilf(threshold * (float)n);
    K = kf >= (float)n ? n : (int64_t)kf;
    if (!workspace || workspace_bytes < topk_workspace_min_bytes(W, n))
      return fail(VCOLL_ERR_INVALID_ARG, "top-K needs a workspace of at least %zu bytes",
                  topk_workspace_min_bytes(W, n));
    if ((uint64_t)workspace % 16) return fail(VCOLL_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  }
  SparseParams prm;
  memset(&prm, 0, sizeof(prm));
  for (int u = 0; u < W; ++u) {
    prm.in[u] = in[u];
    prm.out[u] = out[u];
    prm.acc[u] = accum ? accum[u] : nullptr;
  }
  prm.nnz = nnz;
  prm.n = n;
  prm.W = W;
  prm.K = K;
  prm.phase = vec ? phase : -1;
  prm.has_acc = accum ? 1 : 0;
  prm.threshold = threshold;
  prm.tile_elems = kSparseTileElems;
  prm.tiles_per_rank = ceil_div(n, prm.tile_elems);
  prm.num_tiles = prm.tiles_per_rank;
  return sparse_launch(prm, topk, workspace, workspace_bytes, stream);
}

int vcoll_selftest_wait_timeout(unsigned limit_us, void* stream) {
  g_err[0] = 0;
  if (limit_us == 0 || limit_us > 1000000)
    return fail(VCOLL_ERR_INVALID_ARG, "limit_us = %u outside [1, 1000000]", limit_us);
  uint64_t limit_ns = (uint64_t)limit_us * 1000ull;
  void* args[] = {&limit_ns};
  cudaError_t e = cudaLaunchKernel(selftest_timeout_kernel(), dim3(1), dim3(32), args, 0,
                                   (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return VCOLL_OK;
}

int vcoll_device_errors(unsigned* flags, int clear) {
  g_err[0] = 0;
  if (!flags) return fail(VCOLL_ERR_INVALID_ARG, "flags is NULL");
  unsigned int* sym = device_error_symbol();
  if (!sym) return fail(VCOLL_ERR_CUDA, "cannot resolve the device error word");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(flags, sym, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  if (clear) {
    e = cudaMemset(sym, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  }
  return VCOLL_OK;
}

int vcoll_segment(int64_t n, int W, int j, int64_t* off, int64_t* len) {
  g_err[0] = 0;
  if (n < 0 || W < 1 || W > VCOLL_MAX_RANKS || j < 0 || j >= W || !off || !len)
    return fail(VCOLL_ERR_INVALID_ARG, "invalid segment arguments");
  segment_of(n, W, j, off, len);
  return VCOLL_OK;
}

const char* vcoll_status_string(int status) {
  switch (status) {
    case VCOLL_OK:
      return "success";
    case VCOLL_ERR_INVALID_ARG:
      return "invalid argument";
    case VCOLL_ERR_INVALID_TYPE:
      return "invalid data type";
    case VCOLL_ERR_INVALID_OP:
      return "invalid reduction operation";
    case VCOLL_ERR_UNSUPPORTED:
      return "unsupported request";
    case VCOLL_ERR_CUDA:
      return "CUDA error";
    default:
      return "unknown status";
  }
}

const char* vcoll_last_error(void) { return g_err; }

}  // extern "C"

namespace vcoll {
// lets entry points defined in other translation units report a failure
// through vcoll_last_error()
int report_error(int status, const char* message) { return fail(status, "%s", message); }
}  // namespace vcoll

extern "C" {

int vcoll_version(void) { return 200; }

}  // extern "C"

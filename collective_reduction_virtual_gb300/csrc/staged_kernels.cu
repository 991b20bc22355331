// Staged reduce-scatter / allreduce: the W input slices of each tile travel
// HBM -> shared memory by bulk asynchronous copies (TMA, cp.async.bulk, no
// multicast), through a ring of kStagedStages stages guarded by mbarriers.
//
// One producer warp (one elected lane) issues, per tile, W bulk copies of one
// rank's slice each -- placed in fold order (ring: rank (j+1) mod W first) --
// and arms the stage's "full" barrier with the expected byte count.  Eight
// consumer warps wait on "full", fold the W slices from shared memory in fp32
// (same fold and rounding as the direct kernels, so the bits are identical),
// apply the avg scale and the output cast, store to global memory, and
// release the stage on its "empty" barrier.  Up to kStagedStages * 32 KB of
// input is in flight per SM without holding it in registers.
//
// Every wait is bounded: after kWaitLimitNs of wall-clock time (the GPU's
// global timer) the waiting thread records VCOLL_DEVICE_ERR_TIMEOUT in
// g_vcoll_device_error and the CTA stops issuing work; the producer then
// waits, again bounded, for the copies it has already issued before it
// returns.
#include "device_common.cuh"
#include "reduce_kernels.cuh"
#include "vcoll_internal.h"

namespace vcoll {

__device__ unsigned int g_vcoll_device_error = 0;

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// The drain before a producer returns: copies already issued cannot be
// cancelled, and the CTA (its shared memory and mbarriers) must stay resident
// until they land, so this wait is allowed much longer before it gives up.
constexpr uint64_t kDrainLimitNs = 20000000000ull;  // 20 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity; false on timeout (after
// limit_ns of wall-clock time), with VCOLL_DEVICE_ERR_TIMEOUT recorded.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) {
      atomicOr(&g_vcoll_device_error, (unsigned)VCOLL_DEVICE_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, unsigned bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most N committed bulk groups may still be reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace

template <typename T, int WT, class Op, int KIND, int RING>
__global__ void __launch_bounds__(kStagedThreads, 1)
    vc_reduce_staged(const __grid_constant__ ReduceParams p) {
  pdl_enter();
  using E = Elem<T>;
  constexpr int V = E::kVec;
  constexpr int SLICE = staged_slice_bytes(WT);
  constexpr int STAGE = WT * SLICE;
  constexpr int S = kStagedStages;
  constexpr int TREE_W = RING ? 0 : WT;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStagedConsumerWarps);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kStagedConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++issued) {
        const int s = issued % S;
        if (issued >= S && !mbar_wait(&empty[s], ((issued / S) - 1) & 1)) {
          abort_flag = 1;
          break;
        }
        if (abort_flag) break;
        const TileRange tr = tile_range<V>(p, tile);
        const int64_t n_el = tr.e1 > tr.e0 ? tr.e1 - tr.e0 : 0;
        const unsigned bytes = (unsigned)(n_el * E::kBytes);
        mbar_arrive_expect_tx(&full[s], bytes * WT);
        if (bytes) {
          const int start = RING ? p.ring_start[tr.j] : 0;
          unsigned char* st = smem + s * STAGE;
#pragma unroll
          for (int t = 0; t < WT; ++t) {
            const int src = RING ? rotate(start, t, WT) : t;
            bulk_load(st + t * SLICE, (const char*)p.in[src] + tr.e0 * E::kBytes, bytes, &full[s]);
          }
        }
      }
      // wait (bounded, with the longer drain limit) until every copy this
      // CTA issued has landed; the other threads may have returned, but the
      // CTA stays resident while this lane waits
      for (int i = issued - S < 0 ? 0 : issued - S; i < issued; ++i)
        mbar_wait(&full[i % S], (i / S) & 1, kDrainLimitNs);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int it = 0;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
    const int s = it % S;
    if (!mbar_wait(&full[s], (it / S) & 1)) {
      abort_flag = 1;
      break;
    }
    const TileRange tr = tile_range<V>(p, tile);
    const int start = RING ? p.ring_start[tr.j] : 0;
    const int64_t nvec = tr.e1 > tr.e0 ? (tr.e1 - tr.e0) / V : 0;
    const unsigned char* st = smem + s * STAGE;
    for (int64_t vi = tid; vi < nvec; vi += kStagedConsumerWarps * 32) {
      uint4 v[WT];
#pragma unroll
      for (int t = 0; t < WT; ++t)
        v[t] = *reinterpret_cast<const uint4*>(st + t * SLICE + vi * 16);
      float acc[V];
      if (RING)
        left_fold<T, Op, WT>(v, acc);
      else
        TreeFold<T, Op, WT, 0, WT>::run(v, acc);
      if (p.do_scale) {
#pragma unroll
        for (int x = 0; x < V; ++x) acc[x] = __fmul_rn(acc[x], p.scale);
      }
      const uint4 o = E::narrow(acc);
      const int64_t e = tr.e0 + vi * V;
      if (KIND == KIND_AR) {
#pragma unroll
        for (int r = 0; r < WT; ++r) st_stream((char*)p.out[r] + e * E::kBytes, o);
      } else {
        st_stream((char*)p.out[tr.j] + (e - tr.a) * E::kBytes, o);
      }
    }
    if (tr.first) head_tail<T, Op, KIND, TREE_W>(p, tr, WT, start);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (abort_flag) break;
  }
}

namespace {
template <typename T, class Op, int KIND>
const void* pick_staged(int W_t, int ring) {
  switch (W_t) {
    case 2:
      return (const void*)&vc_reduce_staged<T, 2, Op, KIND, 0>;
    case 4:
      return ring ? (const void*)&vc_reduce_staged<T, 4, Op, KIND, 1>
                  : (const void*)&vc_reduce_staged<T, 4, Op, KIND, 0>;
    case 8:
      return ring ? (const void*)&vc_reduce_staged<T, 8, Op, KIND, 1>
                  : (const void*)&vc_reduce_staged<T, 8, Op, KIND, 0>;
    case 16:
      return ring ? (const void*)&vc_reduce_staged<T, 16, Op, KIND, 1>
                  : (const void*)&vc_reduce_staged<T, 16, Op, KIND, 0>;
    default:
      return nullptr;
  }
}

template <typename T>
const void* staged_table(int op, int kind, int W_t, int ring) {
  if (op == VCOLL_MAX)  // order-independent: the tree instantiation serves both orders
    return kind == KIND_AR ? pick_staged<T, OpMax, KIND_AR>(W_t, 0)
                           : pick_staged<T, OpMax, KIND_RS>(W_t, 0);
  if (op == VCOLL_MIN)
    return kind == KIND_AR ? pick_staged<T, OpMin, KIND_AR>(W_t, 0)
                           : pick_staged<T, OpMin, KIND_RS>(W_t, 0);
  if (op == VCOLL_PROD)
    return kind == KIND_AR ? pick_staged<T, OpProd, KIND_AR>(W_t, ring)
                           : pick_staged<T, OpProd, KIND_RS>(W_t, ring);
  return kind == KIND_AR ? pick_staged<T, OpSum, KIND_AR>(W_t, ring)
                         : pick_staged<T, OpSum, KIND_RS>(W_t, ring);
}
}  // namespace

// ---------------------------------------------------------------------------
// Allgather on the TMA engine: one thread per CTA moves each tile of segment j
// HBM -> shared memory with one bulk copy, then shared memory -> the W
// outputs with W bulk stores; kGatherStages tiles in flight.  Before a stage
// is refilled, the stores that read it (kGatherStages - 1 groups ago) must
// have finished reading.  The unaligned head and tail of each segment (< 16
// bytes each) are copied by ordinary threads.
constexpr int kGatherStages = kGatherTmaStages;
constexpr int kGatherTileBytes = kGatherTmaTileBytes;

template <int ES>
__global__ void __launch_bounds__(kGatherTmaThreads, 1) vc_gather_tma(const __grid_constant__ GatherParams p) {
  pdl_enter();
  using B = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
  constexpr int V = 16 / ES;
  constexpr int S = kGatherStages;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kGatherTileBytes);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int W = p.W;
  // tile i of this CTA: its aligned body [e0, e1) inside segment j
  auto range = [&](int64_t tile, int& j, int64_t& a, int64_t& b, int64_t& e0, int64_t& e1,
                   int64_t& av, int64_t& bv) {
    j = (int)(tile / p.tiles_per_seg);
    const int64_t k = tile - (int64_t)j * p.tiles_per_seg;
    a = p.disp[j];
    b = p.disp[j + 1];
    aligned_body<V>(a, b, p.phase, av, bv);
    e0 = av + k * p.tile_elems;
    e1 = e0 + p.tile_elems < bv ? e0 + p.tile_elems : bv;
    if (e1 < e0) e1 = e0;
  };
  // unaligned heads and tails, element by element, by every thread
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    int j;
    int64_t a, b, e0, e1, av, bv;
    range(tile, j, a, b, e0, e1, av, bv);
    if (tile - (int64_t)j * p.tiles_per_seg != 0) continue;
    const char* src = (const char*)p.in[j] - a * ES;
    int64_t i = -1;
    if (tid < av - a) i = a + tid;
    if (tid >= 32 && tid - 32 < b - bv) i = bv + (tid - 32);
    if (i >= 0) {
      const B x = ld1<B>(src + i * ES);
      for (int r = 0; r < W; ++r) st1((char*)p.out[r] + i * ES, x);
    }
  }
  if (tid != 0) return;
  // bodies: one thread drives the TMA engine
  const int64_t n_mine = blockIdx.x < p.num_tiles
                             ? (p.num_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x
                             : 0;
  auto issue = [&](int64_t i) {  // load tile i into stage i % S
    int j;
    int64_t a, b, e0, e1, av, bv;
    range(blockIdx.x + i * gridDim.x, j, a, b, e0, e1, av, bv);
    const int s = (int)(i % S);
    const unsigned bytes = (unsigned)((e1 - e0) * ES);
    mbar_arrive_expect_tx(&full[s], bytes);
    if (bytes)
      bulk_load(smem + s * kGatherTileBytes, (const char*)p.in[j] + (e0 - a) * ES, bytes, &full[s]);
  };
  for (int64_t i = 0; i < n_mine && i < S; ++i) issue(i);
  int64_t issued = n_mine < S ? n_mine : S;
  int64_t consumed = 0;
  for (int64_t i = 0; i < n_mine; ++i) {
    const int s = (int)(i % S);
    if (!mbar_wait(&full[s], (unsigned)((i / S) & 1))) break;
    consumed = i + 1;
    int j;
    int64_t a, b, e0, e1, av, bv;
    range(blockIdx.x + i * gridDim.x, j, a, b, e0, e1, av, bv);
    const unsigned bytes = (unsigned)((e1 - e0) * ES);
    if (bytes) {
      fence_proxy_async_smem();
      for (int r = 0; r < W; ++r)
        bulk_store((char*)p.out[r] + e0 * ES, smem + s * kGatherTileBytes, bytes);
    }
    bulk_commit();
    // refill the stage used one tile ago once its stores have read it
    if (i >= 1 && issued < n_mine) {
      bulk_wait_read<1>();
      issue(issued);
      ++issued;
    }
  }
  // after a timeout: wait (bounded, with the longer drain limit) for the
  // loads issued but not consumed
  for (int64_t i = consumed; i < issued; ++i)
    mbar_wait(&full[i % S], (unsigned)((i / S) & 1), kDrainLimitNs);
  bulk_wait_all();
}

// Diagnostics: one thread waits on a barrier that nothing arrives at; the
// wait must give up after limit_ns and record the timeout.
__global__ void vc_selftest_wait_timeout(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(&bar, 0, limit_ns);
  }
}

const void* selftest_timeout_kernel() { return (const void*)&vc_selftest_wait_timeout; }

const void* gather_tma_kernel(int elem_size) {
  return elem_size == 4 ? (const void*)&vc_gather_tma<4> : (const void*)&vc_gather_tma<2>;
}

const void* staged_kernel_f32(int op, int kind, int W_t, int ring) {
  return staged_table<float>(op, kind, W_t, ring);
}
const void* staged_kernel_bf16(int op, int kind, int W_t, int ring) {
  return staged_table<__nv_bfloat16>(op, kind, W_t, ring);
}

unsigned int* device_error_symbol() {
  unsigned int* p = nullptr;
  if (cudaGetSymbolAddress((void**)&p, g_vcoll_device_error) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace vcoll

// Direct-load reduce-scatter / allreduce kernels.
//
// One pass over the element index space: every thread loads the W ranks'
// values at its indices straight into registers (16-byte streaming loads,
// all W * U loads of a tile issued before the first add), folds them in fp32,
// applies the avg scale and the output cast, and stores the result -- once
// (reduce-scatter, into the segment's owner) or W times (allreduce).
//
// The fold order is the early NCCL ring's (ReduceScatterKernel: block j
// starts at the ring position after its owner, every later position applies
// FUNC(buffer, own input), the owner applies it last) when `ring` is set, so
// the bits equal the ring's; otherwise a pairwise tree over the ranks.  Each
// output element is written by the thread that read all W inputs at that
// index, after those reads, so in-place operation is race-free (the
// read-before-write rule of MLX PR #3901's ring scatter-reduce).
#pragma once

#include "device_common.cuh"
#include "vcoll_internal.h"

namespace vcoll {

__device__ __forceinline__ int rotate(int start, int t, int W) {
  int i = start + t;
  return i >= W ? i - W : i;
}

// Pairwise tree over ranks [LO, LO + CNT) of already-loaded vectors.
template <typename T, class Op, int WT, int LO, int CNT>
struct TreeFold {
  static __device__ __forceinline__ void run(const uint4 (&v)[WT], float (&out)[Elem<T>::kVec]) {
    float a[Elem<T>::kVec], b[Elem<T>::kVec];
    TreeFold<T, Op, WT, LO, CNT / 2>::run(v, a);
    TreeFold<T, Op, WT, LO + CNT / 2, CNT - CNT / 2>::run(v, b);
#pragma unroll
    for (int e = 0; e < Elem<T>::kVec; ++e) out[e] = Op::apply(a[e], b[e]);
  }
};
template <typename T, class Op, int WT, int LO>
struct TreeFold<T, Op, WT, LO, 1> {
  static __device__ __forceinline__ void run(const uint4 (&v)[WT], float (&out)[Elem<T>::kVec]) {
    Elem<T>::widen(v[LO], out);
  }
};

// Left fold, accumulator first, over vectors already placed in fold order.
template <typename T, class Op, int WT>
__device__ __forceinline__ void left_fold(const uint4 (&v)[WT], float (&acc)[Elem<T>::kVec]) {
  Elem<T>::widen(v[0], acc);
#pragma unroll
  for (int t = 1; t < WT; ++t) {
    float x[Elem<T>::kVec];
    Elem<T>::widen(v[t], x);
#pragma unroll
    for (int e = 0; e < Elem<T>::kVec; ++e) acc[e] = Op::apply(acc[e], x[e]);
  }
}

// One element at index i (head/tail of a segment, or the element-wise path):
// left fold from rank `start` (ring order, or rank 0), or the same pairwise
// tree as the vector path when TREE_W > 0.
template <typename T, class Op, int TREE_W>
struct ScalarFold;

template <typename T, class Op>
struct ScalarFold<T, Op, 0> {
  static __device__ __forceinline__ float run(const ReduceParams& p, int W, int start, int64_t i) {
    using B = typename Elem<T>::Bits;
    const int64_t off = i * Elem<T>::kBytes;
    float acc = Elem<T>::widen1(ld1<B>((const char*)p.in[start] + off));
#pragma unroll 4
    for (int t = 1; t < W; ++t) {
      const int src = rotate(start, t, W);
      acc = Op::apply(acc, Elem<T>::widen1(ld1<B>((const char*)p.in[src] + off)));
    }
    return acc;
  }
};

template <typename T, class Op, int LO, int CNT>
struct ScalarTree {
  static __device__ __forceinline__ float run(const ReduceParams& p, int64_t off) {
    float a = ScalarTree<T, Op, LO, CNT / 2>::run(p, off);
    float b = ScalarTree<T, Op, LO + CNT / 2, CNT - CNT / 2>::run(p, off);
    return Op::apply(a, b);
  }
};
template <typename T, class Op, int LO>
struct ScalarTree<T, Op, LO, 1> {
  static __device__ __forceinline__ float run(const ReduceParams& p, int64_t off) {
    using B = typename Elem<T>::Bits;
    return Elem<T>::widen1(ld1<B>((const char*)p.in[LO] + off));
  }
};

template <typename T, class Op, int TREE_W>
struct ScalarFold {
  static __device__ __forceinline__ float run(const ReduceParams& p, int, int, int64_t i) {
    return ScalarTree<T, Op, 0, TREE_W>::run(p, i * Elem<T>::kBytes);
  }
};

template <typename T, class Op, int KIND, int TREE_W>
__device__ __forceinline__ void reduce_one(const ReduceParams& p, int W, int start, int j,
                                           int64_t a, int64_t i) {
  using E = Elem<T>;
  float acc = ScalarFold<T, Op, TREE_W>::run(p, W, start, i);
  if (p.do_scale) acc = __fmul_rn(acc, p.scale);
  const typename E::Bits o = E::narrow1(acc);
  if (KIND == KIND_AR) {
    for (int u = 0; u < W; ++u) st1(((char*)p.out[u]) + i * E::kBytes, o);
  } else {
    st1(((char*)p.out[j]) + (i - a) * E::kBytes, o);
  }
}

// Tile bookkeeping shared by the kernels: segment j and tile k of `tile`.
struct TileRange {
  int j;
  int64_t a, b;    // segment bounds
  int64_t av, bv;  // aligned body
  int64_t e0, e1;  // this tile's part of the body
  bool first;      // tile 0 of the segment also does head and tail
};

template <int V>
__device__ __forceinline__ TileRange tile_range(const ReduceParams& p, int64_t tile) {
  TileRange t;
  t.j = (int)(tile / p.tiles_per_seg);
  const int64_t k = tile - (int64_t)t.j * p.tiles_per_seg;
  segment_bounds(p.n, p.q, p.r, p.nseg, t.j, t.a, t.b);
  aligned_body<V>(t.a, t.b, p.phase, t.av, t.bv);
  t.e0 = t.av + k * p.tile_elems;
  t.e1 = t.e0 + p.tile_elems < t.bv ? t.e0 + p.tile_elems : t.bv;
  t.first = (k == 0);
  return t;
}

// Head [a, av) and tail [bv, b) of the segment, one element per thread.
template <typename T, class Op, int KIND, int TREE_W>
__device__ __forceinline__ void head_tail(const ReduceParams& p, const TileRange& t, int W,
                                          int start) {
  const int64_t nh = t.av - t.a;
  const int64_t nt = t.b - t.bv;
  const int tid = threadIdx.x;
  if (tid < nh) reduce_one<T, Op, KIND, TREE_W>(p, W, start, t.j, t.a, t.a + tid);
  const int k = tid - 32;
  if (k >= 0 && k < nt) reduce_one<T, Op, KIND, TREE_W>(p, W, start, t.j, t.a, t.bv + k);
}

// ---------------------------------------------------------------------------
// Vector kernel for a compile-time rank count WT in {2, 4, 8, 16}.
// RING = 1: loads are placed in ring order starting at rank (j+1) mod W and
// folded left; RING = 0: natural rank order, pairwise tree.
template <typename T, int WT, class Op, int KIND, int RING>
__global__ void __launch_bounds__(256) vc_reduce_vec(const __grid_constant__ ReduceParams p) {
  pdl_enter();
  using E = Elem<T>;
  constexpr int V = E::kVec;
  constexpr int U = unroll_for(WT);
  constexpr int TREE_W = RING ? 0 : WT;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const TileRange tr = tile_range<V>(p, tile);
    const int start = RING ? p.ring_start[tr.j] : 0;
    uint4 v[U][WT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e = tr.e0 + ((int64_t)u * nthr + tid) * V;
      if (e < tr.e1) {
#pragma unroll
        for (int t = 0; t < WT; ++t) {
          const int src = RING ? rotate(start, t, WT) : t;
          v[u][t] = ld_stream((const char*)p.in[src] + e * E::kBytes);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int t = 0; t < WT; ++t) reg_fence(v[u][t]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e = tr.e0 + ((int64_t)u * nthr + tid) * V;
      if (e < tr.e1) {
        float acc[V];
        if (RING)
          left_fold<T, Op, WT>(v[u], acc);
        else
          TreeFold<T, Op, WT, 0, WT>::run(v[u], acc);
        if (p.do_scale) {
#pragma unroll
          for (int x = 0; x < V; ++x) acc[x] = __fmul_rn(acc[x], p.scale);
        }
        const uint4 o = E::narrow(acc);
        if (KIND == KIND_AR) {
#pragma unroll
          for (int r = 0; r < WT; ++r) st_stream((char*)p.out[r] + e * E::kBytes, o);
        } else {
          st_stream((char*)p.out[tr.j] + (e - tr.a) * E::kBytes, o);
        }
      }
    }
    if (tr.first) head_tail<T, Op, KIND, TREE_W>(p, tr, WT, start);
  }
}

// ---------------------------------------------------------------------------
// Vector kernel for any W (runtime, <= 64): left fold from rank (j+1) mod W
// (ring) or rank 0; the U vectors of a thread load two ranks at a time
// before folding them.
template <typename T, class Op, int KIND>
__global__ void __launch_bounds__(256) vc_reduce_vec_any(const __grid_constant__ ReduceParams p) {
  pdl_enter();
  using E = Elem<T>;
  constexpr int V = E::kVec;
  constexpr int U = unroll_for(0);
  constexpr int G = 2;  // ranks per round trip: 2 beat 4 for reduce-scatter (W = 9, 12)
  const int W = p.W;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const TileRange tr = tile_range<V>(p, tile);
    const int start = p.ring ? p.ring_start[tr.j] : 0;
    int64_t e[U];
    bool ok[U];
    float acc[U][V];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      e[u] = tr.e0 + ((int64_t)u * nthr + tid) * V;
      ok[u] = e[u] < tr.e1;
    }
    for (int t0 = 0; t0 < W; t0 += G) {
      uint4 g[U][G];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < G; ++i)
          if (ok[u] && t0 + i < W)
            g[u][i] = ld_stream((const char*)p.in[rotate(start, t0 + i, W)] + e[u] * E::kBytes);
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < G; ++i) reg_fence(g[u][i]);
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
          if (ok[u] && t0 + i < W) {
            float x[V];
            E::widen(g[u][i], x);
            if (t0 + i == 0) {
#pragma unroll
              for (int q = 0; q < V; ++q) acc[u][q] = x[q];
            } else {
#pragma unroll
              for (int q = 0; q < V; ++q) acc[u][q] = Op::apply(acc[u][q], x[q]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ok[u]) {
        if (p.do_scale) {
#pragma unroll
          for (int q = 0; q < V; ++q) acc[u][q] = __fmul_rn(acc[u][q], p.scale);
        }
        const uint4 o = E::narrow(acc[u]);
        if (KIND == KIND_AR) {
          for (int r = 0; r < W; ++r) st_stream((char*)p.out[r] + e[u] * E::kBytes, o);
        } else {
          st_stream((char*)p.out[tr.j] + (e[u] - tr.a) * E::kBytes, o);
        }
      }
    }
    if (tr.first) head_tail<T, Op, KIND, 0>(p, tr, W, start);
  }
}

// Vector grid of a realigning kernel's tile: the allreduce's outputs share
// one grid; a reduce-scatter segment j follows its own output (element i at
// out[j] + (i - a) * s).  p.out_phase[j] = element 0's address mod 16 on that
// grid.
template <int V, int KIND>
__device__ __forceinline__ TileRange realign_range(const ReduceParams& p, int64_t tile) {
  constexpr int S = 16 / V;  // element bytes
  TileRange t;
  t.j = (int)(tile / p.tiles_per_seg);
  const int64_t k = tile - (int64_t)t.j * p.tiles_per_seg;
  segment_bounds(p.n, p.q, p.r, p.nseg, t.j, t.a, t.b);
  const int phase = p.out_phase[t.j] / S;
  aligned_body<V>(t.a, t.b, phase, t.av, t.bv);
  t.e0 = t.av + k * p.tile_elems;
  t.e1 = t.e0 + p.tile_elems < t.bv ? t.e0 + p.tile_elems : t.bv;
  t.first = (k == 0);
  return t;
}

// ---------------------------------------------------------------------------
// Realigning vector kernel for inputs whose 16-byte phases differ from the
// outputs': the vector grid follows the outputs (realign_range), and input
// u's four elements at a grid position are bytes [s_u, s_u + 16) of the two
// aligned 16-byte blocks around them (s_u = the input's offset from the grid
// mod 16; one block when 0).
// Both blocks hold bytes of the input, so no load leaves its pages.  (Taking
// the second block from the next lane by a shuffle was slower.)  Same folds
// as vc_reduce_vec_any and vc_reduce_elem (left fold from rank (j+1) mod W,
// or rank 0), hence the same bits as the element-wise kernel.
template <typename T, class Op, int KIND>
__global__ void __launch_bounds__(256) vc_reduce_realign(const __grid_constant__ ReduceParams p) {
  pdl_enter();
  using E = Elem<T>;
  constexpr int V = E::kVec;
  constexpr int U = 2;
  constexpr int G = 2;  // ranks per round trip: measured best (1, 2, 4, 8 tried)
  const int W = p.W;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const TileRange tr = realign_range<V, KIND>(p, tile);
    const int start = p.ring ? p.ring_start[tr.j] : 0;
    const int oph = p.out_phase[tr.j];
    int64_t e[U];
    bool ok[U];
    float acc[U][V];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      e[u] = tr.e0 + ((int64_t)u * nthr + tid) * V;
      ok[u] = e[u] < tr.e1;
    }
    for (int t0 = 0; t0 < W; t0 += G) {
      uint4 lo[U][G], hi[U][G];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < G; ++i)
          if (ok[u] && t0 + i < W) {
            const int src = rotate(start, t0 + i, W);
            const int sh = (p.in_phase[src] - oph) & 15;
            const char* a = (const char*)p.in[src] + e[u] * E::kBytes - sh;
            lo[u][i] = ld_stream(a);
            hi[u][i] = sh ? ld_stream(a + 16) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < G; ++i) {
          reg_fence(lo[u][i]);
          reg_fence(hi[u][i]);
        }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
          if (ok[u] && t0 + i < W) {
            const int sh = (p.in_phase[rotate(start, t0 + i, W)] - oph) & 15;
            float x[V];
            E::widen(sh ? funnel16(lo[u][i], hi[u][i], sh) : lo[u][i], x);
            if (t0 + i == 0) {
#pragma unroll
              for (int q = 0; q < V; ++q) acc[u][q] = x[q];
            } else {
#pragma unroll
              for (int q = 0; q < V; ++q) acc[u][q] = Op::apply(acc[u][q], x[q]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ok[u]) {
        if (p.do_scale) {
#pragma unroll
          for (int q = 0; q < V; ++q) acc[u][q] = __fmul_rn(acc[u][q], p.scale);
        }
        const uint4 o = E::narrow(acc[u]);
        if (KIND == KIND_AR) {
          for (int r = 0; r < W; ++r) st_stream((char*)p.out[r] + e[u] * E::kBytes, o);
        } else {
          st_stream((char*)p.out[tr.j] + (e[u] - tr.a) * E::kBytes, o);
        }
      }
    }
    if (tr.first) head_tail<T, Op, KIND, 0>(p, tr, W, start);
  }
}

// The same for a compile-time rank count WT in 2..8 (shifts from the 8 x 8
// table p.wshift): every rank's blocks of a vector are loaded before the
// fold.
template <typename T, int WT, class Op, int KIND, int RING>
__global__ void __launch_bounds__(256, 3) vc_reduce_realign_w(const __grid_constant__ ReduceParams p) {
  pdl_enter();
  using E = Elem<T>;
  constexpr int V = E::kVec;
  // the fast order is the pairwise tree for the rank counts the plain vector
  // kernels compile (2, 4, 8), the left fold from rank 0 otherwise -- the
  // orders of vc_reduce_vec and vc_reduce_vec_any / the multi-tensor kernel
  constexpr bool TREE = !RING && (WT == 2 || WT == 4 || WT == 8);
  constexpr int TREE_W = TREE ? WT : 0;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const TileRange tr = realign_range<V, KIND>(p, tile);
    const int start = RING ? p.ring_start[tr.j] : 0;
    const uint8_t* shift = p.wshift + tr.j * 8;  // input u's bytes past the grid
    for (int64_t e = tr.e0 + (int64_t)tid * V; e < tr.e1; e += (int64_t)nthr * V) {
      uint4 lo[WT], hi[WT];
#pragma unroll
      for (int t = 0; t < WT; ++t) {
        const int src = RING ? rotate(start, t, WT) : t;
        const int sh = shift[src];
        const char* a = (const char*)p.in[src] + e * E::kBytes - sh;
        lo[t] = ld_stream(a);
        hi[t] = sh ? ld_stream(a + 16) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int t = 0; t < WT; ++t) {
        reg_fence(lo[t]);
        reg_fence(hi[t]);
      }
#pragma unroll
      for (int t = 0; t < WT; ++t) {
        const int sh = shift[RING ? rotate(start, t, WT) : t];
        if (sh) lo[t] = funnel16(lo[t], hi[t], sh);
      }
      float acc[V];
      if (RING || !TREE)
        left_fold<T, Op, WT>(lo, acc);
      else
        TreeFold<T, Op, WT, 0, WT>::run(lo, acc);
      if (p.do_scale) {
#pragma unroll
        for (int x = 0; x < V; ++x) acc[x] = __fmul_rn(acc[x], p.scale);
      }
      const uint4 o = E::narrow(acc);
      if (KIND == KIND_AR) {
#pragma unroll
        for (int r = 0; r < WT; ++r) st_stream((char*)p.out[r] + e * E::kBytes, o);
      } else {
        st_stream((char*)p.out[tr.j] + (e - tr.a) * E::kBytes, o);
      }
    }
    if (tr.first) head_tail<T, Op, KIND, TREE_W>(p, tr, WT, start);
  }
}

// ---------------------------------------------------------------------------
// Element-wise kernel for buffers whose 16-byte phases differ: the same
// folds, one element per thread per step (phase is ignored; V = 1).
template <typename T, class Op, int KIND>
__global__ void __launch_bounds__(256) vc_reduce_elem(const __grid_constant__ ReduceParams p) {
  pdl_enter();
  const int W = p.W;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const TileRange tr = tile_range<1>(p, tile);
    const int start = p.ring ? p.ring_start[tr.j] : 0;
#pragma unroll 4
    for (int64_t e = tr.e0 + tid; e < tr.e1; e += nthr)
      reduce_one<T, Op, KIND, 0>(p, W, start, tr.j, tr.a, e);
  }
}

}  // namespace vcoll

// Instantiation table for one element type (used by reduce_f32.cu and
// reduce_bf16.cu).  Index: [op][kind][wslot][ring][vec]; wslot 0..4 for
// W_t = 0, 2, 4, 8, 16.
#define VCOLL_DEFINE_REDUCE_TABLE(T, FNAME)                                                   \
  namespace vcoll {                                                                           \
  namespace {                                                                                 \
  template <class Op, int KIND>                                                               \
  const void* pick(int W_t, int ring, int vec) {                                              \
    if (!vec) return (const void*)&vc_reduce_elem<T, Op, KIND>;                               \
    switch (W_t) {                                                                            \
      case 2:                                                                                 \
        return (const void*)&vc_reduce_vec<T, 2, Op, KIND, 0>;                                \
      case 4:                                                                                 \
        return ring ? (const void*)&vc_reduce_vec<T, 4, Op, KIND, 1>                          \
                    : (const void*)&vc_reduce_vec<T, 4, Op, KIND, 0>;                         \
      case 8:                                                                                 \
        return ring ? (const void*)&vc_reduce_vec<T, 8, Op, KIND, 1>                          \
                    : (const void*)&vc_reduce_vec<T, 8, Op, KIND, 0>;                         \
      case 16:                                                                                \
        return ring ? (const void*)&vc_reduce_vec<T, 16, Op, KIND, 1>                         \
                    : (const void*)&vc_reduce_vec<T, 16, Op, KIND, 0>;                        \
      default:                                                                                \
        return (const void*)&vc_reduce_vec_any<T, Op, KIND>;                                  \
    }                                                                                         \
  }                                                                                           \
  /* max and min are order-independent: one (tree) instantiation, any order */                 \
  template <class Op, int KIND>                                                                         \
  const void* pick_max(int W_t, int vec) {                                                    \
    if (!vec) return (const void*)&vc_reduce_elem<T, Op, KIND>;                            \
    switch (W_t) {                                                                            \
      case 2:                                                                                 \
        return (const void*)&vc_reduce_vec<T, 2, Op, KIND, 0>;                             \
      case 4:                                                                                 \
        return (const void*)&vc_reduce_vec<T, 4, Op, KIND, 0>;                             \
      case 8:                                                                                 \
        return (const void*)&vc_reduce_vec<T, 8, Op, KIND, 0>;                             \
      case 16:                                                                                \
        return (const void*)&vc_reduce_vec<T, 16, Op, KIND, 0>;                            \
      default:                                                                                \
        return (const void*)&vc_reduce_vec_any<T, Op, KIND>;                               \
    }                                                                                         \
  }                                                                                           \
  }                                                                                           \
  template <class Op, int KIND>                                                               \
  const void* FNAME##_pick_realign(int W, int ring) {                                         \
    switch (W) {                                                                              \
      case 2: return (const void*)&vc_reduce_realign_w<T, 2, Op, KIND, 0>;                    \
      case 3: return ring ? (const void*)&vc_reduce_realign_w<T, 3, Op, KIND, 1>              \
                          : (const void*)&vc_reduce_realign_w<T, 3, Op, KIND, 0>;             \
      case 4: return ring ? (const void*)&vc_reduce_realign_w<T, 4, Op, KIND, 1>              \
                          : (const void*)&vc_reduce_realign_w<T, 4, Op, KIND, 0>;             \
      case 5: return ring ? (const void*)&vc_reduce_realign_w<T, 5, Op, KIND, 1>              \
                          : (const void*)&vc_reduce_realign_w<T, 5, Op, KIND, 0>;             \
      case 6: return ring ? (const void*)&vc_reduce_realign_w<T, 6, Op, KIND, 1>              \
                          : (const void*)&vc_reduce_realign_w<T, 6, Op, KIND, 0>;             \
      case 7: return ring ? (const void*)&vc_reduce_realign_w<T, 7, Op, KIND, 1>              \
                          : (const void*)&vc_reduce_realign_w<T, 7, Op, KIND, 0>;             \
      case 8: return ring ? (const void*)&vc_reduce_realign_w<T, 8, Op, KIND, 1>              \
                          : (const void*)&vc_reduce_realign_w<T, 8, Op, KIND, 0>;             \
      default: return (const void*)&vc_reduce_realign<T, Op, KIND>;                           \
    }                                                                                         \
  }                                                                                           \
  /* inputs at other phases than the outputs; W = the rank count (2..8 compiled in) */       \
  const void* FNAME##_realign(int op, int kind, int W, int ring)   {                          \
    if (op == VCOLL_MAX)                                                                      \
      return kind == KIND_AR ? FNAME##_pick_realign<OpMax, KIND_AR>(W, 0)                     \
                             : FNAME##_pick_realign<OpMax, KIND_RS>(W, 0)  ;                  \
    if (op == VCOLL_MIN)                                                                      \
      return kind == KIND_AR ? FNAME##_pick_realign<OpMin, KIND_AR>(W, 0)                     \
                             : FNAME##_pick_realign<OpMin, KIND_RS>(W, 0)  ;                  \
    if (op == VCOLL_PROD)                                                                     \
      return kind == KIND_AR ? FNAME##_pick_realign<OpProd, KIND_AR>(W, ring)                 \
                             : FNAME##_pick_realign<OpProd, KIND_RS>(W, ring)  ;              \
    return kind == KIND_AR ? FNAME##_pick_realign<OpSum, KIND_AR>(W, ring)                    \
                           : FNAME##_pick_realign<OpSum, KIND_RS>(W, ring)  ;                 \
  }                                                                                           \
  const void* FNAME(int op, int kind, int W_t, int ring, int vec) {                           \
    if (op == VCOLL_MAX)                                                                      \
      return kind == KIND_AR ? pick_max<OpMax, KIND_AR>(W_t, vec)                             \
                             : pick_max<OpMax, KIND_RS>(W_t, vec);                            \
    if (op == VCOLL_MIN)                                                                      \
      return kind == KIND_AR ? pick_max<OpMin, KIND_AR>(W_t, vec)                             \
                             : pick_max<OpMin, KIND_RS>(W_t, vec);                            \
    if (op == VCOLL_PROD)                                                                     \
      return kind == KIND_AR ? pick<OpProd, KIND_AR>(W_t, ring, vec)                          \
                             : pick<OpProd, KIND_RS>(W_t, ring, vec);                         \
    return kind == KIND_AR ? pick<OpSum, KIND_AR>(W_t, ring, vec)                             \
                           : pick<OpSum, KIND_RS>(W_t, ring, vec);                            \
  }                                                                                           \
  }

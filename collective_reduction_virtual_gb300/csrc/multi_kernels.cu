// Multi-tensor allreduce: Horovod's tensor fusion (PerformOperation: pack
// every tensor into the fusion buffer, allreduce it in place, unpack) without
// the fusion buffer.  Each thread reads the W ranks' values of a tensor
// straight from the tensors and writes the result straight into the output
// tensors, so the batch moves 2 * W * B bytes instead of the 6 * W * B of the
// three-pass pipeline.  The fold treats the T tensors of a rank as one
// virtual buffer segmented exactly as the fused buffer would be, so the bits
// equal pack -> allreduce -> unpack in ring order and in the fastest order.
#include "device_common.cuh"
#include "reduce_kernels.cuh"
#include "vcoll_internal.h"

namespace vcoll {

namespace {

// Pointer tables are tensor-major: the W pointers a tile needs are adjacent.
__device__ __forceinline__ const char* in_ptr(const MultiParams& p, int rank, int t) {
  return (const char*)p.in[t * p.W + rank];
}
__device__ __forceinline__ char* out_ptr(const MultiParams& p, int rank, int t) {
  return (char*)p.out[t * p.W + rank];
}

// Pairwise tree over ranks [LO, LO + CNT) for one element (matches TreeFold).
template <typename T, class Op, int LO, int CNT>
struct MultiTree {
  static __device__ __forceinline__ float run(const MultiParams& p, int t, int64_t off) {
    const float a = MultiTree<T, Op, LO, CNT / 2>::run(p, t, off);
    const float b = MultiTree<T, Op, LO + CNT / 2, CNT - CNT / 2>::run(p, t, off);
    return Op::apply(a, b);
  }
};
template <typename T, class Op, int LO>
struct MultiTree<T, Op, LO, 1> {
  static __device__ __forceinline__ float run(const MultiParams& p, int t, int64_t off) {
    using B = typename Elem<T>::Bits;
    return Elem<T>::widen1(ld1<B>(in_ptr(p, LO, t) + off));
  }
};

// One element k of tensor t: the tree for a compile-time W in the fastest
// order, otherwise the left fold from rank `start`.
template <typename T, class Op, int WT, int RING>
__device__ __forceinline__ void multi_one(const MultiParams& p, int W, int t, int start,
                                          int64_t k) {
  using E = Elem<T>;
  using B = typename E::Bits;
  const int64_t off = k * E::kBytes;
  float acc;
  if (!RING && WT > 0) {
    acc = MultiTree<T, Op, 0, (WT > 0 ? WT : 1)>::run(p, t, off);
  } else {
    acc = E::widen1(ld1<B>(in_ptr(p, start, t) + off));
#pragma unroll 4
    for (int i = 1; i < W; ++i)
      acc = Op::apply(acc, E::widen1(ld1<B>(in_ptr(p, rotate(start, i, W), t) + off)));
  }
  if (p.do_scale) acc = __fmul_rn(acc, p.scale);
  const B o = E::narrow1(acc);
  for (int u = 0; u < W; ++u) st1(out_ptr(p, u, t) + off, o);
}

}  // namespace

template <typename T, int WT, class Op, int RING>
__global__ void __launch_bounds__(256, 2) vc_allreduce_multi(const __grid_constant__ MultiParams p) {
  pdl_enter();
  using E = Elem<T>;
  constexpr int V = E::kVec;
  constexpr int U = unroll_for(WT);
  constexpr int WR = WT > 0 ? WT : 1;  // register array extent for the compile-time path
  const int W = WT > 0 ? WT : p.W;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  // the piece table moves to shared memory once, so that finding a tile's
  // piece is a short search in shared memory rather than a chain of
  // dependent parameter-space loads
  __shared__ MultiPiece s_piece[kMultiMaxPieces];
  for (int i = tid; i < p.npieces; i += nthr) s_piece[i] = p.piece[i];
  __syncthreads();
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    int lo = 0, hi = p.npieces - 1;  // last piece with tile_begin <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_piece[mid].tile_begin <= tile)
        lo = mid;
      else
        hi = mid - 1;
    }
    const MultiPiece pc = s_piece[lo];
    const int64_t k = tile - pc.tile_begin;
    const int t = pc.t;
    const int start = RING ? pc.start : 0;
    if (pc.phase < 0) {
      // buffers at different 16-byte phases: element-wise
      const int64_t e0 = k * p.tile_elems;
      const int64_t e1 = e0 + p.tile_elems < pc.len ? e0 + p.tile_elems : pc.len;
      for (int64_t e = e0 + tid; e < e1; e += nthr)
        multi_one<T, Op, WT, RING>(p, W, t, start, pc.k0 + e);
      continue;
    }
    int64_t av, bv;
    aligned_body<V>(0, pc.len, pc.phase, av, bv);
    const int64_t e0 = av + k * p.tile_elems;
    const int64_t e1 = e0 + p.tile_elems < bv ? e0 + p.tile_elems : bv;
    if (WT > 0) {
      uint4 v[U][WR];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = e0 + ((int64_t)u * nthr + tid) * V;
        if (e < e1) {
#pragma unroll
          for (int r = 0; r < WR; ++r) {
            const int src = RING ? rotate(start, r, WR) : r;
            v[u][r] = ld_stream(in_ptr(p, src, t) + (pc.k0 + e) * E::kBytes);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < WR; ++r) reg_fence(v[u][r]);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = e0 + ((int64_t)u * nthr + tid) * V;
        if (e < e1) {
          float acc[V];
          if (RING)
            left_fold<T, Op, WR>(v[u], acc);
          else
            TreeFold<T, Op, WR, 0, WR>::run(v[u], acc);
          if (p.do_scale) {
#pragma unroll
            for (int x = 0; x < V; ++x) acc[x] = __fmul_rn(acc[x], p.scale);
          }
          const uint4 o = E::narrow(acc);
#pragma unroll
          for (int r = 0; r < WR; ++r) st_stream(out_ptr(p, r, t) + (pc.k0 + e) * E::kBytes, o);
        }
      }
    } else {
      for (int64_t e = e0 + (int64_t)tid * V; e < e1; e += (int64_t)nthr * V) {
        float acc[V];
        E::widen(ld_stream(in_ptr(p, start, t) + (pc.k0 + e) * E::kBytes), acc);
        for (int i = 1; i < W; ++i) {
          float x[V];
          E::widen(ld_stream(in_ptr(p, rotate(start, i, W), t) + (pc.k0 + e) * E::kBytes), x);
#pragma unroll
          for (int q = 0; q < V; ++q) acc[q] = Op::apply(acc[q], x[q]);
        }
        if (p.do_scale) {
#pragma unroll
          for (int q = 0; q < V; ++q) acc[q] = __fmul_rn(acc[q], p.scale);
        }
        const uint4 o = E::narrow(acc);
        for (int r = 0; r < W; ++r) st_stream(out_ptr(p, r, t) + (pc.k0 + e) * E::kBytes, o);
      }
    }
    if (k == 0) {
      // unaligned head [0, av) and tail [bv, len) of the piece, < V elements each
      int64_t i = -1;
      if (tid < av) i = tid;
      if (tid >= 32 && tid - 32 < pc.len - bv) i = bv + (tid - 32);
      if (i >= 0) multi_one<T, Op, WT, RING>(p, W, t, start, pc.k0 + i);
    }
  }
}

namespace {
template <typename T, class Op>
const void* pick_multi(int W_t, int ring) {
  switch (W_t) {
    case 2:
      return (const void*)&vc_allreduce_multi<T, 2, Op, 0>;
    case 4:
      return ring ? (const void*)&vc_allreduce_multi<T, 4, Op, 1>
                  : (const void*)&vc_allreduce_multi<T, 4, Op, 0>;
    case 8:
      return ring ? (const void*)&vc_allreduce_multi<T, 8, Op, 1>
                  : (const void*)&vc_allreduce_multi<T, 8, Op, 0>;
    case 16:
      return ring ? (const void*)&vc_allreduce_multi<T, 16, Op, 1>
                  : (const void*)&vc_allreduce_multi<T, 16, Op, 0>;
    default:
      return ring ? (const void*)&vc_allreduce_multi<T, 0, Op, 1>
                  : (const void*)&vc_allreduce_multi<T, 0, Op, 0>;
  }
}
template <typename T>
const void* multi_table(int op, int W_t, int ring) {
  if (op == VCOLL_MAX) return pick_multi<T, OpMax>(W_t, 0);
  if (op == VCOLL_MIN) return pick_multi<T, OpMin>(W_t, 0);
  if (op == VCOLL_PROD) return pick_multi<T, OpProd>(W_t, ring);
  return pick_multi<T, OpSum>(W_t, ring);
}
}  // namespace

const void* multi_kernel_f32(int op, int W_t, int ring) { return multi_table<float>(op, W_t, ring); }
const void* multi_kernel_bf16(int op, int W_t, int ring) {
  return multi_table<__nv_bfloat16>(op, W_t, ring);
}

}  // namespace vcoll

// Reduced-precision "wire" allreduce (Apache SINGA Communicator::synchHalf /
// fusedSynchHalf): fp32 inputs are converted to a 16-bit wire type
// (float2half), allreduced in that type and converted back (half2float).
// In the NCCL ring the intermediate buffers hold the wire type, so every hop
// rounds to it; here each thread reads the W fp32 inputs at its indices,
// rounds each to the wire type, folds with a rounding after every
// application of the op (ring order, or a pairwise tree), and writes the
// widened result to the W fp32 outputs -- one pass, no wire buffers, the
// bits of convert -> ring allreduce in the wire type -> convert.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "reduce_kernels.cuh"
#include "vcoll_internal.h"

namespace vcoll {

namespace {

// v rounded to the wire type (round to nearest even) and widened back (exact)
template <int WIRE>
__device__ __forceinline__ float wround(float v) {
  if (WIRE == VCOLL_F16) return __half2float(__float2half_rn(v));
  return __bfloat162float(__float2bfloat16_rn(v));
}

template <class Op, int WIRE>
struct WireOp {
  static __device__ __forceinline__ float apply(float acc, float x) {
    return wround<WIRE>(Op::apply(acc, x));
  }
};

// x[t][e]: rank t's value (already in the wire type), tree over [LO, LO+CNT)
template <class Op, int WIRE, int WT, int LO, int CNT>
struct WireTree {
  static __device__ __forceinline__ void run(const float (&x)[WT][4], float (&out)[4]) {
    float a[4], b[4];
    WireTree<Op, WIRE, WT, LO, CNT / 2>::run(x, a);
    WireTree<Op, WIRE, WT, LO + CNT / 2, CNT - CNT / 2>::run(x, b);
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = WireOp<Op, WIRE>::apply(a[e], b[e]);
  }
};
template <class Op, int WIRE, int WT, int LO>
struct WireTree<Op, WIRE, WT, LO, 1> {
  static __device__ __forceinline__ void run(const float (&x)[WT][4], float (&out)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = x[LO][e];
  }
};

template <class Op, int WIRE, int LO, int CNT>
struct WireTreeScalar {
  static __device__ __forceinline__ float run(const ReduceParams& p, int64_t off) {
    const float a = WireTreeScalar<Op, WIRE, LO, CNT / 2>::run(p, off);
    const float b = WireTreeScalar<Op, WIRE, LO + CNT / 2, CNT - CNT / 2>::run(p, off);
    return WireOp<Op, WIRE>::apply(a, b);
  }
};
template <class Op, int WIRE, int LO>
struct WireTreeScalar<Op, WIRE, LO, 1> {
  static __device__ __forceinline__ float run(const ReduceParams& p, int64_t off) {
    return wround<WIRE>(__uint_as_float(ld1<uint32_t>((const char*)p.in[LO] + off)));
  }
};

// one element i: tree for a compile-time W in the fastest order, otherwise
// the left fold from rank `start`; then avg's scale (rounded) and W stores
template <class Op, int WIRE, int WT, int RING>
__device__ __forceinline__ void wire_one(const ReduceParams& p, int W, int start, int64_t i) {
  const int64_t off = i * 4;
  float acc;
  if (!RING && WT > 0) {
    acc = WireTreeScalar<Op, WIRE, 0, (WT > 0 ? WT : 1)>::run(p, off);
  } else {
    acc = wround<WIRE>(__uint_as_float(ld1<uint32_t>((const char*)p.in[start] + off)));
    for (int t = 1; t < W; ++t) {
      const float x =
          wround<WIRE>(__uint_as_float(ld1<uint32_t>((const char*)p.in[rotate(start, t, W)] + off)));
      acc = WireOp<Op, WIRE>::apply(acc, x);
    }
  }
  if (p.do_scale) acc = wround<WIRE>(__fmul_rn(acc, p.scale));
  const uint32_t o = __float_as_uint(acc);
  for (int u = 0; u < W; ++u) st1((char*)p.out[u] + off, o);
}

}  // namespace

template <int WIRE, int WT, class Op, int RING>
__global__ void __launch_bounds__(256) vc_allreduce_wire(const __grid_constant__ ReduceParams p) {
  pdl_enter();
  constexpr int V = 4;  // fp32 lanes per 16-byte vector
  constexpr int WR = WT > 0 ? WT : 1;
  const int W = WT > 0 ? WT : p.W;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const TileRange tr = tile_range<V>(p, tile);
    const int start = RING ? p.ring_start[tr.j] : 0;
    if (p.phase < 0) {  // buffers at different 16-byte phases: element-wise
      for (int64_t e = tr.a + (tile - (int64_t)tr.j * p.tiles_per_seg) * p.tile_elems + tid;
           e < tr.b && e < tr.a + (tile - (int64_t)tr.j * p.tiles_per_seg + 1) * p.tile_elems;
           e += nthr)
        wire_one<Op, WIRE, WT, RING>(p, W, start, e);
      continue;
    }
    for (int64_t e = tr.e0 + (int64_t)tid * V; e < tr.e1; e += (int64_t)nthr * V) {
      float acc[V];
      if (WT > 0) {
        uint4 v[WR];
#pragma unroll
        for (int t = 0; t < WR; ++t) {
          const int src = RING ? rotate(start, t, WR) : t;
          v[t] = ld_stream((const char*)p.in[src] + e * 4);
        }
#pragma unroll
        for (int t = 0; t < WR; ++t) reg_fence(v[t]);
        float x[WR][4];
#pragma unroll
        for (int t = 0; t < WR; ++t) {
          x[t][0] = wround<WIRE>(__uint_as_float(v[t].x));
          x[t][1] = wround<WIRE>(__uint_as_float(v[t].y));
          x[t][2] = wround<WIRE>(__uint_as_float(v[t].z));
          x[t][3] = wround<WIRE>(__uint_as_float(v[t].w));
        }
        if (RING) {
#pragma unroll
          for (int q = 0; q < V; ++q) acc[q] = x[0][q];
#pragma unroll
          for (int t = 1; t < WR; ++t)
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = WireOp<Op, WIRE>::apply(acc[q], x[t][q]);
        } else {
          WireTree<Op, WIRE, WR, 0, WR>::run(x, acc);
        }
      } else {
        for (int t = 0; t < W; ++t) {
          const uint4 v = ld_stream((const char*)p.in[rotate(start, t, W)] + e * 4);
          const float x[4] = {wround<WIRE>(__uint_as_float(v.x)), wround<WIRE>(__uint_as_float(v.y)),
                              wround<WIRE>(__uint_as_float(v.z)), wround<WIRE>(__uint_as_float(v.w))};
#pragma unroll
          for (int q = 0; q < V; ++q) acc[q] = t == 0 ? x[q] : WireOp<Op, WIRE>::apply(acc[q], x[q]);
        }
      }
      if (p.do_scale) {
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = wround<WIRE>(__fmul_rn(acc[q], p.scale));
      }
      const uint4 o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                                 __float_as_uint(acc[2]), __float_as_uint(acc[3]));
      for (int r = 0; r < W; ++r) st_stream((char*)p.out[r] + e * 4, o);
    }
    if (tr.first) {
      const int64_t nh = tr.av - tr.a, nt = tr.b - tr.bv;
      if (tid < nh) wire_one<Op, WIRE, WT, RING>(p, W, start, tr.a + tid);
      const int k = tid - 32;
      if (k >= 0 && k < nt) wire_one<Op, WIRE, WT, RING>(p, W, start, tr.bv + k);
    }
  }
}

namespace {
template <int WIRE>
const void* pick_wire(int W_t, int ring) {
  switch (W_t) {
    case 2:
      return (const void*)&vc_allreduce_wire<WIRE, 2, OpSum, 0>;
    case 4:
      return ring ? (const void*)&vc_allreduce_wire<WIRE, 4, OpSum, 1>
                  : (const void*)&vc_allreduce_wire<WIRE, 4, OpSum, 0>;
    case 8:
      return ring ? (const void*)&vc_allreduce_wire<WIRE, 8, OpSum, 1>
                  : (const void*)&vc_allreduce_wire<WIRE, 8, OpSum, 0>;
    case 16:
      return ring ? (const void*)&vc_allreduce_wire<WIRE, 16, OpSum, 1>
                  : (const void*)&vc_allreduce_wire<WIRE, 16, OpSum, 0>;
    default:
      return ring ? (const void*)&vc_allreduce_wire<WIRE, 0, OpSum, 1>
                  : (const void*)&vc_allreduce_wire<WIRE, 0, OpSum, 0>;
  }
}
}  // namespace

const void* wire_kernel(int wire, int W_t, int ring) {
  return wire == VCOLL_F16 ? pick_wire<VCOLL_F16>(W_t, ring) : pick_wire<VCOLL_BF16>(W_t, ring);
}

}  // namespace vcoll

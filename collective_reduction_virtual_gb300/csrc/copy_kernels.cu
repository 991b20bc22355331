// Bit-copy kernels: allgather and tensor-fusion pack / unpack.
//
// Allgather ("Distributed primitives": AllGather propagates the reduced
// segments so that every node holds their concatenation): each tile reads a
// piece of segment j once and writes it to all W outputs.
//
// Fusion (Horovod PerformOperation: copy each tensor to buffer + offset with
// offset += size, no padding; SINGA Communicator::fusedSynch likewise): one
// launch moves up to kFuseMaxTensors tensors of every rank.  Tensor offsets
// in the fused buffer are arbitrary element multiples, so source and
// destination usually sit at different 16-byte phases; the copy then stores
// aligned 16-byte vectors and assembles each from the two aligned source
// vectors that cover it (a funnel shift), keeping both sides at full width.
#include "device_common.cuh"
#include "vcoll_internal.h"

namespace vcoll {

// ------------------------------------------------------------- allgather

// VM: 0 element-wise, 1 16-byte vectors, 2 vectors with pieces realigned to
// the outputs' grid
template <int ES, int VM>
__global__ void __launch_bounds__(256) vc_gather(const __grid_constant__ GatherParams p) {
  pdl_enter();
  constexpr bool VEC = VM >= 1;
  using B = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
  constexpr int V = VEC ? 16 / ES : 1;
  constexpr int U = 4;
  const int W = p.W;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const int j = (int)(tile / p.tiles_per_seg);
    const int64_t k = tile - (int64_t)j * p.tiles_per_seg;
    int64_t a, b, av, bv;
    a = p.disp[j];
    b = p.disp[j + 1];
    if (VEC) {
      aligned_body<V>(a, b, p.phase, av, bv);
    } else {
      av = a;
      bv = b;
    }
    const int64_t e0 = av + k * p.tile_elems;
    const int64_t e1 = e0 + p.tile_elems < bv ? e0 + p.tile_elems : bv;
    const char* src = (const char*)p.in[j] - a * ES;  // element i of segment j at src + i*ES
    if (VEC) {
      // the vectors follow the outputs' grid; a piece at another phase is
      // read as the two aligned blocks around each vector and funnel-shifted
      // (both blocks hold bytes of the piece)
      const int sh = VM == 2 ? p.ishift[j] : 0;
      uint4 v[U], hi[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = e0 + ((int64_t)u * nthr + tid) * V;
        hi[u] = make_uint4(0u, 0u, 0u, 0u);
        if (e < e1) {
          v[u] = ld_stream(src + e * ES - sh);
          if (sh) hi[u] = ld_stream(src + e * ES - sh + 16);
        }
      }
      if (sh) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          reg_fence(v[u]);
          reg_fence(hi[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = funnel16(v[u], hi[u], sh);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t e = e0 + ((int64_t)u * nthr + tid) * V;
        if (e < e1)
          for (int r = 0; r < W; ++r) st_stream((char*)p.out[r] + e * ES, v[u]);
      }
      if (k == 0) {
        // head [a, av) and tail [bv, b): fewer than V elements each
        int64_t i = -1;
        if (tid < av - a) i = a + tid;
        if (tid >= 32 && tid - 32 < b - bv) i = bv + (tid - 32);
        if (i >= 0) {
          const B x = ld1<B>(src + i * ES);
          for (int r = 0; r < W; ++r) st1((char*)p.out[r] + i * ES, x);
        }
      }
    } else {
      for (int64_t e = e0 + tid; e < e1; e += nthr) {
        const B x = ld1<B>(src + e * ES);
        for (int r = 0; r < W; ++r) st1((char*)p.out[r] + e * ES, x);
      }
    }
  }
}

// ------------------------------------------------------------------ fusion


// Block-cooperative copy of nbytes (a multiple of ES) from src to dst, both
// ES-aligned.  Destination-aligned 16-byte stores; the body loads either one
// aligned source vector (same phase) or the two aligned vectors covering the
// shifted source bytes.  Both of those lie in 16-byte blocks that hold at
// least one byte of the source range, so no access leaves the source's pages.
template <int ES>
__device__ __forceinline__ void copy_range(char* dst, const char* src, int64_t nbytes) {
  using B = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
  constexpr int U = 4;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const uint64_t d0 = (uint64_t)dst;
  int64_t head = (int64_t)((16 - (d0 & 15)) & 15);
  if (head > nbytes) head = nbytes;
  const int64_t body = (nbytes - head) & ~(int64_t)15;
  const int64_t tail0 = head + body;
  // head and tail, one element per thread
  {
    int64_t off = -1;
    if ((int64_t)tid * ES < head) off = (int64_t)tid * ES;
    const int t2 = tid - 32;
    if (t2 >= 0 && tail0 + (int64_t)t2 * ES < nbytes) off = tail0 + (int64_t)t2 * ES;
    if (off >= 0) st1(dst + off, ld1<B>(src + off));
  }
  const int64_t nv = body >> 4;
  char* vd = dst + head;
  const char* vs = src + head;
  const int sh = (int)((uint64_t)vs & 15);
  if (sh == 0) {
    for (int64_t base = 0; base < nv; base += (int64_t)U * nthr) {
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = base + (int64_t)u * nthr + tid;
        if (i < nv) x[u] = ld_stream(vs + i * 16);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = base + (int64_t)u * nthr + tid;
        if (i < nv) st_stream(vd + i * 16, x[u]);
      }
    }
  } else {
    const char* as = vs - sh;  // aligned source base
    for (int64_t base = 0; base < nv; base += (int64_t)U * nthr) {
      uint4 lo[U], hi[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = base + (int64_t)u * nthr + tid;
        if (i < nv) {
          lo[u] = ld_stream(as + i * 16);
          hi[u] = ld_stream(as + i * 16 + 16);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = base + (int64_t)u * nthr + tid;
        if (i < nv) st_stream(vd + i * 16, funnel16(lo[u], hi[u], sh));
      }
    }
  }
}

template <int ES>
__global__ void __launch_bounds__(256) vc_fuse(const __grid_constant__ FuseParams p) {
  pdl_enter();
  // tile table in shared memory: the per-tile search stays on chip
  __shared__ int64_t s_begin[kFuseMaxTensors + 1];
  for (int i = threadIdx.x; i <= p.T; i += blockDim.x) s_begin[i] = p.tile_begin[i];
  __syncthreads();
  const int64_t total = s_begin[p.T];
  for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    // tensor t with tile_begin[t] <= tile < tile_begin[t + 1]
    int lo = 0, hi = p.T - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_begin[mid] <= tile)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int t = lo;
    const int64_t k = tile - s_begin[t];
    const int64_t e0 = k * p.tile_elems;
    const int64_t e1 = e0 + p.tile_elems < p.count[t] ? e0 + p.tile_elems : p.count[t];
    for (int u = 0; u < p.W; ++u) {
      char* tens = (char*)p.tensor[t * p.W + u] + e0 * ES;
      char* fus = (char*)p.fused[u] + (p.offset[t] + e0) * ES;
      if (p.unpack)
        copy_range<ES>(tens, fus, (e1 - e0) * ES);
      else
        copy_range<ES>(fus, tens, (e1 - e0) * ES);
    }
  }
}

// The 16-byte body of one tile for ranks g .. g + G - 1: nv destination
// vectors at dst_of(u) + head, the source sh bytes past a 16-byte boundary.
// Aligned: every thread issues 8 vector loads (8 / G per rank) before its
// first store; shifted: one vector per rank, loaded as the two aligned blocks
// that cover it and funnel-shifted.
template <int G, class DstOf, class SrcOf>
__device__ __forceinline__ void fuse_group_body(DstOf dst_of, SrcOf src_of, int g, int64_t head,
                                                int64_t nv, int sh) {
  const int tid = threadIdx.x;
  const int64_t nthr = blockDim.x;
  if (sh == 0) {
    constexpr int U = 8 / G;
    for (int64_t base = tid; base < nv; base += U * nthr) {
      uint4 x[U][G];
#pragma unroll
      for (int v = 0; v < U; ++v)
#pragma unroll
        for (int q = 0; q < G; ++q)
          if (base + v * nthr < nv) x[v][q] = ld_stream(src_of(g + q) + head + (base + v * nthr) * 16);
#pragma unroll
      for (int v = 0; v < U; ++v)
#pragma unroll
        for (int q = 0; q < G; ++q) reg_fence(x[v][q]);
#pragma unroll
      for (int v = 0; v < U; ++v)
#pragma unroll
        for (int q = 0; q < G; ++q)
          if (base + v * nthr < nv) st_stream(dst_of(g + q) + head + (base + v * nthr) * 16, x[v][q]);
    }
  } else {
    for (int64_t i = tid; i < nv; i += nthr) {
      uint4 a[G], b[G];
#pragma unroll
      for (int q = 0; q < G; ++q) {
        const char* as = src_of(g + q) + head - sh + i * 16;  // aligned source blocks
        a[q] = ld_stream(as);
        b[q] = ld_stream(as + 16);
      }
#pragma unroll
      for (int q = 0; q < G; ++q) {
        reg_fence(a[q]);
        reg_fence(b[q]);
      }
#pragma unroll
      for (int q = 0; q < G; ++q) st_stream(dst_of(g + q) + head + i * 16, funnel16(a[q], b[q], sh));
    }
  }
}

// Pack / unpack with the W ranks' copies of a tile done together, G ranks at
// a time, each thread keeping at least G 16-byte loads in flight before its
// first store, so a tile's copies overlap instead of running rank after
// rank (copy_range, rank by rank, keeps 4).  Needs tensors whose
// copies share their phases on all ranks (the usual case: every buffer
// 256-byte aligned); the others take copy_range rank by rank.
template <int ES, int G>
__global__ void __launch_bounds__(256, 2) vc_fuse_grouped(const __grid_constant__ FuseParams p) {
  pdl_enter();
  using B = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
  __shared__ int64_t s_begin[kFuseMaxTensors + 1];
  for (int i = threadIdx.x; i <= p.T; i += blockDim.x) s_begin[i] = p.tile_begin[i];
  __syncthreads();
  const int64_t total = s_begin[p.T];
  const int W = p.W;
  const int tid = threadIdx.x;
  for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = p.T - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_begin[mid] <= tile)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int t = lo;
    const int64_t k = tile - s_begin[t];
    const int64_t e0 = k * p.tile_elems;
    const int64_t e1 = e0 + p.tile_elems < p.count[t] ? e0 + p.tile_elems : p.count[t];
    const int64_t nbytes = (e1 - e0) * ES;
    const int64_t foff = (p.offset[t] + e0) * ES;
    auto dst_of = [&](int u) -> char* {
      return p.unpack ? (char*)p.tensor[t * W + u] + e0 * ES : (char*)p.fused[u] + foff;
    };
    auto src_of = [&](int u) -> const char* {
      return p.unpack ? (const char*)p.fused[u] + foff : (const char*)p.tensor[t * W + u] + e0 * ES;
    };
    if (!((p.uniform >> t) & 1u)) {
      for (int u = 0; u < W; ++u) copy_range<ES>(dst_of(u), src_of(u), nbytes);
      continue;
    }
    // phases shared by every rank: split the range once
    int64_t head = (int64_t)((16 - ((uint64_t)dst_of(0) & 15)) & 15);
    if (head > nbytes) head = nbytes;
    const int64_t body = (nbytes - head) & ~(int64_t)15;
    const int64_t tail0 = head + body;
    const int sh = (int)(((uint64_t)src_of(0) + head) & 15);
    const int64_t nv = body >> 4;
    {  // head and tail, one element per thread, every rank
      int64_t off = -1;
      if ((int64_t)tid * ES < head) off = (int64_t)tid * ES;
      const int t2 = tid - 32;
      if (t2 >= 0 && tail0 + (int64_t)t2 * ES < nbytes) off = tail0 + (int64_t)t2 * ES;
      if (off >= 0)
        for (int u = 0; u < W; ++u) st1(dst_of(u) + off, ld1<B>(src_of(u) + off));
    }
    for (int g = 0; g < W; g += G) fuse_group_body<G>(dst_of, src_of, g, head, nv, sh);
  }
}

const void* gather_kernel(int elem_size, int vec) {
  if (elem_size == 4)
    return vec == 2 ? (const void*)&vc_gather<4, 2>
                    : vec ? (const void*)&vc_gather<4, 1> : (const void*)&vc_gather<4, 0>;
  return vec == 2 ? (const void*)&vc_gather<2, 2>
                  : vec ? (const void*)&vc_gather<2, 1> : (const void*)&vc_gather<2, 0>;
}

const void* fuse_kernel(int elem_size, int W) {
  // G = min(W, 8) ranks per group for W in {2, 4, 8, 16}; any other W rank by rank
  if (elem_size == 4) {
    switch (W) {
      case 2: return (const void*)&vc_fuse_grouped<4, 2>;
      case 4: return (const void*)&vc_fuse_grouped<4, 4>;
      case 8: case 16: return (const void*)&vc_fuse_grouped<4, 8>;
      default: return (const void*)&vc_fuse<4>;
    }
  }
  switch (W) {
    case 2: return (const void*)&vc_fuse_grouped<2, 2>;
    case 4: return (const void*)&vc_fuse_grouped<2, 4>;
    case 8: case 16: return (const void*)&vc_fuse_grouped<2, 8>;
    default: return (const void*)&vc_fuse<2>;
  }
}

}  // namespace vcoll

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

constexpr int kFuseThreads = 256;  // the pack / unpack launch's CTA size

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

// Bytes [sh, sh + 16) of the 32 bytes lo:hi, sh in 1..15: the word shift
// ws = sh / 4 picks five words with selects (ws is uniform, so the
// predicates are computed once) and a funnel shift moves the remaining
// (sh % 4) bytes -- no branch per shift, so that four vectors in flight stay
// in registers.
__device__ __forceinline__ uint4 shift_window(const uint4& lo, const uint4& hi, int sh) {
  const int ws = sh >> 2, bs = (sh & 3) * 8;
  const bool s0 = ws == 0, s1 = ws == 1, s2 = ws == 2;
  const uint32_t w0 = s0 ? lo.x : s1 ? lo.y : s2 ? lo.z : lo.w;
  const uint32_t w1 = s0 ? lo.y : s1 ? lo.z : s2 ? lo.w : hi.x;
  const uint32_t w2 = s0 ? lo.z : s1 ? lo.w : s2 ? hi.x : hi.y;
  const uint32_t w3 = s0 ? lo.w : s1 ? hi.x : s2 ? hi.y : hi.z;
  const uint32_t w4 = s0 ? hi.x : s1 ? hi.y : s2 ? hi.z : hi.w;
  return make_uint4(__funnelshift_r(w0, w1, bs), __funnelshift_r(w1, w2, bs),
                    __funnelshift_r(w2, w3, bs), __funnelshift_r(w3, w4, bs));
}

// Pack / unpack with one CTA per (tile, rank): grid.y = rank.  Each CTA
// copies one tile of one tensor for one rank -- at most 1024 destination-
// aligned 16-byte vectors, four per thread, all loads in flight before the
// first store; a source at another 16-byte phase is read as the two aligned
// blocks around each vector and funnel-shifted.  Addresses are one base per
// thread plus constant offsets, so the kernel fits 64 registers (4 CTAs per
// SM) where the grouped kernel below keeps 2 CTAs per SM (128 registers).
template <int ES>
__global__ void __launch_bounds__(256, 4) vc_fuse_flat(const __grid_constant__ FuseParams p) {
  pdl_enter();
  using B = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
  constexpr int U = 4;
  __shared__ int64_t s_begin[kFuseMaxTensors + 1];
  for (int i = threadIdx.x; i <= p.T; i += blockDim.x) s_begin[i] = p.tile_begin[i];
  __syncthreads();
  const int64_t total = s_begin[p.T];
  const int u = blockIdx.y;
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
    const int64_t e0 = (tile - s_begin[t]) * p.tile_elems;
    const int64_t e1 = e0 + p.tile_elems < p.count[t] ? e0 + p.tile_elems : p.count[t];
    char* tens = (char*)p.tensor[t * p.W + u] + e0 * ES;
    char* fus = (char*)p.fused[u] + (p.offset[t] + e0) * ES;
    char* dst = p.unpack ? tens : fus;
    const char* src = p.unpack ? fus : tens;
    const int nbytes = (int)((e1 - e0) * ES);
    int head = (int)((16 - ((uint64_t)dst & 15)) & 15);
    if (head > nbytes) head = nbytes;
    const int body = (nbytes - head) & ~15;
    const int tail0 = head + body;
    {  // head and tail, one element per thread
      int off = -1;
      if (tid * ES < head) off = tid * ES;
      if (tid >= 32 && tail0 + (tid - 32) * ES < nbytes) off = tail0 + (tid - 32) * ES;
      if (off >= 0) st1(dst + off, ld1<B>(src + off));
    }
    const int nv = body >> 4;
    char* vd = dst + head + tid * 16;
    const int sh = (int)((uint64_t)(src + head) & 15);
    if (sh == 0) {
      const char* vs = src + head + tid * 16;
      uint4 x[U];
#pragma unroll
      for (int q = 0; q < U; ++q)
        if (tid + q * kFuseThreads < nv) x[q] = ld_stream(vs + q * kFuseThreads * 16);
#pragma unroll
      for (int q = 0; q < U; ++q) reg_fence(x[q]);
#pragma unroll
      for (int q = 0; q < U; ++q)
        if (tid + q * kFuseThreads < nv) st_stream(vd + q * kFuseThreads * 16, x[q]);
    } else {
      const char* as = src + head - sh + tid * 16;  // the aligned block below each vector
      uint4 a4[U], b4[U];
#pragma unroll
      for (int q = 0; q < U; ++q)
        if (tid + q * kFuseThreads < nv) {
          a4[q] = ld_stream(as + q * kFuseThreads * 16);
          b4[q] = ld_stream(as + q * kFuseThreads * 16 + 16);
        }
#pragma unroll
      for (int q = 0; q < U; ++q) {
        reg_fence(a4[q]);
        reg_fence(b4[q]);
      }
#pragma unroll
      for (int q = 0; q < U; ++q)
        if (tid + q * kFuseThreads < nv)
          st_stream(vd + q * kFuseThreads * 16, shift_window(a4[q], b4[q], sh));
    }
  }
}

const void* gather_kernel(int elem_size, int vec) {
  if (elem_size == 4)
    return vec == 2 ? (const void*)&vc_gather<4, 2>
                    : vec ? (const void*)&vc_gather<4, 1> : (const void*)&vc_gather<4, 0>;
  return vec == 2 ? (const void*)&vc_gather<2, 2>
                  : vec ? (const void*)&vc_gather<2, 1> : (const void*)&vc_gather<2, 0>;
}

const void* fuse_flat_kernel(int elem_size) {
  return elem_size == 4 ? (const void*)&vc_fuse_flat<4> : (const void*)&vc_fuse_flat<2>;
}

}  // namespace vcoll

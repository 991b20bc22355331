// Device helpers shared by the vcoll kernels: element traits for fp32 and
// bf16, the reduction functions, streaming 16-byte loads and stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vcoll {

// ------------------------------------------------------------ reduction ops
// FUNC of the ring (NCCL FuncSum / FuncMax): accumulator first.  Arithmetic is
// fp32 with IEEE round-to-nearest and no flush-to-zero (the library is built
// without fast-math; __fadd_rn also keeps the add out of any contraction).
struct OpSum {
  static __device__ __forceinline__ float apply(float acc, float x) { return __fadd_rn(acc, x); }
};

// max: a NaN operand gives the canonical quiet NaN; equal operands give their
// bitwise AND, which is the operand itself unless they are +0 and -0, where it
// is +0.  Commutative and associative, so every fold order gives equal bits.
struct OpMax {
  static __device__ __forceinline__ float apply(float acc, float x) {
    float r = acc > x ? acc : x;
    r = acc == x ? __uint_as_float(__float_as_uint(acc) & __float_as_uint(x)) : r;
    return (acc != acc || x != x) ? __uint_as_float(0x7FC00000u) : r;
  }
};

// min (NCCL FuncMin): the mirror image of OpMax -- canonical quiet NaN,
// otherwise the smaller operand; equal operands give their bitwise OR, which
// is -0 for +0 and -0.  Order-independent like max.
struct OpMin {
  static __device__ __forceinline__ float apply(float acc, float x) {
    float r = acc < x ? acc : x;
    r = acc == x ? __uint_as_float(__float_as_uint(acc) | __float_as_uint(x)) : r;
    return (acc != acc || x != x) ? __uint_as_float(0x7FC00000u) : r;
  }
};

// prod (NCCL FuncProd): one IEEE fp32 multiply, accumulator first.
struct OpProd {
  static __device__ __forceinline__ float apply(float acc, float x) { return __fmul_rn(acc, x); }
};

// ------------------------------------------------------------ element types
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  static constexpr int kVec = 4;  // elements per 16-byte vector
  using Bits = uint32_t;
  static __device__ __forceinline__ void widen(const uint4& v, float (&f)[kVec]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ uint4 narrow(const float (&f)[kVec]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ float widen1(Bits b) { return __uint_as_float(b); }
  static __device__ __forceinline__ Bits narrow1(float f) { return __float_as_uint(f); }
};

// bf16 is the upper half of an fp32 value: widening shifts it up (exact);
// narrowing rounds to nearest even with the CUDA conversion intrinsic, and a
// NaN keeps its sign and top payload bits and is made quiet (the intrinsic
// gives 0x7FFF for every NaN; the canonical fp32 NaN of max and min must
// become 0x7FC0).
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr int kVec = 8;
  using Bits = uint16_t;
  static __device__ __forceinline__ void widen2(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
  }
  static __device__ __forceinline__ uint32_t quiet_nan(float f) {
    return (__float_as_uint(f) >> 16) | 0x0040u;
  }
  static __device__ __forceinline__ uint32_t narrow2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    uint32_t w = *reinterpret_cast<uint32_t*>(&h);
    if (lo != lo) w = (w & 0xFFFF0000u) | quiet_nan(lo);
    if (hi != hi) w = (w & 0x0000FFFFu) | (quiet_nan(hi) << 16);
    return w;
  }
  static __device__ __forceinline__ void widen(const uint4& v, float (&f)[kVec]) {
    widen2(v.x, f[0], f[1]);
    widen2(v.y, f[2], f[3]);
    widen2(v.z, f[4], f[5]);
    widen2(v.w, f[6], f[7]);
  }
  static __device__ __forceinline__ uint4 narrow(const float (&f)[kVec]) {
    return make_uint4(narrow2(f[0], f[1]), narrow2(f[2], f[3]), narrow2(f[4], f[5]),
                      narrow2(f[6], f[7]));
  }
  static __device__ __forceinline__ float widen1(Bits b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  static __device__ __forceinline__ Bits narrow1(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return f != f ? (Bits)quiet_nan(f) : *reinterpret_cast<uint16_t*>(&h);
  }
};

// --------------------------------------------------------- memory accesses
// Inputs are read exactly once and outputs written once: evict-first
// streaming accesses keep them from displacing anything useful in L2.  The
// load is a volatile asm statement so the compiler keeps every load of a tile
// ahead of the first add that consumes one (all W * U loads in flight).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// Programmatic dependent launch (sm_90+): the host launches these kernels
// with programmatic stream serialization, so a kernel may start while the
// previous one in the stream is still finishing.  Before touching memory it
// waits until that kernel has completed and its writes are visible (a no-op
// when launched without the attribute); then it lets the next kernel begin
// launching, whose blocks in turn wait for this one to finish.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Empty volatile statement that claims to rewrite v: placed after a group of
// ld_stream calls it keeps every consumer of v behind the whole group, so the
// compiler cannot interleave adds between the loads.
__device__ __forceinline__ void reg_fence(uint4& v) {
  asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
}

template <typename B>
__device__ __forceinline__ B ld1(const void* p) {
  return __ldcs(reinterpret_cast<const B*>(p));
}
template <typename B>
__device__ __forceinline__ void st1(void* p, B v) {
  __stcs(reinterpret_cast<B*>(p), v);
}

// Segment bounds [a, b) of segment j (nseg == 1: the whole range).
__device__ __forceinline__ void segment_bounds(int64_t n, int64_t q, int64_t r, int nseg, int j,
                                               int64_t& a, int64_t& b) {
  if (nseg == 1) {
    a = 0;
    b = n;
  } else {
    a = (int64_t)j * q + ((int64_t)j < r ? (int64_t)j : r);
    b = a + q + ((int64_t)j < r ? 1 : 0);
  }
}

// Vector-aligned body [av, bv) inside [a, b): element i starts a 16-byte
// vector when (i + phase) % V == 0.  Head [a, av) and tail [bv, b) each hold
// fewer than V elements.
template <int V>
__device__ __forceinline__ void aligned_body(int64_t a, int64_t b, int phase, int64_t& av,
                                             int64_t& bv) {
  const uint64_t m = V - 1;
  int64_t up = a + (int64_t)((V - ((uint64_t)(a + phase) & m)) & m);
  av = up < b ? up : b;
  int64_t dn = b - (int64_t)((uint64_t)(b + phase) & m);
  bv = dn > av ? dn : av;
}

// out = bytes [sh, sh + 16) of the 32 bytes lo:hi (sh in 1..15).
__device__ __forceinline__ uint4 funnel16(const uint4& lo, const uint4& hi, int sh) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const int bs = (sh & 3) * 8;
  uint4 o;
  switch (sh >> 2) {
    case 0:
      o = make_uint4(__funnelshift_r(w[0], w[1], bs), __funnelshift_r(w[1], w[2], bs),
                     __funnelshift_r(w[2], w[3], bs), __funnelshift_r(w[3], w[4], bs));
      break;
    case 1:
      o = make_uint4(__funnelshift_r(w[1], w[2], bs), __funnelshift_r(w[2], w[3], bs),
                     __funnelshift_r(w[3], w[4], bs), __funnelshift_r(w[4], w[5], bs));
      break;
    case 2:
      o = make_uint4(__funnelshift_r(w[2], w[3], bs), __funnelshift_r(w[3], w[4], bs),
                     __funnelshift_r(w[4], w[5], bs), __funnelshift_r(w[5], w[6], bs));
      break;
    default:
      o = make_uint4(__funnelshift_r(w[3], w[4], bs), __funnelshift_r(w[4], w[5], bs),
                     __funnelshift_r(w[5], w[6], bs), __funnelshift_r(w[6], w[7], bs));
      break;
  }
  return o;
}

}  // namespace vcoll

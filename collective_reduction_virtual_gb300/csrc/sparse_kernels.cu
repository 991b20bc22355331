// Sparsified allreduce with error feedback (Apache SINGA, Communicator::
// valSparsAllReduce and topKSparsAllReduce).
//
// On the pages every rank compacts its surviving (index, value) pairs, the
// lists are allgathered, and each rank scatters them into zeros with
// cusparseSaxpyi, rank after rank.  With all W ranks in one GPU's memory the
// same result is one rank-order fold per index over the entries that
// survived, so the kernels never build the lists:
//
//   threshold: one pass -- x = in (+ accumulation); an entry survives when
//     |x| > threshold (and x != 0, as the index array only holds nonzeros);
//     the accumulation becomes x - (survivor ? x : 0); the output is zeros
//     plus the survivors in rank order, written to every rank.
//   top-K: the K entries of each rank with the largest values (ties: lower
//     index first) are found exactly by a radix select on order-preserving
//     32-bit keys -- three histogram passes over 11, 11 and 10 key bits, each
//     followed by a one-CTA-per-rank selection of the digit that holds the
//     K-th largest key; if keys equal to the K-th one straddle the cut,
//     per-tile counts of equal keys and a scan over them find the last equal
//     entry kept in index order -- then the same apply pass as the threshold
//     mode.
//
// Candidate path (when the workspace has room): a 1/16 - 1/128 sample of the data
// gives a band of first digits that should hold the K-th key (for small K
// everything from a wide lower bound up; otherwise also an upper bound, above
// which entries are only counted), one pass over the data appends every
// entry in the band to the rank's candidate list as (key, index), and the
// select passes then read only the list -- three over the key digits and,
// when keys equal to the K-th one straddle the cut (the K largest
// (key, -index) pairs are the K entries kept), one pass that collects up to
// 256 equal keys' indices and ranks them, or for more three passes over the
// bits of the inverted index.  A rank whose list overflowed, or whose band
// misses the K-th key,
// takes the passes over the whole array instead; the choice is made on the
// device.  The candidate pass also stores x = in + acc back into acc, so the
// later passes read one array (without accumulations a separate form of the
// pass, vc_topk_filter_raw, tests the raw input bits; the list route launches
// a form of it without the band's bodies).  With only a lower bound (small K)
// the lists
// hold every kept entry, grouped by tile, and the output is built from them
// (vc_topk_list_out) instead of by the dense apply pass -- unless a rank fell
// back, which the kernels see on the device.  On that route a second pass
// over the sample (its second key digit) narrows the lower bound and sets a
// settled key, 22 bits fine: with accumulations the candidate pass writes
// the residual of every candidate above it at once, so the output pass
// revisits the accumulation only for the kept entries at or below it (and
// when a rank falls back, a restore pass puts x back from the lists before
// the passes over the whole array read it).  With a band the same second
// pass narrows both band bounds to 22 bits when they lie in one first-digit
// bin, so the lists hold about the band's sampled width rather than whole
// quarter-octave bins.
//
// The histograms (W x 2048 counters), the per-rank selection state, the
// per-tile tie counts and list offsets and the candidate lists live in a
// device workspace the caller provides.
#include "device_common.cuh"
#include "vcoll_internal.h"

namespace vcoll {

namespace {

// larger value -> larger key; -0 just below +0; NaNs beyond the infinities.
// The bits go through an opaque move: without it the sign test was compiled,
// in the dense apply pass, into something that put a positive NaN below the
// cut (the pass then dropped kept NaNs that the selection had counted).
__device__ __forceinline__ uint32_t key_of_bits(uint32_t u) {
  asm("mov.b32 %0, %0;" : "+r"(u));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t order_key(float f) { return key_of_bits(__float_as_uint(f)); }

// inverse of order_key
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// the accumulation's new word for a kept entry: its residual x - (0 + x)
// (the sent values are scattered into zeros first, which turns -0 into +0)
__device__ __forceinline__ uint32_t kept_residual_bits(uint32_t key) {
  const float x = key_value(key);
  return __float_as_uint(__fsub_rn(x, __fadd_rn(0.0f, x)));
}

// x = in (+ accumulation), one element (the accumulation alone once the
// candidate pass has stored x there)
__device__ __forceinline__ float load_x(const SparseParams& p, int r, int64_t i) {
  if (p.x_in_acc) return __uint_as_float(ld1<uint32_t>((const char*)p.acc[r] + i * 4));
  float x = __uint_as_float(ld1<uint32_t>((const char*)p.in[r] + i * 4));
  if (p.has_acc) x = __fadd_rn(x, __uint_as_float(ld1<uint32_t>((const char*)p.acc[r] + i * 4)));
  return x;
}

// the same for a 16-byte vector of four elements
__device__ __forceinline__ void load_x4(const SparseParams& p, int r, int64_t i, float (&x)[4]) {
  const uint4 a = ld_stream((const char*)(p.x_in_acc ? p.acc[r] : p.in[r]) + i * 4);
  x[0] = __uint_as_float(a.x);
  x[1] = __uint_as_float(a.y);
  x[2] = __uint_as_float(a.z);
  x[3] = __uint_as_float(a.w);
  if (p.has_acc && !p.x_in_acc) {
    const uint4 b = ld_stream((const char*)p.acc[r] + i * 4);
    x[0] = __fadd_rn(x[0], __uint_as_float(b.x));
    x[1] = __fadd_rn(x[1], __uint_as_float(b.y));
    x[2] = __fadd_rn(x[2], __uint_as_float(b.z));
    x[3] = __fadd_rn(x[3], __uint_as_float(b.w));
  }
}

// The pass kernels run 256 threads over tiles of kSparseTileElems entries:
// a tile's aligned body is at most kTileVecs 16-byte vectors per thread.
constexpr int kSparseThreads = 256;
constexpr int kTileVecs = (int)(kSparseTileElems / 4 / kSparseThreads);
static_assert(kTileVecs * 4 * kSparseThreads == kSparseTileElems, "tile = threads x vectors");

// A 16-byte load with the default L2 policy: for data read again shortly
// (the sample, whose second-digit pass follows its first-digit pass).
__device__ __forceinline__ uint4 ld_keep(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// x for this thread's vectors v = tid + u * 256 (u < kTileVecs, v < nv) of
// the aligned body starting at av; every load is issued before the first add
// so that each thread keeps up to 2 x kTileVecs x 16 bytes in flight.
// Vectors past nv read as zeros (the caller masks them).  KEEP: loads that
// leave the tile in L2 for a pass that reads it again.
template <bool KEEP = false>
__device__ __forceinline__ void load_tile_x(const SparseParams& p, int r, int64_t av, int64_t nv,
                                            float (&x)[kTileVecs][4]) {
  auto ld = [](const void* q) { return KEEP ? ld_keep(q) : ld_stream(q); };
  uint4 a[kTileVecs], b[kTileVecs];
#pragma unroll
  for (int u = 0; u < kTileVecs; ++u) {
    const int64_t v = threadIdx.x + u * kSparseThreads;
    a[u] = make_uint4(0u, 0u, 0u, 0u);
    b[u] = make_uint4(0u, 0u, 0u, 0u);
    if (v < nv) {
      a[u] = ld((const char*)(p.x_in_acc ? p.acc[r] : p.in[r]) + (av + v * 4) * 4);
      if (p.has_acc && !p.x_in_acc) b[u] = ld((const char*)p.acc[r] + (av + v * 4) * 4);
    }
  }
#pragma unroll
  for (int u = 0; u < kTileVecs; ++u) {
    reg_fence(a[u]);
    reg_fence(b[u]);
  }
#pragma unroll
  for (int u = 0; u < kTileVecs; ++u) {
    x[u][0] = __uint_as_float(a[u].x);
    x[u][1] = __uint_as_float(a[u].y);
    x[u][2] = __uint_as_float(a[u].z);
    x[u][3] = __uint_as_float(a[u].w);
    if (p.has_acc && !p.x_in_acc) {
      x[u][0] = __fadd_rn(x[u][0], __uint_as_float(b[u].x));
      x[u][1] = __fadd_rn(x[u][1], __uint_as_float(b[u].y));
      x[u][2] = __fadd_rn(x[u][2], __uint_as_float(b[u].z));
      x[u][3] = __fadd_rn(x[u][3], __uint_as_float(b[u].w));
    }
  }
}

// digit of pass P and whether the key matches the prefix fixed so far
template <int P>
__device__ __forceinline__ bool digit_of(uint32_t key, uint32_t prefix, uint32_t& d) {
  if (P == 0) {
    d = key >> 21;
    return true;
  }
  if (P == 1) {
    d = (key >> 10) & 0x7FFu;
    return (key >> 21) == prefix;
  }
  d = key & 0x3FFu;
  return (key >> 10) == prefix;
}

// digit of index pass P (3, 4, 5) of an inverted index (larger = lower index)
template <int P>
__device__ __forceinline__ bool index_digit_of(uint32_t inv, uint32_t prefix, uint32_t& d) {
  if (P == 3) {
    d = inv >> 21;
    return true;
  }
  if (P == 4) {
    d = (inv >> 10) & 0x7FFu;
    return (inv >> 21) == prefix;
  }
  d = inv & 0x3FFu;
  return (inv >> 10) == prefix;
}

// the first-digit pass only counts bins from state.low up
template <int MODE>
__device__ __forceinline__ bool counted_bin(uint32_t d, uint32_t low) {
  if constexpr (MODE == 0)
    return d >= low;
  else
    return true;
}

// The first-digit bin the second-digit sample pass refines: the settled
// bound's, else the lower bound's when it still wants keys inside its bin;
// -1: neither (nothing settled, no lower bound)
__device__ __forceinline__ int refined_bin(const TopkState& st) {
  if (st.setkey != 0xFFFFFFFFu) return (int)(st.setkey >> 21);
  if (st.low_rem > 0) return (int)(st.lowkey >> 21);
  return st.hi_rem > 0 ? (int)(st.topkey >> 21) : -1;
}

// shared-memory histogram add, lanes that share a bin combined first
__device__ __forceinline__ void hist_add(uint32_t* h, bool valid, uint32_t d) {
  const unsigned active = __ballot_sync(0xFFFFFFFFu, valid);
  if (!valid) return;
  const unsigned peers = __match_any_sync(active, d);
  if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[d], (uint32_t)__popc(peers));
}

}  // namespace

// ---------------------------------------------------------------- histogram
// grid.y = rank; each CTA counts the digits of its tiles of that rank into a
// shared histogram, then adds it to the rank's global histogram.  The first
// digit above a lower bound clusters in a few bins, so lanes sharing a bin
// combine into one atomic there; the sample's first digit spreads over the
// whole distribution and the later digits over many bins, where plain
// shared atomics are cheaper.
//
// MODE 0: the first digit, bins >= state.low only (a lower bound from the
//         sample pass: keys below it cannot be among the K largest when the
//         counted bins hold at least K keys -- checked by the selection);
// MODE 1, 2: the second and third digits, keys matching the prefix so far;
// MODE 3: the first digit over a sample (every sample_stride-th tile);
// MODE 4: the first digit over all bins, only for ranks whose bound failed;
// MODE 5: the second digit over the same sample, keys in the first-digit bin
//         of the settled bound (which refines it, and the lower bound when
//         that lies in the same bin), else in the lower bound's bin (which
//         refines it, and a band's upper bound when that lies in the same
//         bin), else in the upper bound's bin.
// With candidate lists, MODES 1 and 2 run only for ranks on the full path.
template <int MODE>
__global__ void __launch_bounds__(256) vc_topk_hist(const __grid_constant__ SparseParams p) {
  pdl_enter();
  constexpr int P = (MODE == 1 || MODE == 2) ? MODE : MODE == 5 ? 1 : 0;
  __shared__ uint32_t h[kTopkBins];
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const TopkState& st = p.state[r];
  if (MODE == 4 && !st.redo) return;  // uniform per CTA
  if ((MODE == 1 || MODE == 2) && p.use_cand && !st.full) return;  // read its candidates
  if (MODE == 5 && refined_bin(st) < 0) return;                      // nothing to refine
  for (int i = tid; i < kTopkBins; i += blockDim.x) h[i] = 0;
  const uint32_t prefix = MODE == 5 ? (uint32_t)refined_bin(st) : st.prefix;
  const uint32_t low = MODE == 0 ? st.low : 0u;
  __syncthreads();
  const int64_t step = (MODE == 3 || MODE == 5) ? p.sample_stride : 1;
  for (int64_t tile = (int64_t)blockIdx.x * step; tile < p.tiles_per_rank;
       tile += (int64_t)gridDim.x * step) {
    const int64_t t0 = tile * p.tile_elems;
    const int64_t t1 = t0 + p.tile_elems < p.n ? t0 + p.tile_elems : p.n;
    if (p.phase >= 0) {
      int64_t av, bv;
      aligned_body<4>(t0, t1, p.phase, av, bv);
      // vectors [av, bv), all loads first; every lane of a warp makes the
      // same hist_add calls so that the warp-wide combining stays converged
      const int64_t nv = (bv - av) / 4;
      float x[kTileVecs][4];
      load_tile_x<MODE == 3>(p, r, av, nv, x);  // the sample stays in L2 for MODE 5
#pragma unroll
      for (int u = 0; u < kTileVecs; ++u) {
        const bool in_range = tid + u * kSparseThreads < nv;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t d;
          const bool m = digit_of<P>(order_key(x[u][q]), prefix, d) &&
                         counted_bin<MODE>(d, low) && in_range;
          if (P == 0 && MODE != 3)
            hist_add(h, m, d);
          else if (m)  // later digits (and the sample's first digit, which
            atomicAdd(&h[d], 1u);  // spans the whole distribution): plain atomics
        }
      }
      // head [t0, av) and tail [bv, t1): fewer than 4 elements each
      int64_t i = -1;
      if (tid < av - t0) i = t0 + tid;
      if (tid >= 32 && tid - 32 < t1 - bv) i = bv + (tid - 32);
      if (i >= 0) {
        uint32_t d;
        if (digit_of<P>(order_key(load_x(p, r, i)), prefix, d) && counted_bin<MODE>(d, low))
          atomicAdd(&h[d], 1u);
      }
    } else {
      for (int64_t base = t0; base < t1; base += blockDim.x) {
        const int64_t i = base + tid;
        uint32_t d = 0;
        bool m = false;
        if (i < t1) m = digit_of<P>(order_key(load_x(p, r, i)), prefix, d) && counted_bin<MODE>(d, low);
        if (P == 0 && MODE != 3)
          hist_add(h, m, d);
        else if (m)
          atomicAdd(&h[d], 1u);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < kTopkBins; i += blockDim.x)
    if (h[i]) atomicAdd(&p.hist[(int64_t)r * kTopkBins + i], h[i]);
}

// ---------------------------------------------------------------- selection
// One CTA of 1024 threads per rank: thread t owns bins 2047-2t and 2046-2t;
// an inclusive scan from the top bin down finds the digit holding the
// remaining-th largest key; the rank's histogram is cleared for the next pass.
//
// MODE 0, 1, 2: after the histogram pass of that digit (MODE 0 flags a redo
//   when the bins counted from state.low up hold fewer than K keys);
// MODE 3: after the sample pass: state.low = the highest bin whose sampled
//   suffix holds comfortably more keys than K calls for (scaled to the
//   sample), 0 (count everything) when none does; with a band also
//   state.topkey = the last key of the highest bin with comfortably fewer
//   than that strictly above it (entries above it are kept without being
//   listed), else 0xFFFFFFFF; state.lowkey = the first key of state.low; on
//   the list route (with accumulations) state.setkey = the last key of the
//   bin that bound would end without a band (entries above it are listed,
//   and kept for certain unless the sample misled), else 0xFFFFFFFF;
//   low_rem, set_rem and hi_rem keep what each bound still needs inside its
//   bin;
// MODE 4: after the redo pass, for ranks that needed it;
// MODE 5, 6, 7: after index pass 3, 4, 5 over the candidates equal to T, for
//   ranks on the candidate path whose equal keys straddle the cut; the last
//   one sets the boundary index;
// MODE 8: after the second-digit sample pass: setkey moves down to the last
//   key of the second-digit bin holding its set_rem-th sampled key, lowkey,
//   when it starts the refined first-digit bin, up to the first key of the
//   second-digit bin holding its low_rem-th one, and a band's topkey, when it
//   ends the refined bin, down to the last key of the second-digit bin
//   holding its hi_rem-th one.
template <int MODE>
__global__ void __launch_bounds__(1024) vc_topk_select(const __grid_constant__ SparseParams p) {
  pdl_enter();
  const int r = blockIdx.x;
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  __shared__ unsigned long long warp_sum[32];
  uint32_t* hist = p.hist + (int64_t)r * kTopkBins;
  TopkState* st = p.state + r;
  if (MODE == 4 && !st->redo) return;
  // (uniform per CTA; nothing was counted for these ranks, the bins are zero)
  if (MODE >= 5 && MODE <= 7 &&
      (p.K == 0 || st->full || st->need >= st->equal || st->tie_resolved))
    return;
  if (MODE == 8 && refined_bin(*st) < 0) return;
  const int b0 = kTopkBins - 1 - 2 * t, b1 = b0 - 1;
  const unsigned long long c0 = hist[b0], c1 = hist[b1];
  unsigned long long s = c0 + c1;
  // inclusive scan over threads (descending bins)
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, s, o);
    if (lane >= o) s += y;
  }
  if (lane == 31) warp_sum[warp] = s;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = warp_sum[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    warp_sum[lane] = w;
  }
  __syncthreads();
  const unsigned long long incl = s + (warp > 0 ? warp_sum[warp - 1] : 0ull);
  const unsigned long long above = incl - c0 - c1;  // keys in bins > b0
  const unsigned long long total = warp_sum[31];
  constexpr int P = (MODE == 1 || MODE == 2) ? MODE : 0;
  long long rem;
  long long rhi = 0;  // MODE 3: sampled keys allowed strictly above the band
  long long rset = 0; // MODE 3: sampled keys allowed strictly above the settled bin
  if (MODE == 3) {
    // K's share of the sample; keys wanted at or above the lower bound: twice
    // that plus 64 (wide bound), or that plus a margin -- a few standard
    // deviations, at least 1/16 of the smaller tail -- with an upper bound
    // the same margin below it (band); nothing when K = n.  The settled bin
    // of the wide bound leaves the same margin below K.
    const long long ks = (long long)(((unsigned long long)p.K * total) / (unsigned long long)p.n);
    if (p.K >= p.n) {
      rem = -1;
    } else if (!p.band) {
      rem = 2 * ks + 64;
      if (p.list_out && p.has_acc)
        rset = ks - max((long long)(4.0f * sqrtf((float)ks)) + 64, ks / 16);
    } else {
      const long long tail = min(ks, (long long)total - ks);
      const long long m = max((long long)(4.0f * sqrtf((float)tail)) + 64, tail / 16);
      rem = ks + m;
      rhi = ks - m;
    }
  } else if (MODE == 5) {
    rem = st->need;
  } else if (MODE == 8) {
    rem = 0;  // two targets, below
  } else if (MODE == 0) {  // on the candidate path the band's share of K
    rem = p.K - (p.use_cand ? (long long)p.cand_n[p.W + r] : 0ll);
  } else {
    rem = (P == 0 && MODE < 5) ? p.K : st->remaining;
  }
  const uint32_t prefix = (P == 0 && MODE < 6) ? 0u : st->prefix;
  // MODE 8: the refined first-digit bin, what both bounds still need inside
  // it, and whether each bound lies in it
  const uint32_t sbin = MODE == 8 ? (uint32_t)refined_bin(*st) : 0u;
  const bool set_here = MODE == 8 && st->setkey != 0xFFFFFFFFu;
  const long long set_rem = MODE == 8 ? st->set_rem : 0, low_rem = MODE == 8 ? st->low_rem : 0;
  const bool low_here = MODE == 8 && low_rem > 0 && st->lowkey == sbin << 21;
  const long long hi_rem = MODE == 8 ? st->hi_rem : 0;
  const bool hi_here = MODE == 8 && hi_rem > 0 && st->topkey != 0xFFFFFFFFu &&
                       (st->topkey >> 21) == sbin;
  __syncthreads();  // every thread has read the state before it changes
  // the bin (b0 or b1) holding the target-th key, and the keys above it
  auto pick = [&](long long target, unsigned long long& more) -> uint32_t {
    if ((long long)(above + c0) >= target) {
      more = above;
      return (uint32_t)b0;
    }
    more = above + c0;
    return (uint32_t)b1;
  };
  if (MODE == 3) {
    unsigned long long more;
    if (t == 0 && (rem < 0 || (long long)total < rem)) {
      st->low = 0;
      st->lowkey = 0;
      st->low_rem = 0;
    }
    if (rem >= 0 && (long long)total >= rem && (long long)above < rem && rem <= (long long)incl) {
      const uint32_t bin = pick(rem, more);
      st->low = bin;
      st->lowkey = bin << 21;
      st->low_rem = rem - (long long)more;
    }
    if (t == 0 && (rhi <= 0 || (long long)total < rhi)) {
      st->topkey = 0xFFFFFFFFu;
      st->hi_rem = 0;
    }
    if (rhi > 0 && (long long)total >= rhi && (long long)above < rhi && rhi <= (long long)incl) {
      const uint32_t bin = pick(rhi, more);
      st->topkey = (uint32_t)((((uint64_t)bin + 1) << 21) - 1);
      st->hi_rem = rhi - (long long)more;
    }
    if (t == 0 && (rset <= 0 || (long long)total < rset)) {
      st->setkey = 0xFFFFFFFFu;
      st->set_rem = 0;
    }
    if (rset > 0 && (long long)total >= rset && (long long)above < rset && rset <= (long long)incl) {
      const uint32_t bin = pick(rset, more);
      st->setkey = (uint32_t)((((uint64_t)bin + 1) << 21) - 1);
      st->set_rem = rset - (long long)more;
    }
    if (t == 0) st->redo = 0;
  } else if (MODE == 8) {
    unsigned long long more;
    if (set_here && set_rem > 0 && (long long)above < set_rem && set_rem <= (long long)incl) {
      const uint64_t p22 = ((uint64_t)sbin << 11) | pick(set_rem, more);
      st->setkey = (uint32_t)(((p22 + 1) << 10) - 1);
    }
    if (low_here && (long long)above < low_rem && low_rem <= (long long)incl)
      st->lowkey = (sbin << 21) | (pick(low_rem, more) << 10);
    if (hi_here && (long long)above < hi_rem && hi_rem <= (long long)incl) {
      const uint64_t p22 = ((uint64_t)sbin << 11) | pick(hi_rem, more);
      st->topkey = (uint32_t)(((p22 + 1) << 10) - 1);
    }
  } else if (MODE == 0 && (rem <= 0 || (long long)total < rem)) {
    if (t == 0) {  // a bound missed the K-th key (or the list overflowed): count every bin again
      st->redo = 1;
      st->full = 1;
    }
  } else if (rem > 0 && (long long)above < rem && rem <= (long long)incl) {
    int bin;
    unsigned long long more;  // keys strictly above the chosen bin
    if ((long long)(above + c0) >= rem) {
      bin = b0;
      more = above;
    } else {
      bin = b1;
      more = above + c0;
    }
    const long long left = rem - (long long)more;
    if (MODE == 5) {
      st->prefix = (uint32_t)bin;
      st->remaining = left;
    } else if (MODE == 6) {
      st->prefix = (prefix << 11) | (uint32_t)bin;
      st->remaining = left;
    } else if (MODE == 7) {  // one index per inverted index: left == 1
      st->boundary = (int64_t)(0xFFFFFFFFu - ((prefix << 10) | (uint32_t)bin));
    } else if (P == 0) {
      st->prefix = (uint32_t)bin;
      st->remaining = left;
      st->redo = 0;
    } else if (P == 1) {
      st->prefix = (prefix << 11) | (uint32_t)bin;
      st->remaining = left;
    } else {
      st->T = (prefix << 10) | (uint32_t)bin;
      st->need = left;
      st->equal = (long long)(bin == b0 ? c0 : c1);
      st->boundary = left == st->equal ? 0x7FFFFFFFFFFFFFFFll : -1;
    }
  }
  hist[b0] = 0;
  hist[b1] = 0;
}

// ---------------------------------------------------------------------- ties
// Only for ranks whose keys equal to the K-th largest straddle the cut
// (need < equal): (1) every tile counts its entries equal to T; (2) one CTA
// per rank scans the tile counts to the tile holding the need-th equal entry
// and then that tile in index order; the entry's index is the boundary.
__global__ void __launch_bounds__(256) vc_topk_tie_count(const __grid_constant__ SparseParams p) {
  pdl_enter();
  __shared__ int wc[8];
  const int r = blockIdx.y;
  const TopkState* st = p.state + r;
  if (p.K == 0 || st->need >= st->equal) return;  // uniform per CTA
  if (p.use_cand && !st->full) return;            // the index passes handle it
  const uint32_t T = st->T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int64_t tile = blockIdx.x; tile < p.tiles_per_rank; tile += gridDim.x) {
    const int64_t t0 = tile * p.tile_elems;
    const int64_t t1 = t0 + p.tile_elems < p.n ? t0 + p.tile_elems : p.n;
    int c = 0;
    if (p.phase >= 0) {
      int64_t av, bv;
      aligned_body<4>(t0, t1, p.phase, av, bv);
      const int64_t nv = (bv - av) / 4;
      for (int64_t v = tid; v < nv; v += blockDim.x) {
        float x[4];
        load_x4(p, r, av + v * 4, x);
#pragma unroll
        for (int q = 0; q < 4; ++q) c += order_key(x[q]) == T;
      }
      if (tid < av - t0) c += order_key(load_x(p, r, t0 + tid)) == T;
      if (tid >= 32 && tid - 32 < t1 - bv) c += order_key(load_x(p, r, bv + (tid - 32))) == T;
    } else {
      for (int64_t i = t0 + tid; i < t1; i += blockDim.x) c += order_key(load_x(p, r, i)) == T;
    }
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) wc[warp] = c;
    __syncthreads();
    if (tid == 0) {
      int sum = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) sum += wc[w];
      p.tilecnt[(int64_t)r * p.tiles_per_rank + tile] = (uint32_t)sum;
    }
    __syncthreads();
  }
}

// block-wide exclusive scan of one int per thread (1024 threads); *total gets
// the sum
__device__ __forceinline__ long long block_excl_scan(long long v, long long* total) {
  __shared__ long long ws[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long s = v;
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xFFFFFFFFu, s, o);
    if (lane >= o) s += y;
  }
  if (lane == 31) ws[warp] = s;
  __syncthreads();
  if (warp == 0) {
    long long w = ws[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    ws[lane] = w;
  }
  __syncthreads();
  const long long excl = s - v + (warp > 0 ? ws[warp - 1] : 0);
  *total = ws[31];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(1024) vc_topk_tie_find(const __grid_constant__ SparseParams p) {
  pdl_enter();
  const int r = blockIdx.x;
  TopkState* st = p.state + r;
  const long long need = st->need, equal = st->equal;
  if (p.K == 0 || need >= equal) return;
  if (p.use_cand && !st->full) return;
  const uint32_t T = st->T;
  const uint32_t* cnt = p.tilecnt + (int64_t)r * p.tiles_per_rank;
  __shared__ long long s_tile, s_before, s_found;
  if (threadIdx.x == 0) {
    s_tile = -1;
    s_found = -1;
  }
  __syncthreads();
  // the tile where the running count of equal entries reaches need
  long long seen = 0;
  for (int64_t base = 0; base < p.tiles_per_rank; base += blockDim.x) {
    const int64_t k = base + threadIdx.x;
    const long long c = k < p.tiles_per_rank ? cnt[k] : 0;
    long long total;
    const long long before = seen + block_excl_scan(c, &total);
    if (c > 0 && before < need && need <= before + c) {
      s_tile = k;
      s_before = before;
    }
    __syncthreads();
    seen += total;
    if (s_tile >= 0) break;
  }
  const int64_t tile = s_tile;
  if (tile < 0) return;  // cannot happen when the histograms are consistent
  // inside that tile, in index order
  const int64_t t0 = tile * p.tile_elems;
  const int64_t t1 = t0 + p.tile_elems < p.n ? t0 + p.tile_elems : p.n;
  seen = s_before;
  for (int64_t base = t0; base < t1; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    const bool eq = i < t1 && order_key(load_x(p, r, i)) == T;
    long long total;
    const long long before = seen + block_excl_scan(eq ? 1 : 0, &total);
    if (eq && before + 1 == need) s_found = i;
    __syncthreads();
    seen += total;
    if (s_found >= 0) break;
  }
  if (threadIdx.x == 0) st->boundary = s_found;
}

// ------------------------------------------------------------ candidates
// Keys above this one are settled (0xFFFFFFFF: none are).
__device__ __forceinline__ uint32_t settled_key(const SparseParams& p, int r) {
  if (!p.list_out || !p.has_acc) return 0xFFFFFFFFu;
  return p.state[r].setkey;
}

// One pass over the data (grid.y = rank, one tile per CTA iteration): every
// entry whose key lies in the sample's band [lowkey, topkey] is appended to
// the rank's candidate list as (key, index), and the entries above the band
// are counted (they are kept whatever the K-th key).  With an
// accumulation, x = in + acc is stored back into acc, so that every later
// pass reads one array instead of two -- except that a candidate above the
// settled key gets its residual x - (0 + x) instead, kept when its whole
// tile is listed (the output pass undoes it in the rare case the entry is
// not kept after all, and so does vc_topk_restore when the result does not
// come from the lists).  Each thread looks at 16 entries of the tile (four
// 16-byte vectors, all loaded before the first is used) plus at most one of
// the tile's unaligned head or tail; a warp-wide scan of the per-thread counts
// places every candidate, one shared atomic per warp and one global atomic
// per tile reserve room, and each thread then visits only its own candidates
// (their keys parked in shared memory, so the loop over set bits needs no
// register indexing).  The list is compact; the order between tiles is
// arbitrary (the index travels with the key).  Entries past the capacity are
// counted but not stored, which sends the rank to the full path.  Only the
// form with accumulations (ACC) runs; the pass without them is
// vc_topk_filter_raw below.
template <bool ACC>
__global__ void __launch_bounds__(256) vc_topk_filter(const __grid_constant__ SparseParams p) {
  pdl_enter();
  constexpr int E = 4 * kTileVecs;  // entries per thread and tile (plus one extra)
  __shared__ __align__(16) uint32_t s_key[kSparseThreads * E];
  __shared__ uint32_t s_n, s_sure;
  __shared__ unsigned long long s_base;
  __shared__ int s_listed;  // the whole tile fits in the list
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31;
  // candidates: keys in [lowkey, topkey]; keys above topkey are kept for sure
  const uint32_t lowkey = p.state[r].lowkey;
  const uint32_t topkey = p.state[r].topkey;
  const uint32_t setkey = ACC ? settled_key(p, r) : 0xFFFFFFFFu;
  uint32_t* ckey = p.cand_key + (int64_t)r * p.cand_cap;
  uint32_t* cidx = p.cand_idx + (int64_t)r * p.cand_cap;
  uint32_t* my = s_key + tid * E;
  for (int64_t tile = blockIdx.x; tile < p.tiles_per_rank; tile += gridDim.x) {
    const int64_t t0 = tile * p.tile_elems;
    const int64_t t1 = t0 + p.tile_elems < p.n ? t0 + p.tile_elems : p.n;
    if (tid == 0) {
      s_n = 0;
      s_sure = 0;
    }
    uint32_t mask = 0;     // bit j < E: entry j is a candidate
    uint32_t settle = 0;   // bit j: a candidate above the settled key
    int sure = 0;          // entries above the band
    uint32_t xkey = 0;     // the extra entry (head or tail)
    bool xhit = false;
    int64_t av = t0, extra = -1;
    const bool vec = p.phase >= 0;
    int64_t nv = 0;
    if (vec) {
      int64_t bv;
      aligned_body<4>(t0, t1, p.phase, av, bv);
      nv = (bv - av) / 4;
      float x[kTileVecs][4];
      load_tile_x(p, r, av, nv, x);
#pragma unroll
      for (int u = 0; u < kTileVecs; ++u) {
        uint4 k4;
        k4.x = order_key(x[u][0]);
        k4.y = order_key(x[u][1]);
        k4.z = order_key(x[u][2]);
        k4.w = order_key(x[u][3]);
        uint32_t m4 = 0, s4 = 0;
        if (tid + u * kSparseThreads < nv) {
          m4 = (uint32_t)(k4.x >= lowkey && k4.x <= topkey) |
               (uint32_t)(k4.y >= lowkey && k4.y <= topkey) << 1 |
               (uint32_t)(k4.z >= lowkey && k4.z <= topkey) << 2 |
               (uint32_t)(k4.w >= lowkey && k4.w <= topkey) << 3;
          s4 = m4 & ((uint32_t)(k4.x > setkey) | (uint32_t)(k4.y > setkey) << 1 |
                     (uint32_t)(k4.z > setkey) << 2 | (uint32_t)(k4.w > setkey) << 3);
          sure += (k4.x > topkey) + (k4.y > topkey) + (k4.z > topkey) + (k4.w > topkey);
          // later passes read x from the accumulation; a settled candidate
          // gets its residual at once (undone below in the rare tile that
          // does not fit in the list)
          if (ACC) {
            uint4 o = make_uint4(__float_as_uint(x[u][0]), __float_as_uint(x[u][1]),
                                 __float_as_uint(x[u][2]), __float_as_uint(x[u][3]));
            if (s4 & 1u) o.x = kept_residual_bits(k4.x);
            if (s4 & 2u) o.y = kept_residual_bits(k4.y);
            if (s4 & 4u) o.z = kept_residual_bits(k4.z);
            if (s4 & 8u) o.w = kept_residual_bits(k4.w);
            st_stream((char*)p.acc[r] + (av + (int64_t)(tid + u * kSparseThreads) * 4) * 4, o);
          }
        }
        mask |= m4 << (u * 4);
        settle |= s4 << (u * 4);
        reinterpret_cast<uint4*>(my)[u] = k4;
      }
      // head [t0, av) and tail [bv, t1): fewer than 4 entries each
      if (tid < av - t0) extra = t0 + tid;
      if (tid >= 32 && tid - 32 < t1 - bv) extra = bv + (tid - 32);
    } else {  // element-wise: entries t0 + tid + 256 j, stored below
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int64_t i = t0 + tid + (int64_t)j * kSparseThreads;
        uint32_t k = 0;
        if (i < t1) {
          k = order_key(load_x(p, r, i));
          const bool hit = k >= lowkey && k <= topkey;
          mask |= (uint32_t)hit << j;
          settle |= (uint32_t)(hit && k > setkey) << j;
          sure += k > topkey;
        }
        my[j] = k;
      }
    }
    if (extra >= 0) {  // stored below
      xkey = order_key(load_x(p, r, extra));
      xhit = xkey >= lowkey && xkey <= topkey;
      sure += xkey > topkey;
    }
    // this thread's place among the warp's candidates
    const int c = __popc(mask) + (xhit ? 1 : 0);
    int incl = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const int wtotal = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const unsigned wsure = __reduce_add_sync(0xFFFFFFFFu, (unsigned)sure);
    __syncthreads();  // s_n and s_sure are zero
    uint32_t wbase = 0;
    if (lane == 31 && wtotal) wbase = atomicAdd(&s_n, (uint32_t)wtotal);
    if (lane == 0 && wsure) atomicAdd(&s_sure, wsure);
    wbase = __shfl_sync(0xFFFFFFFFu, wbase, 31);
    __syncthreads();  // every warp has reserved its share of the tile's room
    if (tid == 0) {
      const uint32_t tot = s_n;
      s_base = tot ? atomicAdd(p.cand_n + r, (unsigned long long)tot) : 0ull;
      s_listed = s_base + tot <= (unsigned long long)p.cand_cap;
      if (s_sure) atomicAdd(p.cand_n + p.W + r, (unsigned long long)s_sure);
      // where this tile's entries sit in the list (read by the output pass
      // of the list route; the start only matters below the capacity)
      p.tilecnt[(int64_t)r * p.tiles_per_rank + tile] = tot;
      p.chunk[(int64_t)r * p.tiles_per_rank + tile] = (uint32_t)s_base;
    }
    __syncthreads();
    unsigned long long pos = s_base + wbase + (uint32_t)(incl - c);
    const unsigned long long cap = (unsigned long long)p.cand_cap;
    for (uint32_t m = mask; m; m &= m - 1u) {  // this thread's candidates only
      const int j = __ffs(m) - 1;
      const int64_t i = vec ? av + (int64_t)(tid + (j >> 2) * kSparseThreads) * 4 + (j & 3)
                            : t0 + tid + (int64_t)j * kSparseThreads;
      if (pos < cap) {
        ckey[pos] = my[j];
        cidx[pos] = (uint32_t)i;
      }
      ++pos;
    }
    if (xhit && pos < cap) {
      ckey[pos] = xkey;
      cidx[pos] = (uint32_t)extra;
    }
    if (ACC) {
      // settled candidates keep their residual only when the whole tile is
      // listed (else the rank goes to the full path, which reads x)
      const bool listed = s_listed;
      const uint32_t res = listed ? settle : 0u;
      auto word = [&](uint32_t key, bool settled) -> uint32_t {
        return settled ? kept_residual_bits(key) : __float_as_uint(key_value(key));
      };
      if (vec) {
        if (!listed)  // x again where a residual went
#pragma unroll
          for (int u = 0; u < kTileVecs; ++u)
            if (tid + u * kSparseThreads < nv && ((settle >> (u * 4)) & 15u)) {
              const uint4 k4 = reinterpret_cast<const uint4*>(my)[u];
              st_stream((char*)p.acc[r] + (av + (int64_t)(tid + u * kSparseThreads) * 4) * 4,
                        make_uint4(word(k4.x, false), word(k4.y, false), word(k4.z, false),
                                   word(k4.w, false)));
            }
      } else {
#pragma unroll
        for (int j = 0; j < E; ++j) {
          const int64_t i = t0 + tid + (int64_t)j * kSparseThreads;
          if (i < t1) st1((char*)p.acc[r] + i * 4, word(my[j], (res >> j) & 1u));
        }
      }
      if (extra >= 0) st1((char*)p.acc[r] + extra * 4, word(xkey, listed && xhit && xkey > setkey));
    }
    // (after the second barrier only thread 0 reads s_n and s_sure, so it
    // may reset them for the next tile; s_base and s_listed change only
    // after the next tile's second barrier, which every thread passes after
    // these reads; each thread reads only its own row of s_key)
  }
}

// "key >= bound" on the raw fp32 bits u, without forming the key: for a
// bound at or above the key of +0 (sign bit set) it is a signed compare of u
// against the bound's low 31 bits (negative u, -0 included, lies below);
// below it an unsigned compare against ~bound (every non-negative u passes,
// a negative u when ~u >= bound).  NaNs order as their keys do.
struct RawBound {
  uint32_t t;
  bool sgn;
};
__device__ __forceinline__ RawBound raw_bound(uint32_t key) {
  return (key & 0x80000000u) ? RawBound{key & 0x7FFFFFFFu, true} : RawBound{~key, false};
}
template <bool SGN>
__device__ __forceinline__ bool raw_at_least(uint32_t u, uint32_t t) {
  return SGN ? (int32_t)u >= (int32_t)t : u <= t;
}

// One tile of the candidate pass without accumulations: each thread loads
// four 16-byte vectors (vector v = tid + 256 u of the tile's aligned body)
// and at most one of the tile's unaligned head or tail entries; bit 4 u + q
// of the thread's mask is entry q of its vector u.  LOW_SGN: the lower
// bound's compare form (uniform per rank); HI: no upper bound (0), or a
// band's upper bound in the unsigned (1) or signed (2) compare form --
// entries at or above it are counted, not listed: one mask of them per
// thread, counted once.  The keys of the listed entries are formed only for
// those entries.
template <bool LOW_SGN, int HI>
__device__ __forceinline__ void filter_tile_raw(const SparseParams& p, int r, int64_t tile,
                                                const RawBound lo, const RawBound hi,
                                                uint32_t* s_raw, uint32_t* s_n, uint32_t* s_sure,
                                                int par, unsigned long long& s_base) {
  constexpr int E = 4 * kTileVecs;  // entries per thread (plus one extra)
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr bool BAND = HI != 0;
  auto above = [&](uint32_t u) -> bool { return BAND && raw_at_least<HI == 2>(u, hi.t); };
  auto cand = [&](uint32_t u) -> bool { return raw_at_least<LOW_SGN>(u, lo.t) && !above(u); };
  const char* src = (const char*)p.in[r];
  const bool vec = p.phase >= 0;
  const int64_t t0 = tile * p.tile_elems;
  const int64_t t1 = t0 + p.tile_elems < p.n ? t0 + p.tile_elems : p.n;
  int64_t av = t0, bv = t0;
  if (vec) aligned_body<4>(t0, t1, p.phase, av, bv);
  const int nv = (int)((bv - av) / 4);
  uint32_t mask = 0;
  uint32_t hmask = 0;  // entries above the band (as mask)
  int sure = 0;        // entries above the band
  // the one extra entry: threads 0-31 take the tile's head, 32-63 its tail
  int64_t extra = -1;
  uint32_t xraw = 0;
  bool xhit = false;
  if (vec) {
    uint4 a[kTileVecs];
    const char* tp = src + av * 4 + tid * 16;
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
      a[u] = make_uint4(0u, 0u, 0u, 0u);
      if (tid + u * kSparseThreads < nv) a[u] = ld_stream(tp + u * kSparseThreads * 16);
    }
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) reg_fence(a[u]);
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
      const uint4 x = a[u];
      if (tid + u * kSparseThreads < nv) {
        const uint32_t ge = (uint32_t)raw_at_least<LOW_SGN>(x.x, lo.t) |
                            (uint32_t)raw_at_least<LOW_SGN>(x.y, lo.t) << 1 |
                            (uint32_t)raw_at_least<LOW_SGN>(x.z, lo.t) << 2 |
                            (uint32_t)raw_at_least<LOW_SGN>(x.w, lo.t) << 3;
        if (BAND) {
          const uint32_t up = (uint32_t)above(x.x) | (uint32_t)above(x.y) << 1 |
                              (uint32_t)above(x.z) << 2 | (uint32_t)above(x.w) << 3;
          mask |= (ge & ~up) << (u * 4);
          hmask |= up << (u * 4);
        } else {
          mask |= ge << (u * 4);
        }
      }
      // vector u of every thread side by side: a warp's stores are contiguous
      reinterpret_cast<uint4*>(s_raw)[u * kSparseThreads + tid] = x;
    }
    if (tid < av - t0) extra = t0 + tid;
    if (tid >= 32 && tid - 32 < t1 - bv) extra = bv + (tid - 32);
  } else {  // element-wise: entries t0 + tid + 256 j
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int64_t i = t0 + tid + (int64_t)j * kSparseThreads;
      uint32_t x = 0;
      if (i < t1) {
        x = ld1<uint32_t>(src + i * 4);
        mask |= (uint32_t)cand(x) << j;
        if (BAND) sure += above(x);
      }
      s_raw[j * kSparseThreads + tid] = x;
    }
  }
  if (extra >= 0) {
    xraw = ld1<uint32_t>(src + extra * 4);
    xhit = cand(xraw);
    if (BAND) sure += above(xraw);
  }
  // this thread's place among the warp's candidates
  const uint32_t c = __popc(mask) + (xhit ? 1u : 0u);
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t wtotal = __shfl_sync(0xFFFFFFFFu, incl, 31);
  unsigned wsure = 0;
  if (BAND) wsure = __reduce_add_sync(0xFFFFFFFFu, (unsigned)(sure + __popc(hmask)));
  // the tile's counters s_n[par], s_sure[par] are zero (cleared by thread 0
  // before the previous tile's last barrier, or before the first tile)
  uint32_t wbase = 0;
  if (lane == 31 && wtotal) wbase = atomicAdd(&s_n[par], wtotal);
  if (BAND && lane == 0 && wsure) atomicAdd(&s_sure[par], wsure);
  wbase = __shfl_sync(0xFFFFFFFFu, wbase, 31);
  __syncthreads();  // every warp has reserved its share of the tile's room
  if (tid == 0) {
    const uint32_t tot = s_n[par];
    const unsigned long long base = tot ? atomicAdd(p.cand_n + r, (unsigned long long)tot) : 0ull;
    s_base = base;
    if (BAND && s_sure[par]) atomicAdd(p.cand_n + p.W + r, (unsigned long long)s_sure[par]);
    p.tilecnt[(int64_t)r * p.tiles_per_rank + tile] = tot;
    p.chunk[(int64_t)r * p.tiles_per_rank + tile] = (uint32_t)base;
    s_n[par ^ 1] = 0;  // for the next tile (last read by this thread, a tile ago)
    s_sure[par ^ 1] = 0;
  }
  __syncthreads();
  const unsigned long long cap = (unsigned long long)p.cand_cap;
  const unsigned long long pos0 = s_base + wbase + (incl - c);
  uint32_t* ckey = p.cand_key + (int64_t)r * p.cand_cap + pos0;
  uint32_t* cidx = p.cand_idx + (int64_t)r * p.cand_cap + pos0;
  // entry j of this thread sits at offset off of the tile's body both in
  // s_raw and in the array (list indices are 32-bit)
  const uint32_t ibase = (uint32_t)(vec ? av : t0);
  auto offset = [&](int j) -> uint32_t {
    return vec ? (uint32_t)(((j >> 2) * kSparseThreads + tid) * 4 + (j & 3))
               : (uint32_t)(j * kSparseThreads + tid);
  };
  if (pos0 + c <= cap) {  // the usual case: all of this thread's entries fit
    uint32_t k = 0;
    for (uint32_t m = mask; m; m &= m - 1u, ++k) {
      const uint32_t off = offset(__ffs(m) - 1);
      ckey[k] = order_key(__uint_as_float(s_raw[off]));
      cidx[k] = ibase + off;
    }
    if (xhit) {
      ckey[k] = order_key(__uint_as_float(xraw));
      cidx[k] = (uint32_t)extra;
    }
  } else {
    uint32_t k = 0;
    for (uint32_t m = mask; m; m &= m - 1u, ++k) {
      if (pos0 + k >= cap) break;
      const uint32_t off = offset(__ffs(m) - 1);
      ckey[k] = order_key(__uint_as_float(s_raw[off]));
      cidx[k] = ibase + off;
    }
    if (xhit && pos0 + k < cap) {
      ckey[k] = order_key(__uint_as_float(xraw));
      cidx[k] = (uint32_t)extra;
    }
  }
  // (on to the next tile without a barrier: only thread 0 reads s_n and
  // s_sure, the next tile's warps add to the other pair, s_base changes only
  // after the next tile's first barrier, which every thread passes after its
  // reads above, and each thread reads only its own slots of s_raw)
}

// The candidate pass without accumulations reads one array per rank, and its
// cost per tile is latency -- the tile's loads, then the list reservation (a
// global atomic round trip behind two barriers) -- more than bytes.  So this
// form keeps as many tiles in flight as it can: 32 registers and 16 KiB of
// shared memory per 256-thread CTA give 8 CTAs per SM (the form with
// accumulations needs 40 registers and gets 6).  It spends few instructions
// per entry: the band test is one integer compare on the raw fp32 bits per
// bound, the count above the band runs only when there is one, and keys are
// formed only for the listed entries.  Every warp's shared-memory stores are
// contiguous (vector u of all threads side by side).  The grid covers a
// quarter of the tiles and each CTA loops over four, so its setup (state,
// bounds, pointers) is paid once for four tiles (per call at W = 8, 2^26 per
// rank: one tile per CTA 0.813 ms, two 0.803, four 0.800).
// BANDED: launched on the band route, where a rank may have an upper bound;
// the list route's form holds only the bodies without one (a smaller kernel
// measured 3-4 us faster per call at W = 8, 2^26).
template <bool BANDED>
__global__ void __launch_bounds__(256, 8) vc_topk_filter_raw(const __grid_constant__ SparseParams p) {
  pdl_enter();
  __shared__ __align__(16) uint32_t s_raw[kSparseThreads * 4 * kTileVecs];
  __shared__ uint32_t s_n[2], s_sure[2];  // per tile, alternating
  __shared__ unsigned long long s_base;
  const int r = blockIdx.y;
  if (threadIdx.x < 2) {
    s_n[threadIdx.x] = 0;
    s_sure[threadIdx.x] = 0;
  }
  __syncthreads();
  const uint32_t topkey = p.state[r].topkey;
  const bool band = topkey != 0xFFFFFFFFu;  // uniform per CTA
  const RawBound lo = raw_bound(p.state[r].lowkey);
  // above the band: key >= topkey + 1 (so only with a band)
  const RawBound hi = raw_bound(band ? topkey + 1 : 0xFFFFFFFFu);
  int par = 0;
  const int hmode = band ? (hi.sgn ? 2 : 1) : 0;  // the upper bound's compare form
  for (int64_t tile = blockIdx.x; tile < p.tiles_per_rank; tile += gridDim.x, par ^= 1) {
    if (!BANDED) {  // no upper bound on the list route
      if (lo.sgn)
        filter_tile_raw<true, 0>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
      else
        filter_tile_raw<false, 0>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
    } else if (lo.sgn) {
      if (hmode == 2)
        filter_tile_raw<true, 2>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
      else if (hmode == 1)  // (not reached: a bound above a signed-form one is signed-form)
        filter_tile_raw<true, 1>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
      else
        filter_tile_raw<true, 0>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
    } else {
      if (hmode == 2)
        filter_tile_raw<false, 2>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
      else if (hmode == 1)
        filter_tile_raw<false, 1>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
      else
        filter_tile_raw<false, 0>(p, r, tile, lo, hi, s_raw, s_n, s_sure, par, s_base);
    }
  }
}

// Histogram of digit P over a rank's candidate list: P = 0, 1, 2 the key
// digits (as vc_topk_hist), P = 3, 4, 5 the digits of the inverted index of
// the candidates whose key equals T.  Ranks on the full path count nothing;
// an overflowed list counts nothing at P = 0, so the selection sends the
// rank to the full path.
template <int P>
__global__ void __launch_bounds__(256) vc_topk_cand_hist(const __grid_constant__ SparseParams p) {
  pdl_enter();
  __shared__ uint32_t h[kTopkBins];
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const TopkState& st = p.state[r];
  // uniform per CTA
  if (st.full) return;
  if (P >= 3 && (st.need >= st.equal || st.tie_resolved)) return;
  const unsigned long long cn = p.cand_n[r];
  if (cn > (unsigned long long)p.cand_cap) return;
  for (int i = tid; i < kTopkBins; i += blockDim.x) h[i] = 0;
  const uint32_t prefix = st.prefix, T = st.T;
  const uint32_t* ckey = p.cand_key + (int64_t)r * p.cand_cap;
  const uint32_t* cidx = p.cand_idx + (int64_t)r * p.cand_cap;
  __syncthreads();
  auto count = [&](bool in_list, uint32_t key, int64_t i) {  // every lane calls it
    bool valid = false;
    uint32_t d = 0;
    if (in_list) {
      if (P <= 2) {
        valid = digit_of<P>(key, prefix, d);
      } else if (key == T) {
        valid = index_digit_of<P>(~cidx[i], prefix, d);
      }
    }
    // the first digit clusters (combine equal bins across the warp); the
    // later digits spread over the bins, where plain atomics are cheaper
    if (P == 0)
      hist_add(h, valid, d);
    else if (valid)
      atomicAdd(&h[d], 1u);
  };
  // keys four at a time (the list starts 16-byte aligned), U vectors per
  // thread loaded before any is counted; then the last m % 4 keys
  constexpr int U = 4;
  const int64_t m = (int64_t)cn, m4 = m / 4;
  const uint4* k4 = reinterpret_cast<const uint4*>(ckey);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < m4; base += stride * U) {
    uint4 kv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + u * stride + tid;
      kv[u] = v < m4 ? k4[v] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + u * stride + tid;
      const bool ok = v < m4;
      count(ok, kv[u].x, v * 4);
      count(ok, kv[u].y, v * 4 + 1);
      count(ok, kv[u].z, v * 4 + 2);
      count(ok, kv[u].w, v * 4 + 3);
    }
  }
  if (blockIdx.x == 0 && tid < 32) {
    const int64_t i = m4 * 4 + tid;
    count(i < m, i < m ? ckey[i] : 0u, i);
  }
  __syncthreads();
  for (int i = tid; i < kTopkBins; i += blockDim.x)
    if (h[i]) atomicAdd(&p.hist[(int64_t)r * kTopkBins + i], h[i]);
}

// ------------------------------------------------------------- list ties
// Keys equal to the K-th one (T) straddling the cut on the candidate path:
// the kept ones are the `need` lowest indices among the candidates whose key
// is T, so the boundary is the need-th smallest such index.  When there are
// at most kTieCap equal keys (at W = 8, 2^26 per rank and K = 1 % a handful
// of fp32 keys repeat on most calls), one pass finds it: every CTA scans its
// share of the rank's list and appends the indices of the equal keys to a
// small buffer (the first kTieCap slots of the rank's histogram, zero at
// this point); the last CTA of the rank to finish (a counter, no waiting)
// ranks them by counting the smaller ones, sets the boundary, marks the rank
// resolved and clears the slots.  More equal keys (massive ties, such as
// quantised values) are left to the three index-digit passes that follow,
// which skip resolved ranks.
constexpr uint32_t kTieCap = 256;

__global__ void __launch_bounds__(256) vc_topk_ties(const __grid_constant__ SparseParams p) {
  pdl_enter();
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  TopkState* st = p.state + r;
  // uniform per rank: nothing to resolve, the rank is on the full path, or
  // too many equal keys for the buffer
  if (p.K == 0 || st->full || st->need >= st->equal) return;
  if ((unsigned long long)st->equal > kTieCap) return;
  const unsigned long long cn = p.cand_n[r];
  if (cn > (unsigned long long)p.cand_cap) return;
  const int64_t m = (int64_t)cn;
  const uint32_t T = st->T;
  const uint32_t* ckey = p.cand_key + (int64_t)r * p.cand_cap;
  const uint32_t* cidx = p.cand_idx + (int64_t)r * p.cand_cap;
  uint32_t* slots = p.hist + (int64_t)r * kTopkBins;  // zero here
  auto take = [&](uint32_t key, int64_t i) {
    if (key == T) {
      const uint32_t pos = atomicAdd(&st->tie_n, 1u);
      if (pos < kTieCap) slots[pos] = cidx[i];
    }
  };
  // keys four at a time (the list starts 16-byte aligned), U vectors per
  // thread loaded before any is tested; then the last m % 4 keys
  constexpr int U = 4;
  const int64_t m4 = m / 4;
  const uint4* k4 = reinterpret_cast<const uint4*>(ckey);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < m4; base += stride * U) {
    uint4 kv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + u * stride + tid;
      kv[u] = v < m4 ? k4[v] : make_uint4(~T, ~T, ~T, ~T);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + u * stride + tid;
      take(kv[u].x, v * 4);
      take(kv[u].y, v * 4 + 1);
      take(kv[u].z, v * 4 + 2);
      take(kv[u].w, v * 4 + 3);
    }
  }
  if (blockIdx.x == 0 && tid < 4 && m4 * 4 + tid < m) take(ckey[m4 * 4 + tid], m4 * 4 + tid);
  // the last CTA of this rank to get here resolves it
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&st->tie_done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int64_t need = st->need;
  const uint32_t cnt = *(volatile uint32_t*)&st->tie_n;  // == equal <= kTieCap
  __shared__ uint32_t s_idx[kTieCap];
  for (uint32_t i = tid; i < cnt && i < kTieCap; i += blockDim.x)
    s_idx[i] = *(volatile uint32_t*)&slots[i];
  __syncthreads();
  for (uint32_t i = tid; i < cnt && i < kTieCap; i += blockDim.x) {
    uint32_t below = 0;
    for (uint32_t j = 0; j < cnt && j < kTieCap; ++j) below += s_idx[j] < s_idx[i];
    if ((int64_t)below == need - 1) st->boundary = (int64_t)s_idx[i];
    slots[i] = 0;
  }
  if (tid == 0) st->tie_resolved = 1;
}

// ------------------------------------------------------------- list route
// The result comes from the candidate lists when every rank's K kept entries
// are listed: the lists were usable (no rank sent to the whole-array
// passes) and had no entries above the band.  Uniform over the grid.  The
// output pass then reads, per tile, each rank's list entries of that tile
// instead of the whole arrays.  (Final once the first-digit selection has
// run: no later pass sends a rank to the full path.)
__device__ __forceinline__ bool list_route(const SparseParams& p) {
  if (!p.list_out) return false;
  for (int r = 0; r < p.W; ++r)
    if (p.state[r].full) return false;
  return true;
}

// After the first selection, when the result will not come from the lists
// (a rank's list overflowed or missed its K-th key): the passes that follow
// read x from the accumulations, so the residuals the candidate pass wrote
// for settled entries are undone from the lists (x is the key's value; an
// entry of a tile that was not wholly listed holds x already, and writing it
// again changes nothing).  grid.y = rank.
__global__ void __launch_bounds__(256) vc_topk_restore(const __grid_constant__ SparseParams p) {
  pdl_enter();
  if (!p.list_out || !p.has_acc || list_route(p)) return;  // uniform over the grid
  const int r = blockIdx.y;
  const uint32_t setkey = settled_key(p, r);
  if (setkey == 0xFFFFFFFFu) return;
  const unsigned long long cn = p.cand_n[r], cap = (unsigned long long)p.cand_cap;
  const int64_t m = (int64_t)(cn < cap ? cn : cap);
  const uint32_t* ckey = p.cand_key + (int64_t)r * p.cand_cap;
  const uint32_t* cidx = p.cand_idx + (int64_t)r * p.cand_cap;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < m;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t k = ckey[i];
    if (k > setkey) st1((char*)p.acc[r] + (int64_t)cidx[i] * 4, __float_as_uint(key_value(k)));
  }
}

// List route output pass (one CTA per tile; the dense apply pass returns at
// once on this route): the lists hold every kept entry, grouped by tile, so
// each tile's kept entries are folded into zeros in shared memory, rank after
// rank, their accumulations (which hold x, or already the residual above the
// settled key) become x - (0 + x), and the tile is written to every output.
// Each thread loads its entry of eight ranks' chunks before folding them, so
// a tile costs one round trip for the chunk bounds and one per eight ranks
// for the entries; the first tile's chunk bounds come in the same round trip
// as the ranks' states (the route, the cut), loaded before the route is
// known (the workspace holds them either way).  Those round trips are
// latency the tile's writes cannot hide, so the kernel is held to 32
// registers (32-bit list indices) for 8 CTAs per SM.
__global__ void __launch_bounds__(256, 8) vc_topk_list_out(const __grid_constant__ SparseParams p) {
  pdl_enter();
  if (!p.list_out) return;
  __shared__ uint32_t s_T[VCOLL_MAX_RANKS], s_set[VCOLL_MAX_RANKS];
  __shared__ long long s_bound[VCOLL_MAX_RANKS];
  __shared__ uint32_t s_cnt4[VCOLL_MAX_RANKS];
  __shared__ int64_t s_c0[VCOLL_MAX_RANKS];
  const int W = p.W;
  const int tid = threadIdx.x;
  auto chunk_bounds = [&](int r, int64_t tile) {
    s_cnt4[r] = p.tilecnt[(int64_t)r * p.tiles_per_rank + tile];
    s_c0[r] = (int64_t)r * p.cand_cap + p.chunk[(int64_t)r * p.tiles_per_rank + tile];
  };
  bool full = false;  // a rank on the full path: the lists do not hold the result
  for (int r = tid; r < W; r += blockDim.x) {
    const TopkState& st = p.state[r];
    full |= st.full != 0;
    s_T[r] = st.T;
    s_bound[r] = st.boundary;
    s_set[r] = settled_key(p, r);
    chunk_bounds(r, blockIdx.x);  // (grid <= tiles)
  }
  if (__syncthreads_or(full)) return;  // the route, uniform over the grid
  constexpr int R = 8;  // ranks whose list entries are loaded together
  // the tile's sums, shifted by pad (0-3) so that the aligned body starts on
  // a 16-byte boundary of shared memory
  __shared__ __align__(16) float s_res[kSparseTileElems + 4];
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const int64_t t0 = tile * p.tile_elems;
    const int64_t t1 = t0 + p.tile_elems < p.n ? t0 + p.tile_elems : p.n;
    int64_t av = t0, bv = t0;
    if (p.phase >= 0) aligned_body<4>(t0, t1, p.phase, av, bv);
    const int64_t base = t0 - ((4 - ((av - t0) & 3)) & 3);  // s_res[i - base] holds entry i
    for (int j = tid; j < kSparseTileElems + 4; j += blockDim.x) s_res[j] = 0.0f;
    if (tile != blockIdx.x)
      for (int r = tid; r < W; r += blockDim.x) chunk_bounds(r, tile);
    __syncthreads();
    // (an entry above the settled key already holds its residual: only a
    // settled entry that is not kept after all gets x back)
    auto fold = [&](int r, uint32_t key, int64_t idx) {
      if (key > s_T[r] || (key == s_T[r] && idx <= s_bound[r])) {
        const float x = key_value(key);
        s_res[idx - base] = __fadd_rn(x, s_res[idx - base]);
        if (p.has_acc && key <= s_set[r]) st1((char*)p.acc[r] + idx * 4, kept_residual_bits(key));
      } else if (p.has_acc && key > s_set[r]) {
        st1((char*)p.acc[r] + idx * 4, __float_as_uint(key_value(key)));
      }
    };
    for (int g = 0; g < W; g += R) {
      // entry tid of the chunks of ranks g .. g + R - 1, loaded together
      uint32_t pk[R];
      uint32_t pi[R];  // list indices are 32-bit; 0xFFFFFFFF: none
#pragma unroll
      for (int q = 0; q < R; ++q) {
        pk[q] = 0;
        pi[q] = 0xFFFFFFFFu;
        if (g + q < W && (uint32_t)tid < s_cnt4[g + q]) {
          pk[q] = p.cand_key[s_c0[g + q] + tid];
          pi[q] = p.cand_idx[s_c0[g + q] + tid];
        }
      }
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int r = g + q;
        if (r >= W) break;
        if (pi[q] != 0xFFFFFFFFu) fold(r, pk[q], (int64_t)pi[q]);
        for (uint32_t j = tid + blockDim.x; j < s_cnt4[r]; j += blockDim.x)
          fold(r, p.cand_key[s_c0[r] + j], p.cand_idx[s_c0[r] + j]);
        __syncthreads();  // rank order: rank r's adds land before rank r + 1's
      }
    }
    const int64_t nv = (bv - av) / 4;
    for (int64_t v = tid; v < nv; v += blockDim.x) {
      const uint4 o = *reinterpret_cast<const uint4*>(&s_res[av + v * 4 - base]);
      for (int u = 0; u < W; ++u) st_stream((char*)p.out[u] + (av + v * 4) * 4, o);
    }
    const int64_t head = av - t0, tail = t1 - bv;
    for (int64_t j = tid; j < head + tail; j += blockDim.x) {
      const int64_t i = j < head ? t0 + j : bv + (j - head);
      for (int u = 0; u < W; ++u) st1((char*)p.out[u] + i * 4, __float_as_uint(s_res[i - base]));
    }
    __syncthreads();  // s_res is reused by the next tile
  }
  if (p.nnz && blockIdx.x == 0)
    for (int r = tid; r < W; r += blockDim.x) p.nnz[r] = p.K;  // exactly K kept per rank
}

// -------------------------------------------------------------------- apply
// One pass: survivors, error feedback, rank-order sum written to every rank,
// survivor counts per rank.
template <int TOPK>
__global__ void __launch_bounds__(256) vc_sparse_apply(const __grid_constant__ SparseParams p) {
  pdl_enter();
  __shared__ uint32_t s_T[VCOLL_MAX_RANKS];
  __shared__ long long s_bound[VCOLL_MAX_RANKS];
  __shared__ unsigned long long s_cnt[VCOLL_MAX_RANKS];
  const int W = p.W;
  const int tid = threadIdx.x;
  for (int r = tid; r < W; r += blockDim.x) {
    if (TOPK && p.K > 0) {  // with K == 0 no selection ran and nothing survives
      s_T[r] = p.state[r].T;
      s_bound[r] = p.state[r].boundary;
    }
    s_cnt[r] = 0;
  }
  __syncthreads();
  // xb: the bits of x (the top-K key is taken from the bits themselves, so a
  // NaN keeps its place in the key order)
  auto keep = [&](int r, uint32_t xb, int64_t i) -> bool {
    if (TOPK) {
      if (p.K == 0) return false;
      const uint32_t k = key_of_bits(xb);
      return k > s_T[r] || (k == s_T[r] && i <= s_bound[r]);
    }
    const float x = __uint_as_float(xb);
    return fabsf(x) > p.threshold && x != 0.0f;
  };
  // the value the residual subtracts: top-K scatters the sent values into
  // zeros first (0 + x, which turns -0 into +0), threshold mode subtracts x
  auto sent = [&](float x) -> float { return TOPK ? __fadd_rn(0.0f, x) : x; };
  auto count = [&](int r, int c) {
    // per-warp sum of this rank's survivors, one shared atomic per warp
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if ((tid & 31) == 0 && c) atomicAdd(&s_cnt[r], (unsigned long long)c);
  };
  if (TOPK && list_route(p)) return;  // vc_topk_list_out writes the result
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    const int64_t t0 = tile * p.tile_elems;
    const int64_t t1 = t0 + p.tile_elems < p.n ? t0 + p.tile_elems : p.n;
    int64_t av = t0, bv = t0;
    if (p.phase >= 0) aligned_body<4>(t0, t1, p.phase, av, bv);
    const int64_t nv = (bv - av) / 4;
    for (int64_t base = 0; base < nv; base += blockDim.x) {
      const int64_t v = base + tid;
      const bool in_range = v < nv;
      const int64_t e = av + v * 4;
      float res[4] = {0.f, 0.f, 0.f, 0.f};
      for (int r = 0; r < W; ++r) {
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        int c = 0;
        if (in_range) {
          load_x4(p, r, e, x);
          float s[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const bool k = keep(r, __float_as_uint(x[q]), e + q);
            s[q] = k ? sent(x[q]) : 0.0f;
            if (k) res[q] = __fadd_rn(x[q], res[q]);
            c += k;
          }
          if (p.has_acc)
            st_stream((char*)p.acc[r] + e * 4,
                      make_uint4(__float_as_uint(__fsub_rn(x[0], s[0])),
                                 __float_as_uint(__fsub_rn(x[1], s[1])),
                                 __float_as_uint(__fsub_rn(x[2], s[2])),
                                 __float_as_uint(__fsub_rn(x[3], s[3]))));
        }
        if (p.nnz) count(r, c);
      }
      if (in_range) {
        const uint4 o = make_uint4(__float_as_uint(res[0]), __float_as_uint(res[1]),
                                   __float_as_uint(res[2]), __float_as_uint(res[3]));
        for (int r = 0; r < W; ++r) st_stream((char*)p.out[r] + e * 4, o);
      }
    }
    // the elements outside whole vectors (all of the tile when the phases
    // differ), one per thread
    const int64_t head = av - t0, tail = t1 - bv;
    for (int64_t base = 0; base < head + tail; base += blockDim.x) {
      const int64_t j = base + tid;
      const bool in_range = j < head + tail;
      const int64_t i = j < head ? t0 + j : bv + (j - head);
      float res = 0.0f;
      for (int r = 0; r < W; ++r) {
        int c = 0;
        if (in_range) {
          const float x = load_x(p, r, i);
          const bool k = keep(r, __float_as_uint(x), i);
          const float s = k ? sent(x) : 0.0f;
          if (k) res = __fadd_rn(x, res);
          c = k;
          if (p.has_acc) st1((char*)p.acc[r] + i * 4, __float_as_uint(__fsub_rn(x, s)));
        }
        if (p.nnz) count(r, c);
      }
      if (in_range)
        for (int r = 0; r < W; ++r) st1((char*)p.out[r] + i * 4, __float_as_uint(res));
    }
  }
  __syncthreads();
  if (p.nnz)
    for (int r = tid; r < W; r += blockDim.x)
      if (s_cnt[r]) atomicAdd((unsigned long long*)&p.nnz[r], s_cnt[r]);
}

const void* sparse_apply_kernel(int topk) {
  return topk ? (const void*)&vc_sparse_apply<1> : (const void*)&vc_sparse_apply<0>;
}
const void* topk_sample_kernel() { return (const void*)&vc_topk_hist<3>; }
const void* topk_select_low_kernel() { return (const void*)&vc_topk_select<3>; }
const void* topk_sample2_kernel() { return (const void*)&vc_topk_hist<5>; }
const void* topk_select_refine_kernel() { return (const void*)&vc_topk_select<8>; }
const void* topk_redo_hist_kernel() { return (const void*)&vc_topk_hist<4>; }
const void* topk_redo_select_kernel() { return (const void*)&vc_topk_select<4>; }
const void* topk_hist_kernel(int pass) {
  return pass == 0 ? (const void*)&vc_topk_hist<0>
                   : pass == 1 ? (const void*)&vc_topk_hist<1> : (const void*)&vc_topk_hist<2>;
}
const void* topk_select_kernel(int pass) {
  return pass == 0 ? (const void*)&vc_topk_select<0>
                   : pass == 1 ? (const void*)&vc_topk_select<1> : (const void*)&vc_topk_select<2>;
}
const void* topk_filter_kernel(int has_acc, int band) {
  if (has_acc) return (const void*)&vc_topk_filter<true>;
  return band ? (const void*)&vc_topk_filter_raw<true> : (const void*)&vc_topk_filter_raw<false>;
}
const void* topk_list_out_kernel() { return (const void*)&vc_topk_list_out; }
const void* topk_restore_kernel() { return (const void*)&vc_topk_restore; }
const void* topk_cand_hist_kernel(int pass) {
  switch (pass) {
    case 0: return (const void*)&vc_topk_cand_hist<0>;
    case 1: return (const void*)&vc_topk_cand_hist<1>;
    case 2: return (const void*)&vc_topk_cand_hist<2>;
    case 3: return (const void*)&vc_topk_cand_hist<3>;
    case 4: return (const void*)&vc_topk_cand_hist<4>;
    default: return (const void*)&vc_topk_cand_hist<5>;
  }
}
const void* topk_index_select_kernel(int pass) {
  return pass == 3 ? (const void*)&vc_topk_select<5>
                   : pass == 4 ? (const void*)&vc_topk_select<6> : (const void*)&vc_topk_select<7>;
}
const void* topk_tie_count_kernel() { return (const void*)&vc_topk_tie_count; }
const void* topk_tie_find_kernel() { return (const void*)&vc_topk_tie_find; }
const void* topk_ties_kernel() { return (const void*)&vc_topk_ties; }

}  // namespace vcoll

/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for virtual-rank ring
 * reduce-scatter / allgather / allreduce and Horovod-style tensor fusion.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * checked against.  It shares no code, header, table or helper with the
 * library under collective_reduction_virtual_gb300/, and the library never
 * loads it.  Only the tests, the smoke check in __graft_entry__.py and the CPU
 * baseline / reference arm of bench.py may load liboracle.so.
 *
 * Every routine here follows its source step by step; nothing is blocked,
 * fused or reordered beyond what that source states:
 *
 *  - Ring reduce-scatter: early NCCL "src/reduce_scatter.cu" (pytorch mirror),
 *    GetBlock() and ReduceScatterKernel(): at step 0 every ring position copies
 *    one block of its input into the next position's buffer, at steps
 *    1..W-2 it writes NextBuffer = FUNC(ThisBuffer, ThisInput), and at step
 *    W-1 ThisOutput = FUNC(ThisBuffer, ThisInput).  The block handled by ring
 *    position p at step s is userFromRing[(W + p - 1 - s) % W]; the page's
 *    4-GPU table (userFromRing = {1,2,0,3}) is reproduced by
 *    oracle_ring_schedule().  The single-GPU case is a plain copy
 *    (ncclReduceScatterWithTypeAndFunc, nDev == 1) and an empty message is a
 *    no-op (recvcount == 0).
 *  - Allgather: "Distributed primitives" notes, "In practice": AllGather
 *    propagates the reduced segments around the ring; section 2 (All-Gather):
 *    every node ends with the concatenation of all segments.
 *  - Allreduce: same notes, Ring AllReduce = ReduceScatter + AllGather, and
 *    section 1 (All-Reduce): every node ends with the same aggregate.
 *  - Fusion: Horovod "horovod/common/operations.cc": the coordinator's fusion
 *    batching in BackgroundThreadLoop (append responses in order while the
 *    fused size stays <= tensor_fusion_threshold, stop at the first that does
 *    not fit), and PerformOperation's NCCL path (copy each tensor to
 *    buffer + offset with offset += size, allreduce the buffer in place, copy
 *    each tensor back out); Apache SINGA "src/io/communicator.cc",
 *    Communicator::fusedSynch, packs the same way (sendBuffOffset += Size).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - Uneven segments: NCCL only handles n = W * recvcount.  For any n, segment
 *    j starts at j*q + min(j, r) and has q + (j < r) elements, q = n / W,
 *    r = n % W (contiguous, larger segments first).
 *  - Accumulator: fp32 for fp32 and bf16 inputs; bf16 values are widened
 *    exactly, there is no rounding between hops, and one final cast.
 *  - avg: the ring sum multiplied once by fl32(1/W) at the last step.
 *  - max: NaN in either operand gives the canonical quiet NaN; otherwise the
 *    larger operand, and +0 over -0 when they compare equal.
 *  - min (NCCL FuncMin, body not on the page): the mirror image of max --
 *    canonical quiet NaN, otherwise the smaller operand, -0 over +0 on a tie.
 *  - prod (NCCL FuncProd): one IEEE fp32 multiply per hop, accumulator first.
 *  - bf16 output: IEEE round-to-nearest-even from fp32; NaN stays a quiet NaN.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no -ffast-math),
 * so every float add or multiply is one IEEE single-precision operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F16 2

#define ORACLE_SUM 0
#define ORACLE_MAX 1
#define ORACLE_AVG 2
#define ORACLE_MIN 3
#define ORACLE_PROD 4

#define ORACLE_MAX_RANKS 64

/* ---------------------------------------------------------------- helpers */

static int elem_size(int dtype) {
  if (dtype == ORACLE_F32) return 4;
  if (dtype == ORACLE_BF16 || dtype == ORACLE_F16) return 2;
  return 0;
}

/* bf16 holds the upper 16 bits of an fp32 value, so widening is exact. */
static float widen_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* IEEE round-to-nearest-even from fp32 to bf16 by bit arithmetic: add half
 * an ulp of the result (0x7FFF) plus the result's lowest kept bit, then
 * truncate.  A NaN keeps its sign and top payload bits and is made quiet. */
uint16_t oracle_bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* IEEE binary16 from fp32, round to nearest even, with gradual underflow:
 * rebias the exponent; below the normal range shift the 24-bit significand
 * (implicit bit restored) into the 10-bit subnormal field; round on the bits
 * shifted out (above half: up; exactly half: to even); a carry out of the
 * significand moves into the exponent, up to infinity.  NaN stays a quiet
 * NaN with its top payload bits. */
uint16_t oracle_f16_from_f32(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  const uint32_t sign = (x >> 16) & 0x8000u;
  const uint32_t exp = (x >> 23) & 0xFFu;
  uint32_t man = x & 0x7FFFFFu;
  if (exp == 0xFFu) return (uint16_t)(sign | (man ? 0x7E00u | (man >> 13) : 0x7C00u));
  const int e = (int)exp - 127 + 15;
  if (e >= 31) return (uint16_t)(sign | 0x7C00u);
  if (e <= 0) {
    if (e < -10) return (uint16_t)sign; /* below half the smallest subnormal */
    man |= 0x800000u;
    const int shift = 14 - e; /* 14..24 */
    uint32_t r = man >> shift;
    const uint32_t rem = man & ((1u << shift) - 1u);
    const uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (r & 1u))) ++r;
    return (uint16_t)(sign | r);
  }
  uint32_t r = ((uint32_t)e << 10) | (man >> 13);
  const uint32_t rem = man & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) ++r;
  return (uint16_t)(sign | r);
}

/* binary16 -> fp32, exact: normal numbers rebias the exponent, subnormals
 * are scaled by 2^-24, infinities and NaNs keep their class. */
float oracle_f32_from_f16(uint16_t h) {
  const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  const uint32_t exp = (h >> 10) & 0x1Fu;
  const uint32_t man = h & 0x3FFu;
  float f;
  if (exp == 0x1Fu) {
    uint32_t u = sign | 0x7F800000u | (man << 13);
    memcpy(&f, &u, 4);
    return f;
  }
  if (exp == 0) {
    f = ldexpf((float)man, -24);
    return sign ? -f : f;
  }
  uint32_t u = sign | ((exp - 15 + 127) << 23) | (man << 13);
  memcpy(&f, &u, 4);
  return f;
}

static float load_elem(const void* base, int64_t k, int dtype) {
  if (dtype == ORACLE_F32) {
    float v;
    memcpy(&v, (const char*)base + 4 * k, 4);
    return v;
  }
  uint16_t h;
  memcpy(&h, (const char*)base + 2 * k, 2);
  if (dtype == ORACLE_F16) return oracle_f32_from_f16(h);
  return widen_bf16(h);
}

static void store_elem(void* base, int64_t k, int dtype, float v) {
  if (dtype == ORACLE_F32) {
    memcpy((char*)base + 4 * k, &v, 4);
  } else {
    uint16_t h = dtype == ORACLE_F16 ? oracle_f16_from_f32(v) : oracle_bf16_from_f32(v);
    memcpy((char*)base + 2 * k, &h, 2);
  }
}

/* The value a buffer of element type dtype holds after storing v (NCCL keeps
 * the ring's intermediate buffers in the element type T). */
static float round_to(float v, int dtype) {
  if (dtype == ORACLE_F16) return oracle_f32_from_f16(oracle_f16_from_f32(v));
  if (dtype == ORACLE_BF16) return widen_bf16(oracle_bf16_from_f32(v));
  return v;
}

static float canonical_qnan(void) {
  uint32_t u = 0x7FC00000u;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* FUNC of the ring: accumulator first, the rank's own input second. */
static float ring_func(int op, float acc, float x) {
  if (op == ORACLE_MAX) {
    if (isnan(acc) || isnan(x)) return canonical_qnan();
    if (acc > x) return acc;
    if (x > acc) return x;
    /* equal: identical bits, except +0 == -0 where +0 wins */
    if (acc == 0.0f) return (signbit(acc) && signbit(x)) ? -0.0f : 0.0f;
    return acc;
  }
  if (op == ORACLE_MIN) {
    if (isnan(acc) || isnan(x)) return canonical_qnan();
    if (acc < x) return acc;
    if (x < acc) return x;
    /* equal: identical bits, except +0 == -0 where -0 wins */
    if (acc == 0.0f) return (signbit(acc) || signbit(x)) ? -0.0f : 0.0f;
    return acc;
  }
  if (op == ORACLE_PROD) return acc * x;
  return acc + x; /* sum and avg */
}

static int valid_op(int op) {
  return op == ORACLE_SUM || op == ORACLE_MAX || op == ORACLE_AVG || op == ORACLE_MIN ||
         op == ORACLE_PROD;
}

static int check_ring(int W, const int* user_from_ring, int* ufr) {
  int seen[ORACLE_MAX_RANKS];
  memset(seen, 0, sizeof(seen));
  for (int p = 0; p < W; ++p) {
    int u = user_from_ring ? user_from_ring[p] : p;
    if (u < 0 || u >= W || seen[u]) return -1;
    seen[u] = 1;
    ufr[p] = u;
  }
  return 0;
}

/* ---------------------------------------------------------- segmentation */

int oracle_segment(int64_t n, int W, int j, int64_t* off, int64_t* len) {
  if (n < 0 || W < 1 || j < 0 || j >= W || !off || !len) return -1;
  int64_t q = n / W;
  int64_t r = n % W;
  *off = (int64_t)j * q + (j < r ? j : r);
  *len = q + (j < r ? 1 : 0);
  return 0;
}

/* Block handled by ring position p at step s (NCCL GetBlock). */
static int get_block(int p, int s, const int* ufr, int W) {
  return ufr[(W + p - 1 - s) % W];
}

/* table[s * W + p] = block processed by ring position p at step s. */
int oracle_ring_schedule(int W, const int* user_from_ring, int* table) {
  int ufr[ORACLE_MAX_RANKS];
  if (W < 1 || W > ORACLE_MAX_RANKS || !table) return -1;
  if (check_ring(W, user_from_ring, ufr)) return -1;
  for (int s = 0; s < W; ++s)
    for (int p = 0; p < W; ++p) table[s * W + p] = get_block(p, s, ufr, W);
  return 0;
}

/* -------------------------------------------------------- reduce-scatter */

/* in[u]: n elements of user rank u.  out[u]: the len_u elements of segment u.
 * user_from_ring: ring order (NULL = identity).  The ring is simulated
 * step by step: cur[p] is the buffer ring position p received in the previous
 * step (ThisBuffer), nxt[p] what it receives in this step (the previous
 * position's NextBuffer). */
/* hop != 0: every intermediate buffer is rounded to dtype after each FUNC,
 * as in NCCL where ThisBuffer / NextBuffer hold values of the element type T
 * (the fp32-accumulating reading is hop == 0). */
static int ring_reduce_scatter(const void* const* in, void* const* out, int W, int64_t n,
                               int dtype, int op, const int* user_from_ring, int hop);

int oracle_reduce_scatter(const void* const* in, void* const* out, int W, int64_t n,
                          int dtype, int op, const int* user_from_ring) {
  return ring_reduce_scatter(in, out, W, n, dtype, op, user_from_ring, 0);
}

int oracle_reduce_scatter_hop(const void* const* in, void* const* out, int W, int64_t n,
                              int dtype, int op, const int* user_from_ring) {
  return ring_reduce_scatter(in, out, W, n, dtype, op, user_from_ring, 1);
}

static int ring_reduce_scatter(const void* const* in, void* const* out, int W, int64_t n,
                               int dtype, int op, const int* user_from_ring, int hop) {
  int ufr[ORACLE_MAX_RANKS];
  int es = elem_size(dtype);
  if (!in || !out || W < 1 || W > ORACLE_MAX_RANKS || n < 0 || !es) return -1;
  if (!valid_op(op)) return -1;
  if (check_ring(W, user_from_ring, ufr)) return -1;
  if (n == 0) return 0;
  if (W == 1) {
    if (out[0] != in[0]) memcpy(out[0], in[0], (size_t)n * es);
    return 0;
  }
  int64_t off, maxlen;
  oracle_segment(n, W, 0, &off, &maxlen); /* segment 0 is a longest one */
  float* cur = (float*)malloc(sizeof(float) * W * (maxlen ? maxlen : 1));
  float* nxt = (float*)malloc(sizeof(float) * W * (maxlen ? maxlen : 1));
  if (!cur || !nxt) {
    free(cur);
    free(nxt);
    return -2;
  }
  const float scale = 1.0f / (float)W;
  for (int s = 0; s < W; ++s) {
    for (int p = 0; p < W; ++p) {
      int b = get_block(p, s, ufr, W);
      int me = ufr[p]; /* the user rank sitting at ring position p */
      int64_t boff, blen;
      oracle_segment(n, W, b, &boff, &blen);
      const float* this_buffer = cur + (int64_t)p * maxlen;
      float* next_buffer = nxt + (int64_t)((p + 1) % W) * maxlen;
      for (int64_t k = 0; k < blen; ++k) {
        float x = load_elem(in[me], boff + k, dtype);
        if (s == 0) {
          next_buffer[k] = x; /* step 0: copy to the next position */
        } else if (s < W - 1) {
          next_buffer[k] = ring_func(op, this_buffer[k], x);
          if (hop) next_buffer[k] = round_to(next_buffer[k], dtype);
        } else {
          /* step W-1: b == me, the finished block stays here */
          float v = ring_func(op, this_buffer[k], x);
          if (hop) v = round_to(v, dtype);
          if (op == ORACLE_AVG) v = v * scale;
          store_elem(out[me], k, dtype, v);
        }
      }
    }
    float* t = cur;
    cur = nxt;
    nxt = t;
  }
  free(cur);
  free(nxt);
  return 0;
}

/* ------------------------------------------------------------- allgather */

/* in[u]: the len_u elements of segment u held by user rank u.  out[u]: n
 * elements.  At step 0 every position places its own segment; at step s it
 * receives from the previous position the block that one held at step s-1. */
int oracle_allgather(const void* const* in, void* const* out, int W, int64_t n,
                     int dtype, const int* user_from_ring) {
  int ufr[ORACLE_MAX_RANKS];
  int es = elem_size(dtype);
  if (!in || !out || W < 1 || W > ORACLE_MAX_RANKS || n < 0 || !es) return -1;
  if (check_ring(W, user_from_ring, ufr)) return -1;
  if (n == 0) return 0;
  for (int s = 0; s < W; ++s) {
    for (int p = 0; p < W; ++p) {
      int me = ufr[p];
      int b = ufr[(p - s + W) % W];
      int64_t boff, blen;
      oracle_segment(n, W, b, &boff, &blen);
      char* dst = (char*)out[me] + boff * es;
      const char* src;
      if (s == 0)
        src = (const char*)in[me];
      else
        src = (const char*)out[ufr[(p - 1 + W) % W]] + boff * es;
      if (dst != src) memmove(dst, src, (size_t)blen * es);
    }
  }
  return 0;
}

/* Allgather with per-rank sizes (Horovod's allgatherv path: every rank's
 * tensor, first dimensions possibly different, concatenated in rank order on
 * every rank).  in[u]: counts[u] elements; out[u]: the sum of all counts,
 * rank j's piece at counts[0] + ... + counts[j-1].  Same ring propagation as
 * oracle_allgather, with the displacements in place of the even segments. */
int oracle_allgatherv(const void* const* in, const int64_t* counts, void* const* out, int W,
                      int dtype, const int* user_from_ring) {
  int ufr[ORACLE_MAX_RANKS];
  int64_t disp[ORACLE_MAX_RANKS + 1];
  int es = elem_size(dtype);
  if (!in || !out || !counts || W < 1 || W > ORACLE_MAX_RANKS || !es) return -1;
  if (check_ring(W, user_from_ring, ufr)) return -1;
  disp[0] = 0;
  for (int u = 0; u < W; ++u) {
    if (counts[u] < 0) return -1;
    disp[u + 1] = disp[u] + counts[u];
  }
  for (int s = 0; s < W; ++s) {
    for (int p = 0; p < W; ++p) {
      int me = ufr[p];
      int b = ufr[(W + p - s) % W]; /* block held at step s */
      char* dst = (char*)out[me] + disp[b] * es;
      const char* src;
      if (s == 0)
        src = (const char*)in[me];
      else
        src = (const char*)out[ufr[(p - 1 + W) % W]] + disp[b] * es;
      if (dst != src && counts[b]) memmove(dst, src, (size_t)counts[b] * es);
    }
  }
  return 0;
}

/* ------------------------------------------------------------- allreduce */

/* Ring allreduce = reduce-scatter followed by allgather.  in[u], out[u]: n
 * elements each.  The reduce-scatter lands in temporaries, so out may alias
 * in. */
int oracle_allreduce(const void* const* in, void* const* out, int W, int64_t n,
                     int dtype, int op, const int* user_from_ring) {
  int ufr[ORACLE_MAX_RANKS];
  int es = elem_size(dtype);
  if (!in || !out || W < 1 || W > ORACLE_MAX_RANKS || n < 0 || !es) return -1;
  if (!valid_op(op)) return -1;
  if (check_ring(W, user_from_ring, ufr)) return -1;
  if (n == 0) return 0;
  void* seg[ORACLE_MAX_RANKS];
  int64_t off, len;
  int rc = 0;
  for (int u = 0; u < W; ++u) {
    oracle_segment(n, W, u, &off, &len);
    seg[u] = malloc((size_t)(len ? len : 1) * es);
    if (!seg[u]) rc = -2;
  }
  if (!rc) rc = oracle_reduce_scatter(in, seg, W, n, dtype, op, user_from_ring);
  if (!rc) rc = oracle_allgather((const void* const*)seg, out, W, n, dtype, user_from_ring);
  for (int u = 0; u < W; ++u) free(seg[u]);
  return rc;
}

/* Reduced-precision "wire" allreduce (Apache SINGA, Communicator::synchHalf
 * and fusedSynchHalf): fp32 inputs are converted to the wire type (float2half,
 * here fp16 or bf16), allreduced in that type -- an NCCL ring whose buffers
 * hold wire values, so every hop rounds to the wire type -- and converted back
 * to fp32 (half2float).  in[u], out[u]: n fp32 elements. */
int oracle_allreduce_wire(const void* const* in, void* const* out, int W, int64_t n, int wire,
                          int op, const int* user_from_ring) {
  if (!in || !out || W < 1 || W > ORACLE_MAX_RANKS || n < 0) return -1;
  if (wire != ORACLE_F16 && wire != ORACLE_BF16) return -1;
  if (!valid_op(op)) return -1;
  void* win[ORACLE_MAX_RANKS];
  void* seg[ORACLE_MAX_RANKS];
  void* wout[ORACLE_MAX_RANKS];
  int rc = 0;
  for (int u = 0; u < W; ++u) {
    int64_t off, len;
    oracle_segment(n, W, u, &off, &len);
    win[u] = malloc((size_t)(n ? n : 1) * 2);
    wout[u] = malloc((size_t)(n ? n : 1) * 2);
    seg[u] = malloc((size_t)(len ? len : 1) * 2);
    if (!win[u] || !wout[u] || !seg[u]) rc = -2;
  }
  for (int u = 0; !rc && u < W; ++u)
    for (int64_t i = 0; i < n; ++i) store_elem(win[u], i, wire, load_elem(in[u], i, ORACLE_F32));
  if (!rc) rc = oracle_reduce_scatter_hop((const void* const*)win, seg, W, n, wire, op,
                                          user_from_ring);
  if (!rc) rc = oracle_allgather((const void* const*)seg, wout, W, n, wire, user_from_ring);
  for (int u = 0; !rc && u < W; ++u)
    for (int64_t i = 0; i < n; ++i) store_elem(out[u], i, ORACLE_F32, load_elem(wout[u], i, wire));
  for (int u = 0; u < W; ++u) {
    free(win[u]);
    free(wout[u]);
    free(seg[u]);
  }
  return rc;
}

/* ------------------------------------------------- sparsified allreduce */

/* Total order on fp32 values as unsigned keys: larger value, larger key
 * (negative values have their bits inverted, non-negative ones get the sign
 * bit set).  -0 sorts just below +0; NaNs sort beyond the infinities. */
static uint32_t order_key(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

typedef struct {
  uint32_t key;
  int64_t idx; /* 1-based, as SINGA's index arrays */
  float val;
} sparse_entry;

/* "sort the values from large to small" with their indices; equal values
 * keep index order (a stable sort) */
static int by_value_desc(const void* a, const void* b) {
  const sparse_entry* x = (const sparse_entry*)a;
  const sparse_entry* y = (const sparse_entry*)b;
  if (x->key != y->key) return x->key > y->key ? -1 : 1;
  return x->idx < y->idx ? -1 : (x->idx > y->idx ? 1 : 0);
}

/* SINGA Communicator::valSparsAllReduce (topk == 0) and topKSparsAllReduce
 * (topk != 0), over W virtual ranks.  Per rank u, in the page's order:
 *   send = in[u]; with accumulation: send += accum[u], backup = send;
 *   threshold: send[i] = |send[i]| > threshold ? send[i] : 0, the accumulation
 *     becomes backup - send, and the (1-based index, value) list holds the
 *     nonzero entries of send in index order (sparsindex, removezeroidx,
 *     removezeroval);
 *   top-K: K = ceil(threshold * num) in fp32; (index, value) pairs sorted by
 *     value from large to small; the first K are sent; with accumulation it
 *     becomes zero, then gets the K values scattered in (saxpyi), then
 *     backup - itself.
 * The lists are allgathered; every rank's result starts at zero and receives
 * y[idx - 1] += 1.0 * val for the lists of ranks 0, 1, ..., W-1 in turn
 * (cusparseSaxpyi, index base one).  in/out/accum: W arrays of n fp32;
 * accum may be NULL (no error feedback).  nnz (may be NULL) gets each rank's
 * list length. */
int oracle_sparse_allreduce(const void* const* in, void* const* out, void* const* accum, int W,
                            int64_t n, float threshold, int topk, int64_t* nnz) {
  if (!in || !out || W < 1 || W > ORACLE_MAX_RANKS || n < 0) return -1;
  sparse_entry* lists[ORACLE_MAX_RANKS];
  int64_t len[ORACLE_MAX_RANKS];
  float* send = (float*)malloc(sizeof(float) * (size_t)(n ? n : 1));
  float* backup = (float*)malloc(sizeof(float) * (size_t)(n ? n : 1));
  float* result = (float*)malloc(sizeof(float) * (size_t)(n ? n : 1));
  int rc = (send && backup && result) ? 0 : -2;
  for (int u = 0; u < W; ++u) lists[u] = NULL;
  for (int u = 0; !rc && u < W; ++u) {
    float* acc = accum ? (float*)accum[u] : NULL;
    for (int64_t i = 0; i < n; ++i) send[i] = load_elem(in[u], i, ORACLE_F32);
    if (acc) {
      for (int64_t i = 0; i < n; ++i) send[i] = send[i] + acc[i];
      for (int64_t i = 0; i < n; ++i) backup[i] = send[i];
    }
    lists[u] = (sparse_entry*)malloc(sizeof(sparse_entry) * (size_t)(n ? n : 1));
    if (!lists[u]) {
      rc = -2;
      break;
    }
    if (!topk) {
      for (int64_t i = 0; i < n; ++i) send[i] = fabsf(send[i]) > threshold ? send[i] : 0.0f;
      if (acc)
        for (int64_t i = 0; i < n; ++i) acc[i] = backup[i] - send[i];
      int64_t m = 0;
      for (int64_t i = 0; i < n; ++i)
        if (send[i] != 0.0f) {
          lists[u][m].idx = i + 1;
          lists[u][m].val = send[i];
          ++m;
        }
      len[u] = m;
    } else {
      for (int64_t i = 0; i < n; ++i) {
        lists[u][i].idx = i + 1;
        lists[u][i].val = send[i];
        lists[u][i].key = order_key(send[i]);
      }
      qsort(lists[u], (size_t)n, sizeof(sparse_entry), by_value_desc);
      int64_t K = (int64_t)ceilf(threshold * (float)n);
      if (K > n) K = n;
      if (K < 0) K = 0;
      if (acc) {
        for (int64_t i = 0; i < n; ++i) acc[i] = 0.0f;
        for (int64_t k = 0; k < K; ++k) acc[lists[u][k].idx - 1] += 1.0f * lists[u][k].val;
        for (int64_t i = 0; i < n; ++i) acc[i] = backup[i] - acc[i];
      }
      len[u] = K;
    }
    if (nnz) nnz[u] = len[u];
  }
  if (!rc) {
    for (int64_t i = 0; i < n; ++i) result[i] = 0.0f;
    for (int u = 0; u < W; ++u)
      for (int64_t k = 0; k < len[u]; ++k)
        result[lists[u][k].idx - 1] = 1.0f * lists[u][k].val + result[lists[u][k].idx - 1];
    for (int u = 0; u < W; ++u)
      for (int64_t i = 0; i < n; ++i) store_elem(out[u], i, ORACLE_F32, result[i]);
  }
  for (int u = 0; u < W; ++u) free(lists[u]);
  free(send);
  free(backup);
  free(result);
  return rc;
}

/* Allreduce at sampled indices.  vals[i*W + u] is user rank u's input at
 * index idx[i] of an n-element allreduce; result[i] receives the allreduce
 * output there.  Each sample is run through the same ring reduce-scatter on a
 * W-element problem whose segment j (the segment of idx[i] under the full n)
 * holds the sampled values, so the fold order is the one the full problem
 * uses for that segment. */
int oracle_allreduce_sampled(const void* vals, const int64_t* idx, int64_t m, int64_t n,
                             int W, int dtype, int op, const int* user_from_ring,
                             void* result) {
  int es = elem_size(dtype);
  if (!vals || !idx || !result || W < 1 || W > ORACLE_MAX_RANKS || n < 0 || m < 0 || !es)
    return -1;
  char tiny_in[ORACLE_MAX_RANKS][ORACLE_MAX_RANKS * 4];
  char tiny_out[ORACLE_MAX_RANKS][4];
  const void* ip[ORACLE_MAX_RANKS];
  void* op_[ORACLE_MAX_RANKS];
  for (int u = 0; u < W; ++u) {
    ip[u] = tiny_in[u];
    op_[u] = tiny_out[u];
  }
  for (int64_t i = 0; i < m; ++i) {
    if (idx[i] < 0 || idx[i] >= n) return -1;
    int j = -1;
    for (int u = 0; u < W; ++u) {
      int64_t off, len;
      oracle_segment(n, W, u, &off, &len);
      if (idx[i] >= off && idx[i] < off + len) j = u;
    }
    for (int u = 0; u < W; ++u) {
      memset(tiny_in[u], 0, sizeof(tiny_in[u]));
      memcpy(tiny_in[u] + (int64_t)j * es, (const char*)vals + (i * W + u) * es, es);
    }
    int rc = oracle_reduce_scatter(ip, op_, W, W, dtype, op, user_from_ring);
    if (rc) return rc;
    memcpy((char*)result + i * es, tiny_out[j], es);
  }
  return 0;
}

/* ---------------------------------------------------------------- fusion */

/* Greedy batching in tensor order: a batch starts with the next tensor (even
 * one larger than the threshold) and takes following tensors while the fused
 * byte size stays <= threshold_bytes; the first that does not fit starts the
 * next batch, none is skipped.  batch_begin[0..nb] gets the first tensor of
 * each batch and T at the end. */
int oracle_fuse_plan(const int64_t* counts, int T, int dtype, int64_t threshold_bytes,
                     int* batch_begin, int* nbatches) {
  int es = elem_size(dtype);
  if (!counts || !batch_begin || !nbatches || T < 0 || !es || threshold_bytes < 0) return -1;
  for (int t = 0; t < T; ++t)
    if (counts[t] < 0) return -1;
  int nb = 0;
  int t = 0;
  while (t < T) {
    batch_begin[nb++] = t;
    int64_t size = counts[t] * es;
    ++t;
    while (t < T && size + counts[t] * es <= threshold_bytes) {
      size += counts[t] * es;
      ++t;
    }
  }
  batch_begin[nb] = T;
  *nbatches = nb;
  return 0;
}

/* tensors[u*T + t]: tensor t of user rank u, counts[t] elements.  fused[u]
 * receives the T tensors back to back with no padding. */
int oracle_fuse_pack(const void* const* tensors, const int64_t* counts, int T,
                     void* const* fused, int W, int dtype) {
  int es = elem_size(dtype);
  if (!tensors || !counts || !fused || W < 1 || T < 0 || !es) return -1;
  for (int u = 0; u < W; ++u) {
    int64_t offset = 0;
    for (int t = 0; t < T; ++t) {
      memcpy((char*)fused[u] + offset * es, tensors[(int64_t)u * T + t], (size_t)counts[t] * es);
      offset += counts[t];
    }
  }
  return 0;
}

int oracle_fuse_unpack(const void* const* fused, const int64_t* counts, int T,
                       void* const* tensors, int W, int dtype) {
  int es = elem_size(dtype);
  if (!tensors || !counts || !fused || W < 1 || T < 0 || !es) return -1;
  for (int u = 0; u < W; ++u) {
    int64_t offset = 0;
    for (int t = 0; t < T; ++t) {
      memcpy(tensors[(int64_t)u * T + t], (const char*)fused[u] + offset * es, (size_t)counts[t] * es);
      offset += counts[t];
    }
  }
  return 0;
}

/* Whole tensor-fusion allreduce: plan the batches, then per batch pack into
 * the per-rank fusion buffers fused[u] (each at least the largest batch),
 * allreduce them in place, and unpack into outs[u*T + t].  Horovod reduces a
 * one-tensor batch directly instead of through the buffer; with the same
 * segmentation that gives the same values, so every batch goes through the
 * buffer here. */
int oracle_fusion_allreduce(const void* const* ins, void* const* outs, const int64_t* counts,
                            int T, int W, int dtype, int op, int64_t threshold_bytes,
                            void* const* fused) {
  int es = elem_size(dtype);
  if (!ins || !outs || !counts || !fused || W < 1 || W > ORACLE_MAX_RANKS || T < 0 || !es)
    return -1;
  int* begin = (int*)malloc(sizeof(int) * (T + 1));
  if (!begin) return -2;
  int nb = 0;
  int rc = oracle_fuse_plan(counts, T, dtype, threshold_bytes, begin, &nb);
  const void** bin = (const void**)malloc(sizeof(void*) * (size_t)W * (T ? T : 1));
  void** bout = (void**)malloc(sizeof(void*) * (size_t)W * (T ? T : 1));
  if (!bin || !bout) rc = -2;
  for (int b = 0; !rc && b < nb; ++b) {
    int t0 = begin[b], nt = begin[b + 1] - begin[b];
    int64_t total = 0;
    for (int t = t0; t < t0 + nt; ++t) total += counts[t];
    for (int u = 0; u < W; ++u)
      for (int t = 0; t < nt; ++t) {
        bin[(int64_t)u * nt + t] = ins[(int64_t)u * T + t0 + t];
        bout[(int64_t)u * nt + t] = outs[(int64_t)u * T + t0 + t];
      }
    rc = oracle_fuse_pack(bin, counts + t0, nt, fused, W, dtype);
    if (!rc) rc = oracle_allreduce((const void* const*)fused, fused, W, total, dtype, op, NULL);
    if (!rc) rc = oracle_fuse_unpack((const void* const*)fused, counts + t0, nt, bout, W, dtype);
  }
  free(begin);
  free(bin);
  free(bout);
  return rc;
}

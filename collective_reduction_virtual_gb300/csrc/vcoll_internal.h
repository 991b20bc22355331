// Internal interface between the host entry points (api.cpp) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>

#include "../../include/vcoll.h"

#ifdef __CUDACC__
#define VCOLL_HD __host__ __device__
#else
#define VCOLL_HD
#endif

namespace vcoll {

enum Kind : int { KIND_RS = 0, KIND_AR = 1 };

// Parameters of one reduce-scatter / allreduce launch.  The whole struct is a
// __grid_constant__ kernel parameter (about 1.1 KB).
//
// Index space: element i in [0, n) of every rank.  Segment j is
// [j*q + min(j, r), ... + q + (j < r)).  nseg == W splits the work by segment
// (ring order, and always for reduce-scatter); nseg == 1 treats [0, n) as one
// range (allreduce in the fastest order).
//
// Vector path: element i is 16-byte aligned in every buffer iff
// (i + phase) % V == 0, V = 16 / elemsize.  Segment bodies are processed in
// tiles of tile_elems elements (tiles_per_seg per segment); the unaligned head
// and tail of each segment (< V elements each) are done by tile 0.
struct ReduceParams {
  const void* in[VCOLL_MAX_RANKS];
  void* out[VCOLL_MAX_RANKS];
  int64_t n;
  int64_t q;
  int64_t r;
  int64_t tiles_per_seg;
  int64_t num_tiles;
  int64_t tile_elems;
  int W;
  int nseg;
  int phase;
  int ring;      // 1: ring order (segment j's fold starts at ring_start[j]); 0: fastest order
  float scale;   // fl32(1/W) for avg
  int do_scale;
  // realigning kernels: address mod 16 of input u's element 0, and of
  // element 0 on the output grid of segment j (the allreduce's outputs
  // share one grid)
  uint8_t in_phase[VCOLL_MAX_RANKS];
  uint8_t out_phase[VCOLL_MAX_RANKS];
  // the same for W <= 8 as a table: wshift[j * 8 + u] = (in_phase[u] -
  // out_phase[j]) mod 16, input u's bytes past segment j's grid
  uint8_t wshift[64];
  // ring order: the input (in[] index) whose value starts segment j's fold;
  // the fold then takes in[ring_start[j] + 1], ... (mod W), so it ends at
  // ring_start[j] - 1.  With the identity ring ring_start[j] = (j + 1) mod W;
  // for NCCL's userFromRing permutation the host orders in[] by ring
  // position and sets ring_start[j] to the position after rank j's
  uint8_t ring_start[VCOLL_MAX_RANKS];
};

// Parameters of one allgather launch.  in[j] holds piece j, which lands at
// [disp[j], disp[j+1]) of every output (the even segments for allgather,
// per-rank counts for allgatherv).
struct GatherParams {
  const void* in[VCOLL_MAX_RANKS];
  void* out[VCOLL_MAX_RANKS];
  int64_t disp[VCOLL_MAX_RANKS + 1];
  int64_t tiles_per_seg;
  int64_t num_tiles;
  int64_t tile_elems;
  int W;
  int phase;
  // piece j's source sits ishift[j] bytes past the output grid's 16-byte
  // boundaries (the vector grid follows the outputs)
  uint8_t ishift[VCOLL_MAX_RANKS];
};

// Fusion pack / unpack.  One launch copies up to kFuseMaxTensors tensors of
// every rank.  Copy (t, u) moves count[t] elements between tensor[t * W + u]
// (tensor-major) and fused[u] + offset[t].  Work is tiled per tensor:
// tile_begin[t] is the first tile of tensor t (tile_begin[T] = total), each
// tile covers tile_elems elements of that tensor; one CTA per (tile, rank),
// the rank in grid.y.
constexpr int kFuseMaxTensors = 64;
constexpr int kFuseMaxCopies = 1024;  // W * T per launch
struct FuseParams {
  void* tensor[kFuseMaxCopies];
  void* fused[VCOLL_MAX_RANKS];
  int64_t count[kFuseMaxTensors];
  int64_t offset[kFuseMaxTensors];
  int64_t tile_begin[kFuseMaxTensors + 1];
  int64_t tile_elems;
  int T;
  int W;
  int unpack;  // 0: tensors -> fused, 1: fused -> tensors
};

// Multi-tensor allreduce: per rank u, tensors in[u*T + t] (t < T) form one
// virtual buffer (tensor t at fused offset off_t = counts[0..t) summed), and
// the allreduce of the W virtual buffers lands in out[u*T + t] -- the bits of
// pack -> in-place allreduce -> unpack, without the fusion buffer.  The host
// cuts the fused index space into pieces, each inside one tensor and one
// segment (so the fold's start rank is uniform per piece); a launch covers up
// to kMultiMaxTensors tensors.
constexpr int kMultiMaxTensors = 64;
constexpr int kMultiMaxPtrs = 768;  // W * T per launch (inputs; the same for outputs)
constexpr int kMultiMaxPieces = kMultiMaxTensors + VCOLL_MAX_RANKS;
struct MultiPiece {
  int64_t k0;          // first element of the piece inside tensor t
  int64_t len;         // elements
  int64_t tile_begin;  // first tile of the piece (pieces are tiled back to back)
  int t;               // tensor index inside this launch
  int start;           // first rank of the fold
  int phase;           // piece-local element i is 16-byte aligned in every buffer
                       // iff (i + phase) % V == 0; -1: phases differ, element-wise
  int pad;
};
struct MultiParams {
  // tensor-major: in[t * W + u] is tensor t of rank u
  const void* in[kMultiMaxPtrs];
  void* out[kMultiMaxPtrs];
  MultiPiece piece[kMultiMaxPieces];
  int64_t num_tiles;
  int64_t tile_elems;
  int npieces;
  int T;
  int W;
  float scale;
  int do_scale;
};

// Sparsified allreduce (SINGA valSparsAllReduce / topKSparsAllReduce).
// Top-K keeps, per rank, the K entries with the largest values (ties: lower
// index first), found by an exact radix select over order-preserving 32-bit
// keys in three digit passes (11, 11 and 10 bits).  Per-rank selection state
// and the digit histograms live in a device workspace.
constexpr int kTopkBins = 2048;
struct TopkState {
  uint32_t prefix;    // key bits fixed by the passes so far
  uint32_t T;         // after the last pass: the K-th largest key
  int64_t remaining;  // entries still to take at or below the current prefix
  int64_t need;       // entries equal to T that are kept
  int64_t equal;      // entries equal to T
  int64_t boundary;   // equal entries with index <= boundary are kept
  uint32_t low;       // first-digit bins below this one are not counted
  uint32_t topkey;    // candidate path: the last key listed; keys above it
                      // are kept without selection, counted, not listed (the
                      // end of a first-digit bin, or of a 22-bit prefix
                      // inside it; 0xFFFFFFFF: no band)
  int redo;           // the first-digit pass must be repeated over all bins
  int full;           // this rank's select passes read the whole array (its
                      // candidate list overflowed or missed the K-th key)
  uint32_t lowkey;    // candidate path: keys below this one are not listed
  uint32_t setkey;    // list route: keys above this one are kept for certain
                      // (unless the sample misled), so the candidate pass
                      // writes their residuals itself (0xFFFFFFFF: none)
  int64_t low_rem;    // sample keys still wanted at or above lowkey inside its
  int64_t set_rem;    // bin, allowed above setkey inside its bin, and allowed
  int64_t hi_rem;     // above topkey inside its bin (the second-digit
                      // refinement of the bounds)
  uint32_t tie_n;     // candidate path: candidates equal to T collected so far
  uint32_t tie_done;  // candidate path: CTAs of the tie pass that finished
  int tie_resolved;   // candidate path: the tie pass set the boundary (the
                      // index-digit passes have nothing left to do)
};
struct SparseParams {
  const void* in[VCOLL_MAX_RANKS];
  void* out[VCOLL_MAX_RANKS];
  void* acc[VCOLL_MAX_RANKS];  // error-feedback accumulations, or all NULL
  int64_t* nnz;                // device, W counters (may be NULL)
  uint32_t* hist;              // workspace: W x kTopkBins
  TopkState* state;            // workspace: W entries
  uint32_t* tilecnt;           // workspace: W x tiles_per_rank (tie counts, or
                               // on the candidate path each tile's list entries)
  uint32_t* chunk;             // workspace: W x tiles_per_rank, where each tile's
                               // entries start in its rank's list
  unsigned long long* cand_n;  // workspace: W candidate counts, then W counts of
                               // entries above the candidate band
  uint32_t* cand_key;          // workspace: W x cand_cap candidate keys
  uint32_t* cand_idx;          // workspace: W x cand_cap candidate indices
  int64_t cand_cap;            // candidate list capacity per rank
  int use_cand;                // select passes after the first read candidates
  int band;                    // the sample sets a two-sided band (else a lower
                               // bound with a wide margin)
  int sample_stride;           // the sample pass reads every sample_stride-th tile
  int64_t n;
  int64_t tiles_per_rank;      // histogram passes: grid.y = rank
  int64_t num_tiles;           // apply pass: tiles over [0, n)
  int64_t tile_elems;
  int64_t K;
  int W;
  int phase;                   // 16-byte phase shared by every buffer, or -1
  int has_acc;
  int x_in_acc;                // acc already holds x = in + acc (written by the
                               // top-K candidate pass): later passes read acc alone
  int list_out;                // top-K: the result may come from the candidate lists
  float threshold;
};
constexpr int64_t kSparseTileElems = 4096;
// Top-K working memory, regions 256-byte aligned: histograms, states,
// candidate counts and per-tile tie counts (together the minimum a call
// needs), then per-tile list offsets and the candidate lists: cand_cap keys
// and cand_cap indices per rank.  With room for candidates one pass over the
// data collects every entry in the sample's band, and the later select
// passes read only those.
struct TopkLayout {
  size_t state, cand_n, tilecnt, cands;  // byte offsets; cands = the minimum size
  size_t chunk_bytes;                    // per-tile list offsets (start of the lists' room)
};
inline TopkLayout topk_layout(int W, int64_t n) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const int64_t tiles = (n + kSparseTileElems - 1) / kSparseTileElems;
  TopkLayout L;
  L.state = al((size_t)W * kTopkBins * sizeof(uint32_t));
  L.cand_n = al(L.state + (size_t)W * sizeof(TopkState));
  L.tilecnt = al(L.cand_n + 2 * (size_t)W * sizeof(unsigned long long));
  L.cands = al(L.tilecnt + (size_t)W * (size_t)(tiles > 0 ? tiles : 1) * sizeof(uint32_t));
  L.chunk_bytes = al((size_t)W * (size_t)(tiles > 0 ? tiles : 1) * sizeof(uint32_t));
  return L;
}
inline size_t topk_workspace_min_bytes(int W, int64_t n) { return topk_layout(W, n).cands; }
// candidates per rank the recommended workspace holds: an eighth of the
// entries (room for K up to about n/24 above a lower bound, and for the
// two-sided band of larger K), all
// of them for small arrays; a multiple of 4 so that both lists stay 16-byte
// aligned
inline int64_t topk_cand_cap_default(int64_t n) {
  int64_t c = n / 8 + 4096;
  if (c > n) c = n;
  return (c + 3) & ~(int64_t)3;
}
inline size_t topk_workspace_bytes(int W, int64_t n) {
  const TopkLayout L = topk_layout(W, n);
  return L.cands + L.chunk_bytes + (size_t)W * (size_t)topk_cand_cap_default(n) * 8;
}

const void* selftest_timeout_kernel();

// Sets the thread-local message vcoll_last_error() returns; returns status.
int report_error(int status, const char* message);

// Kernel selection (function pointers for cudaLaunchKernel).  W_t is the
// compile-time rank count (2, 4, 8, 16) or 0 for the runtime-W kernels; vec
// selects the 16-byte vector path.
const void* reduce_kernel_f32(int op, int kind, int W_t, int ring, int vec);
const void* reduce_kernel_bf16(int op, int kind, int W_t, int ring, int vec);
// inputs at other 16-byte phases than the (shared) phase of the outputs
const void* reduce_kernel_f32_realign(int op, int kind, int W_t, int ring);
const void* reduce_kernel_bf16_realign(int op, int kind, int W_t, int ring);
const void* staged_kernel_f32(int op, int kind, int W_t, int ring);
const void* staged_kernel_bf16(int op, int kind, int W_t, int ring);
const void* gather_kernel(int elem_size, int vec);  // vec: 0 element-wise, 1 vectors, 2 realigned
const void* gather_tma_kernel(int elem_size);
const void* wire_kernel(int wire, int W_t, int ring);
const void* sparse_apply_kernel(int topk);
const void* topk_hist_kernel(int pass);
const void* topk_sample_kernel();
const void* topk_select_low_kernel();
const void* topk_sample2_kernel();         // second digit over the sample
const void* topk_select_refine_kernel();   // refines the settled and lower bounds
const void* topk_redo_hist_kernel();
const void* topk_redo_select_kernel();
const void* topk_select_kernel(int pass);
const void* topk_filter_kernel(int has_acc, int band);
const void* topk_list_out_kernel();
const void* topk_restore_kernel();
const void* topk_cand_hist_kernel(int pass);  // 0-2 key digits, 3-5 index digits
const void* topk_index_select_kernel(int pass);  // 3-5
const void* topk_tie_count_kernel();
const void* topk_tie_find_kernel();
const void* topk_ties_kernel();
// dynamic shared memory the realigned allgather requests without using it,
// to run two CTAs per SM
constexpr size_t kGatherRealignSmem = 100 * 1024;
constexpr int kGatherTmaThreads = 64;
constexpr int kGatherTmaStages = 4;
constexpr int kGatherTmaTileBytes = 32768;
// Device address of the per-device error word (VCOLL_DEVICE_ERR_* bits).
unsigned int* device_error_symbol();
const void* fuse_flat_kernel(int elem_size);
const void* multi_kernel_f32(int op, int W_t, int ring);
const void* multi_kernel_bf16(int op, int W_t, int ring);

// Vectors (16 B) per thread per tile of the direct kernels, by W_t.
VCOLL_HD constexpr int unroll_for(int W_t) {
  return W_t == 2 ? 8 : W_t == 4 ? 4 : W_t == 8 ? 2 : W_t == 16 ? 1 : 2;
}

// Staged kernel geometry (shared with the host for launch configuration).
constexpr int kStagedConsumerWarps = 8;
constexpr int kStagedThreads = (kStagedConsumerWarps + 1) * 32;
constexpr int kStagedStages = 4;
// bytes of one rank's slice of one tile; the stage holds W of them
VCOLL_HD constexpr int staged_slice_bytes(int W_t) {
  return W_t == 2 ? 16384 : W_t == 4 ? 8192 : W_t == 8 ? 4096 : 2048;
}
VCOLL_HD constexpr int staged_smem_bytes(int W_t) {
  return kStagedStages * W_t * staged_slice_bytes(W_t) + 256;
}

}  // namespace vcoll

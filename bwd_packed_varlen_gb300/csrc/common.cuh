// Shared definitions of the attention kernels: launch parameters, workspace
// header layout, tile sizes and the work-list decoding used by every kernel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace teattn {

// Tile shape of the tensor-core kernels: 128 query rows (the M of one tcgen05
// MMA) by 128 key rows per step.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// The forward takes two consecutive query tiles of one sequence and head per item.
constexpr int kBlockF = 2 * kBlockM;

// Workspace header (int32 words at the start of every workspace).
enum HeaderWord : int {
  kHdrStatus = 0,    // TE_STATUS_* bits raised by this call's kernels
  kHdrNumQPairs = 1, // number of (sequence, query tile) pairs
  kHdrNumKPairs = 2, // number of (sequence, key tile) pairs
  kHdrNextFwd = 3,   // work counters of the persistent kernels (zeroed per call)
  kHdrNextDkdv = 4,
  kHdrNextDq = 5,
  kHdrNumFPairs = 6, // number of (sequence, 256-row query tile pair) items
  kHdrNextFused = 7, // work counter of the fused backward kernel
  kHdrSelftest = 8,  // words 8..11: results of te_attn_selftest_wait_timeout
  kHdrWords = 64     // header size in int32 words (256 bytes, keeps alignment)
};

// Work lists the scheduler sorts for a call (the prefix sums are always built).
// kListKChain builds the key-tile list in the order the fused backward needs
// (instead of kListK's cost order): sequences with more key tiles first, and within
// a sequence the key tiles in descending order.
constexpr int kListQ = 1, kListK = 2, kListF = 4, kListKChain = 8;

constexpr int kStatusBadSeqlens = 1;
constexpr int kStatusTimeout = 2;
constexpr int kStatusOutOfBounds = 4;
constexpr int kStatusInternal = 8;  // a kernel found its launch unusable (e.g. misaligned shared memory)

// Bounds checks of computed global offsets. In the debug build of the library
// (TEATTN_DEBUG_BOUNDS defined) a failed check records kStatusOutOfBounds in the
// call's status word and the caller skips the access; in the release build the
// check compiles to `true` and costs nothing. Never a trap or an assert: the
// status word is read by the host after the call.
__device__ __forceinline__ bool bounds_ok(bool in_bounds, int* status) {
#ifdef TEATTN_DEBUG_BOUNDS
  if (!in_bounds) atomicOr(status, kStatusOutOfBounds);
  return in_bounds;
#else
  (void)in_bounds;
  (void)status;
  return true;
#endif
}

// Everything a kernel of this library needs, by value.
struct AttnParams {
  const void* q;
  const void* k;
  const void* v;
  const void* out_in;  // backward: forward output (input)
  const void* dout;
  const float* lse_in; // backward: forward lse (input)
  void* out;           // forward output
  float* lse;          // forward lse output
  void* dq;
  void* dk;
  void* dv;
  // Backward, per (query tile pair, head) blocks of 128 rows in the natural pair
  // order (pair = pref_q[b] + row / 128): lse * log2(e) and D = rowsum(dO * O).
  float* lse_t;    // -lse * log2(e), tile-major
  float* delta_t;  // -D = -rowsum(dO * O), tile-major
  const int* pref_q;   // prefix sums of query tiles per sequence (scheduler output)
  // Fused backward: fp32 dQ accumulator, one 128-row tile of dq_cols (64 or 128)
  // columns per (natural query tile pair, head), and one int semaphore per (pair,
  // head) counting the key tiles that have added into that tile.
  float* dq_acc;
  int* dq_sem;
  int dq_cols;
  // Fused backward work items (sequence, key tile, kv head, 0) in chain-major
  // order: for each sequence in the order of the chain-ordered key-tile list, each
  // kv head, the sequence's key tiles from the last to the first.
  int4* k_items;

  const int* cu_q;
  const int* cu_kv;
  const int* cu_q_pad;
  const int* cu_kv_pad;

  int batch;
  int total_q;
  int total_kv;
  int hq;
  int hkv;
  int d;
  int group;         // hq / hkv
  int sbhd;          // 0: packed rows (token i of sequence b at row cu_*_padded[b] + i);
                     // 1: sequence-major (token i of sequence b at row i * batch + b)
  int rs;            // rows between consecutive tokens of a sequence: 1, or batch
  int causal;        // 0 padding; 1 causal, upper-left; 2 causal, lower-right
  float scale;       // attn_scale
  float scale_log2;  // attn_scale * log2(e)

  int* header;       // workspace header (status, pair counts)
  int2* q_pairs;     // sorted (sequence, query tile) pairs
  int2* k_pairs;     // sorted (sequence, key tile) pairs
  int2* f_pairs;     // sorted (sequence, 256-row query tile) pairs (forward)
  int pair_cap_q;    // capacity of q_pairs
  int pair_cap_k;    // capacity of k_pairs
  int pair_cap_f;    // capacity of f_pairs
  int sched_lists;   // kList* bits: lists this call's kernels read
};

// Real length and padded offset of sequence b, validated against the tensor
// extents. Returns false (length 0) for a sequence whose cu_seqlens are
// inconsistent; the scheduler flags those in the status word.
struct SeqInfo {
  int off_q, len_q, off_k, len_k;  // off: token coordinate of token 0 in the tensor maps
  int tb;    // batch coordinate in the tensor maps (0 packed, b sequence-major)
  int diag;  // causal boundary: query i sees key j iff j <= i + diag
  bool ok;
};

__device__ __forceinline__ SeqInfo load_seq(const AttnParams& p, int b) {
  SeqInfo s;
  int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
  int k0 = p.cu_kv[b], k1 = p.cu_kv[b + 1];
  s.len_q = q1 - q0;
  s.len_k = k1 - k0;
  if (p.sbhd) {
    // every sequence spans the whole token extent of its batch entry
    s.off_q = 0;
    s.off_k = 0;
    s.tb = b;
    s.ok = s.len_q >= 0 && s.len_k >= 0 && s.len_q <= p.total_q / p.batch &&
           s.len_k <= p.total_kv / p.batch;
  } else {
    int pq0 = p.cu_q_pad[b], pq1 = p.cu_q_pad[b + 1];
    int pk0 = p.cu_kv_pad[b], pk1 = p.cu_kv_pad[b + 1];
    s.off_q = pq0;
    s.off_k = pk0;
    s.tb = 0;
    s.ok = s.len_q >= 0 && s.len_k >= 0 && pq0 >= 0 && pk0 >= 0 && s.len_q <= pq1 - pq0 &&
           s.len_k <= pk1 - pk0 && pq1 <= p.total_q && pk1 <= p.total_kv;
  }
  if (!s.ok) {
    s.len_q = 0;
    s.len_k = 0;
  }
  // Upper-left alignment puts query i at key position i; lower-right puts it at
  // len_k - len_q + i, so the last query sees every key.
  s.diag = p.causal == 2 ? s.len_k - s.len_q : 0;
  return s;
}

// Tensor rows of query token i / key token j of sequence s (row-major [rows, h, d]).
__device__ __forceinline__ size_t q_row(const AttnParams& p, const SeqInfo& s, int i) {
  return static_cast<size_t>(s.off_q + i) * p.rs + s.tb;
}
__device__ __forceinline__ size_t k_row(const AttnParams& p, const SeqInfo& s, int j) {
  return static_cast<size_t>(s.off_k + j) * p.rs + s.tb;
}

// Sequence holding tensor row r and the token index there (*i); -1 when no
// sequence's span holds it. cu_pad: the padded prefix sums of the row's tensor.
__device__ __forceinline__ int locate_row(const AttnParams& p, const int* cu_pad, int r, int* i) {
  if (p.sbhd) {
    *i = r / p.batch;
    return r % p.batch;
  }
  const int B = p.batch;
  if (r < cu_pad[0] || r >= cu_pad[B]) return -1;
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_pad[mid] <= r) lo = mid; else hi = mid - 1;
  }
  *i = r - cu_pad[lo];
  return lo;
}

// Index of (natural query-tile pair of row i of sequence b, head h, row in tile)
// in the tiled lse / D buffers.
__device__ __forceinline__ size_t tiled_index(const AttnParams& p, int b, int i, int h) {
  const int pair = p.pref_q[b] + i / kBlockM;
  return (static_cast<size_t>(pair) * p.hq + h) * kBlockM + (i % kBlockM);
}

// Number of keys (a prefix 0 .. n-1) that real query row i sees: all of them
// without the causal mask, keys j <= i + diag with it. Zero for a query before
// the lower-right triangle starts.
__device__ __forceinline__ int row_keys(const SeqInfo& s, int i, bool causal) {
  return causal ? min(s.len_k, max(0, i + 1 + s.diag)) : s.len_k;
}

// Work items of the dQ kernel and the one-tile forward are numbered group-major
// (the two-tile forward numbers its own pair-major): all items of kv
// head group 0, then group 1, ...; within a group the pairs in list order (longest
// first) with the group's heads innermost. Blocks running at the same time then
// work on one group's heads, whose Q/dO and K/V tiles stay in L2, rather than on
// every head of a sequence at once. `heads_per_group`: query heads per kv head for
// the per-query-head kernels, the column splits of one kv head for dK/dV.
struct PairHead {
  int pair, head;
};
__device__ __forceinline__ PairHead item_pair_head(int item, int n_pairs, int heads_per_group) {
  const int per_group = n_pairs * heads_per_group;
  const int g = item / per_group, r = item - g * per_group;
  return PairHead{r / heads_per_group, g * heads_per_group + r % heads_per_group};
}

// dK/dV items: the sorted key-tile list is cut into bands of kBand consecutive
// pairs, and within a band the items go head-major (all of the band's pairs for
// head 0, then head 1, ...). Whole-list group-major order would start the last
// groups' longest key tiles late and leave SMs idle at the end of the kernel; the
// bands keep the list's longest-first order at band granularity while items of
// one kv head still run side by side. The last full band and the remainder go
// pair-major instead (every head of a pair, pairs longest first), so the final
// items the blocks take are the shortest ones and the blocks finish together.
// `heads`: kv heads x column splits.
__device__ __forceinline__ PairHead item_pair_head_banded(int item, int n_pairs, int heads) {
  constexpr int kBand = 64;
  const int full = n_pairs / kBand;
  const int banded_pairs = (full > 0 ? full - 1 : 0) * kBand;
  const int banded_items = banded_pairs * heads;
  if (item < banded_items) {
    const int c = item / (kBand * heads), r = item - c * (kBand * heads);
    return PairHead{c * kBand + r % kBand, r / kBand};
  }
  const int r = item - banded_items;
  return PairHead{banded_pairs + r / heads, r % heads};
}

// Number of key rows a query tile can see (the keys its last real row sees).
__device__ __forceinline__ int visible_keys(const SeqInfo& s, int q_tile, bool causal) {
  if (!causal) return s.len_k;
  const int last_q = min((q_tile + 1) * kBlockM, s.len_q);  // exclusive
  return min(s.len_k, max(0, last_q + s.diag));
}

// First query row that sees key j (causal: i >= j - diag).
__device__ __forceinline__ int first_query(const SeqInfo& s, int j, bool causal) {
  return causal ? max(0, j - s.diag) : 0;
}

// Number of key rows some real query sees (the rest get exact-zero dk/dv).
__device__ __forceinline__ int seen_keys(const SeqInfo& s, bool causal) {
  if (s.len_q == 0) return 0;
  return causal ? min(s.len_k, max(0, s.len_q + s.diag)) : s.len_k;
}

}  // namespace teattn

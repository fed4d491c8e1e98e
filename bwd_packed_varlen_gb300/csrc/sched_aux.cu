// Work scheduling (tile lists), exact-zero fill of rows no tile covers, the
// backward preprocess D = rowsum(dO * O), and the e4m3 -> bf16 widening of V for
// the e4m3 forward. All are memory- or latency-bound SIMT kernels; the
// tensor-core kernels consume what they produce.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace teattn {

// ---------------------------------------------------------------------------
// Scheduler
// ---------------------------------------------------------------------------
// One 1024-thread block turns the four cu_seqlens arrays into three lists:
//   q pairs  (sequence, query tile)            -- dQ items (x hq heads)
//   k pairs  (sequence, key tile)              -- dK/dV items (x hkv heads)
//   f pairs  (sequence, pair of query tiles)   -- forward items (x hq heads)
// Tiles cover the REAL length of each sequence; sequences without a real query
// or key produce no pair, and key tiles no real query sees (upper-left causal,
// beyond the query length) produce none either -- those rows are zero-filled
// instead. Query tiles whose rows all precede a lower-right causal triangle are
// listed but see no key: the kernels skip them and the zero fill writes them.
// Each list is sorted by estimated cost (key tiles the item visits), largest
// first, ties by natural order, so a persistent grid takes the long items first.
// Up to kSortCap pairs are sorted in shared memory; a longer list keeps its
// natural order. The result depends only on the cu_seqlens values.
// For the fused backward the key-tile list is built in chain order instead
// (kListKChain): sequences with more key tiles first (ties: lower index), and
// inside a sequence its key tiles in DESCENDING order -- the order in which that
// kernel's blocks add into each dQ tile, so a block only ever waits on key tiles
// claimed before its own. A list longer than kSortCap keeps the sequences in
// natural order, still with each sequence's key tiles descending.
constexpr int kSchedThreads = 1024;
constexpr int kSortCap = 8192;

__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

// Last b in [0, B) with pref[b] <= i (pref is non-decreasing, pref[B] > i).
__device__ __forceinline__ int find_seq(const int* pref, int B, int i) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ int q_pair_cost(const AttnParams& p, int b, int t) {
  SeqInfo s = load_seq(p, b);
  return (visible_keys(s, t, p.causal) + kBlockN - 1) / kBlockN;
}

__device__ int k_pair_cost(const AttnParams& p, int b, int t) {
  SeqInfo s = load_seq(p, b);
  int nq = (s.len_q + kBlockM - 1) / kBlockM;
  return nq - first_query(s, t * kBlockN, p.causal) / kBlockM;
}

// Forward item of two query tiles: both tiles' key tiles (the second sees most).
__device__ int f_pair_cost(const AttnParams& p, int b, int t) {
  SeqInfo s = load_seq(p, b);
  const int a = (visible_keys(s, 2 * t, p.causal) + kBlockN - 1) / kBlockN;
  const int c = 2 * t * kBlockM + kBlockM < s.len_q
                    ? (visible_keys(s, 2 * t + 1, p.causal) + kBlockN - 1) / kBlockN
                    : 0;
  return a + c;
}

// Key tiles of sequence b in chain order: natural index i (sequence b, its j-th
// key tile, j = i - pref[b]) stands for key tile nk_b - 1 - j = pref[b+1] - 1 - i.
__device__ __forceinline__ int2 chain_pair(const int* pref, int B, long long i) {
  const int b = find_seq(pref, B, static_cast<int>(i));
  return make_int2(b, pref[b + 1] - 1 - static_cast<int>(i));
}

__device__ void build_chain_list(const AttnParams& p, const int* pref, int n, int2* out,
                                 uint64_t* keys) {
  const int B = p.batch;
  if (n > kSortCap) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = chain_pair(pref, B, i);
    return;
  }
  int m = 1;
  while (m < n) m <<= 1;
  constexpr uint64_t kLow = (1ull << 40) - 1;
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    uint64_t key = ~0ull;
    if (i < n) {
      const int b = find_seq(pref, B, i);
      const int nk = min(pref[b + 1] - pref[b], 0xffffff);
      key = (static_cast<uint64_t>(0xffffff - nk) << 40) | static_cast<uint64_t>(i);
    }
    keys[i] = key;
  }
  __syncthreads();
  for (int k = 2; k <= m; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < m; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], c = keys[ixj];
          const bool up = (i & k) == 0;
          if ((a > c) == up) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    out[i] = chain_pair(pref, B, static_cast<long long>(keys[i] & kLow));
  __syncthreads();
}

// kKind: 0 query tiles, 1 key tiles, 2 forward pairs of query tiles. The sort of
// a list of n <= kSortCap pairs runs in three phases, each over the threads
// [t, t + nt): the keys (cost descending, then list position) padded to a power of
// two m, the bitonic stages (k, j), and the sorted pairs written out.
template <int kKind>
__device__ void list_keys(const AttnParams& p, const int* pref, int n, int m, uint64_t* keys, int t,
                          int nt) {
  for (int i = t; i < m; i += nt) {
    uint64_t key = ~0ull;
    if (i < n) {
      const int b = find_seq(pref, p.batch, i);
      const int tt = i - pref[b];
      const int cost = kKind == 0 ? q_pair_cost(p, b, tt)
                       : (kKind == 1 ? k_pair_cost(p, b, tt) : f_pair_cost(p, b, tt));
      key = (static_cast<uint64_t>(0x7fffffffu - static_cast<uint32_t>(cost)) << 32) |
            static_cast<uint32_t>(i);
    }
    keys[i] = key;
  }
}

__device__ __forceinline__ void list_stage(uint64_t* keys, int m, int k, int j, int t, int nt) {
  for (int i = t; i < m; i += nt) {
    const int ixj = i ^ j;
    if (ixj > i) {
      const uint64_t a = keys[i], c = keys[ixj];
      const bool up = (i & k) == 0;
      if ((a > c) == up) {
        keys[i] = c;
        keys[ixj] = a;
      }
    }
  }
}

__device__ void list_out(const AttnParams& p, const int* pref, int n, int2* out, const uint64_t* keys,
                         int t, int nt) {
  for (int i = t; i < n; i += nt) {
    const int src = static_cast<int>(keys[i] & 0xffffffffu);
    const int b = find_seq(pref, p.batch, src);
    out[i] = make_int2(b, src - pref[b]);
  }
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int m = 1;
  while (m < n) m <<= 1;
  return m;
}

template <int kKind>
__device__ void build_list(const AttnParams& p, const int* pref, int n, int2* out,
                           uint64_t* keys) {
  if (n <= kSortCap) {
    const int m = pow2_at_least(n);
    list_keys<kKind>(p, pref, n, m, keys, threadIdx.x, blockDim.x);
    __syncthreads();
    for (int k = 2; k <= m; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        list_stage(keys, m, k, j, threadIdx.x, blockDim.x);
        __syncthreads();
      }
    }
    list_out(p, pref, n, out, keys, threadIdx.x, blockDim.x);
    __syncthreads();
  } else {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      int b = find_seq(pref, p.batch, i);
      out[i] = make_int2(b, i - pref[b]);
    }
  }
}

// The backward's query-tile and key-tile lists, sorted side by side: half of the
// threads each, one block-wide barrier per stage of the longer list (the shorter
// list's stages are a prefix of it), so the two sorts cost about one.
__device__ void build_q_k_lists(const AttnParams& p, const int* pref_q, int nq, const int* pref_k, int nk,
                                uint64_t* keys) {
  const int half = blockDim.x / 2;
  const bool first = threadIdx.x < half;
  const int t = first ? threadIdx.x : threadIdx.x - half;
  uint64_t* kq = keys;
  uint64_t* kk = keys + kSortCap;
  const int mq = pow2_at_least(nq), mk = pow2_at_least(nk);
  if (first)
    list_keys<0>(p, pref_q, nq, mq, kq, t, half);
  else
    list_keys<1>(p, pref_k, nk, mk, kk, t, half);
  __syncthreads();
  const int mmax = mq > mk ? mq : mk;
  for (int k = 2; k <= mmax; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (first) {
        if (k <= mq) list_stage(kq, mq, k, j, t, half);
      } else {
        if (k <= mk) list_stage(kk, mk, k, j, t, half);
      }
      __syncthreads();
    }
  }
  if (first)
    list_out(p, pref_q, nq, p.q_pairs, kq, t, half);
  else
    list_out(p, pref_k, nk, p.k_pairs, kk, t, half);
  __syncthreads();
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(AttnParams p, int* pref_q,
                                                                  int* pref_k, int* pref_f) {
  extern __shared__ uint64_t sort_keys[];
  __shared__ int warp_sums[32];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  int carry_q = 0, carry_k = 0, carry_f = 0;
  for (int base = 0; base < p.batch; base += blockDim.x) {
    int b = base + threadIdx.x;
    int cq = 0, ck = 0, cf = 0;
    if (b < p.batch) {
      SeqInfo s = load_seq(p, b);
      if (!s.ok) bad = 1;
      if (s.len_q > 0 && s.len_k > 0) {
        cq = (s.len_q + kBlockM - 1) / kBlockM;
        ck = (seen_keys(s, p.causal) + kBlockN - 1) / kBlockN;
        cf = (s.len_q + kBlockF - 1) / kBlockF;
      }
    }
    int tq, tk, tf;
    int eq = block_excl_scan(cq, warp_sums, &tq);
    int ek = block_excl_scan(ck, warp_sums, &tk);
    int ef = block_excl_scan(cf, warp_sums, &tf);
    if (b < p.batch) {
      pref_q[b] = carry_q + eq;
      pref_k[b] = carry_k + ek;
      pref_f[b] = carry_f + ef;
    }
    carry_q += tq;
    carry_k += tk;
    carry_f += tf;
  }
  if (threadIdx.x == 0) {
    pref_q[p.batch] = carry_q;
    pref_k[p.batch] = carry_k;
    pref_f[p.batch] = carry_f;
  }
  __threadfence_block();
  __syncthreads();
  const int nq = min(carry_q, p.pair_cap_q);
  const int nk = min(carry_k, p.pair_cap_k);
  const int nf = min(carry_f, p.pair_cap_f);
  const bool both = (p.sched_lists & kListQ) && (p.sched_lists & kListK) && nq <= kSortCap &&
                    nk <= kSortCap;
  if (both) {
    build_q_k_lists(p, pref_q, nq, pref_k, nk, sort_keys);
  } else {
    if (p.sched_lists & kListQ) build_list<0>(p, pref_q, nq, p.q_pairs, sort_keys);
    if (p.sched_lists & kListK) build_list<1>(p, pref_k, nk, p.k_pairs, sort_keys);
  }
  if (!(p.sched_lists & kListK) && (p.sched_lists & kListKChain)) {
    build_chain_list(p, pref_k, nk, p.k_pairs, sort_keys);
    __syncthreads();
    // Items of the fused backward, chain-major: sequence b's pairs occupy list
    // positions [P, P + nk_b) (key tiles descending); its items are, per kv head g,
    // those key tiles in the same order, at hkv * P + g * nk_b + (position - P).
    // Running one (sequence, kv head) chain's key tiles together keeps the dQ tiles
    // they all add to in L2.
    for (int j = threadIdx.x; j < nk; j += blockDim.x) {
      const int2 pr = p.k_pairs[j];
      const int len = pref_k[pr.x + 1] - pref_k[pr.x];
      const int start = j - (len - 1 - pr.y);
      for (int g = 0; g < p.hkv; ++g)
        p.k_items[static_cast<size_t>(start) * p.hkv + static_cast<size_t>(g) * len + (j - start)] =
            make_int4(pr.x, pr.y, g, 0);
    }
  }
  if (p.sched_lists & kListF) build_list<2>(p, pref_f, nf, p.f_pairs, sort_keys);
  if (threadIdx.x == 0) {
    int status = bad ? kStatusBadSeqlens : 0;
    if (carry_q > p.pair_cap_q || carry_k > p.pair_cap_k || carry_f > p.pair_cap_f)
      status |= kStatusBadSeqlens;
    p.header[kHdrStatus] = status;
    p.header[kHdrNumQPairs] = nq;
    p.header[kHdrNumKPairs] = nk;
    p.header[kHdrNumFPairs] = nf;
    p.header[kHdrNextFwd] = 0;
    p.header[kHdrNextDkdv] = 0;
    p.header[kHdrNextDq] = 0;
    p.header[kHdrNextFused] = 0;
  }
}

cudaError_t launch_schedule(const AttnParams& p, int* pref_q, int* pref_k, int* pref_f,
                            cudaStream_t st) {
  const size_t smem = 2 * kSortCap * sizeof(uint64_t);  // two lists sorted side by side
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kSchedThreads, smem, st>>>(p, pref_q, pref_k, pref_f);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Zero fill: the rows no tile writes. Of sequence b's query rows these are a
// prefix of real queries that see no key (all of them without keys; before the
// lower-right triangle otherwise) and the pad rows after its real ones; of its key
// rows, those no real query sees and the pad rows. Block (b, y) clears a share of
// sequence b's rows, one warp per row with 16-byte stores; block b = batch clears
// the packed rows outside every sequence. Rows are kept inside the tensors even
// when the lengths are inconsistent (the scheduler reports those).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void zero_row(void* base, long long r, int row_bytes) {
  uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(base) +
                                        static_cast<size_t>(r) * row_bytes);
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x & 31; i < row_bytes / 16; i += 32) dst[i] = z;
}

// mode 0: forward (out, lse); mode 1: backward (dq, dk, dv)
__global__ void __launch_bounds__(256) zero_fill_kernel(AttnParams p, int mode) {
  const int b = blockIdx.x;
  const int nw = blockDim.x >> 5, lane = threadIdx.x & 31;
  const int w0 = blockIdx.y * nw + (threadIdx.x >> 5), wstep = nw * gridDim.y;
  const int qbytes = p.hq * p.d * 2, kbytes = p.hkv * p.d * 2;
  const bool causal = p.causal != 0;
  // query row r: out / lse (v on the lse) or dq
  auto clear_q = [&](long long r, float v) {
    if (r < 0 || r >= p.total_q) return;
    if (mode == 0) {
      zero_row(p.out, r, qbytes);
      for (int h = lane; h < p.hq; h += 32) p.lse[static_cast<size_t>(r) * p.hq + h] = v;
    } else {
      zero_row(p.dq, r, qbytes);
    }
  };
  auto clear_k = [&](long long r) {
    if (r < 0 || r >= p.total_kv) return;
    zero_row(p.dk, r, kbytes);
    zero_row(p.dv, r, kbytes);
  };
  if (b < p.batch) {
    const SeqInfo s = load_seq(p, b);
    // rows of sequence b: base + i * stride for i in [0, n)
    const long long qbase = p.sbhd ? b : p.cu_q_pad[b];
    const int qn = min(max(p.sbhd ? p.total_q / p.batch : p.cu_q_pad[b + 1] - p.cu_q_pad[b], 0), p.total_q);
    const int stride = p.sbhd ? p.batch : 1;
    const int dead = s.len_k == 0 ? s.len_q : (causal ? min(s.len_q, max(0, -s.diag)) : 0);
    const int nq = dead + max(0, qn - s.len_q);
    for (int z = w0; z < nq; z += wstep) {
      const int i = z < dead ? z : s.len_q + (z - dead);
      clear_q(qbase + static_cast<long long>(i) * stride, z < dead ? -INFINITY : 0.0f);
    }
    if (mode == 1) {
      const long long kbase = p.sbhd ? b : p.cu_kv_pad[b];
      const int kn = min(max(p.sbhd ? p.total_kv / p.batch : p.cu_kv_pad[b + 1] - p.cu_kv_pad[b], 0), p.total_kv);
      const int seen = seen_keys(s, causal);
      for (int j = seen + w0; j < kn; j += wstep) clear_k(kbase + static_cast<long long>(j) * stride);
    }
  } else if (!p.sbhd) {
    // packed rows before the first and after the last sequence: [0, lo) and [hi, total)
    auto outside = [&](int first, int last, int total, auto&& clear) {
      const int lo = min(max(first, 0), total), hi = min(max(last, lo), total);
      const int n = lo + (total - hi);
      for (int z = w0; z < n; z += wstep) clear(z < lo ? z : hi + (z - lo));
    };
    outside(p.cu_q_pad[0], p.cu_q_pad[p.batch], p.total_q, [&](long long r) { clear_q(r, 0.0f); });
    if (mode == 1) outside(p.cu_kv_pad[0], p.cu_kv_pad[p.batch], p.total_kv, clear_k);
  }
  // fused backward: the per-(query tile, head) counters of key tiles added to dQ
  if (mode == 1 && p.dq_sem) {
    const size_t n = static_cast<size_t>(p.pair_cap_q) * p.hq;
    const size_t nb = static_cast<size_t>(gridDim.x) * gridDim.y;
    const size_t stride = nb * blockDim.x;
    const size_t bid = static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    for (size_t i = bid * blockDim.x + threadIdx.x; i < n; i += stride) p.dq_sem[i] = 0;
  }
}

cudaError_t launch_zero_fill(const AttnParams& p, int mode, int num_sms, cudaStream_t st) {
  // one block per sequence plus one for the rows outside them, repeated along y
  // so that about four blocks per SM share the rows of few long sequences
  const int nb = p.batch + 1;
  const int y = std::max(1, std::min(65535, (num_sms * 4 + nb - 1) / nb));
  zero_fill_kernel<<<dim3(nb, y), 256, 0, st>>>(p, mode);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Preprocess: for every row the backward tiles read (real query rows of
// sequences with keys), D[r, h] = sum_c float(dO[r,h,c]) * float(O[r,h,c]) and
// lse[r, h] * log2(e), written tile-major (one contiguous block of 128 rows per
// (query tile, head)) so the backward kernels fetch a tile's values with one
// bulk copy. One warp per row; lanes read 16-byte chunks. When d/8 divides 32 the
// lanes of one head are contiguous and reduce by shuffles; otherwise each lane
// owns whole heads. Both orders are fixed (deterministic).
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  const T* x = reinterpret_cast<const T*>(&a);
  const T* y = reinterpret_cast<const T*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = fmaf(static_cast<float>(x[i]), static_cast<float>(y[i]), s);
  return s;
}

template <typename T>
__global__ void __launch_bounds__(256) delta_kernel(AttnParams p) {
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int cpr = p.d / 8;  // 16-byte chunks per head
  const int chunks = p.hq * cpr;
  constexpr float kLog2e = 1.4426950408889634f;
  for (int r = gw; r < p.total_q; r += warps) {
    int i = 0;
    const int b = locate_row(p, p.cu_q_pad, r, &i);
    if (b < 0) continue;
    const SeqInfo s = load_seq(p, b);
    if (i >= s.len_q || s.len_k == 0) continue;  // no tile reads this row
    const size_t row = static_cast<size_t>(r);
    const size_t t0 = tiled_index(p, b, i, 0);   // + h * 128 for head h
    if (!bounds_ok(t0 + static_cast<size_t>(p.hq - 1) * kBlockM <
                       static_cast<size_t>(p.pair_cap_q) * p.hq * kBlockM,
                   p.header + kHdrStatus))
      continue;
    for (int h = lane; h < p.hq; h += 32)
      p.lse_t[t0 + static_cast<size_t>(h) * kBlockM] = -(p.lse_in[row * p.hq + h] * kLog2e);
    const uint4* o = reinterpret_cast<const uint4*>(static_cast<const T*>(p.out_in) +
                                                    row * p.hq * p.d);
    const uint4* g = reinterpret_cast<const uint4*>(static_cast<const T*>(p.dout) +
                                                    row * p.hq * p.d);
    if (32 % cpr == 0) {
      // Four 32-chunk groups per pass: all loads of a pass are in flight together.
      for (int c0 = 0; c0 < chunks; c0 += 128) {
        uint4 oa[4], ga[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + 32 * u + lane;
          if (c < chunks) {
            oa[u] = o[c];
            ga[u] = g[c];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + 32 * u + lane;
          float v = c < chunks ? dot8<T>(oa[u], ga[u]) : 0.f;
          for (int w = cpr >> 1; w > 0; w >>= 1) v += __shfl_xor_sync(0xffffffffu, v, w);
          if (c < chunks && (c % cpr) == 0)
            p.delta_t[t0 + static_cast<size_t>(c / cpr) * kBlockM] = -v;
        }
      }
    } else {
      for (int h = lane; h < p.hq; h += 32) {
        float v = 0.f;
        for (int c = 0; c < cpr; ++c) v += dot8<T>(o[h * cpr + c], g[h * cpr + c]);
        p.delta_t[t0 + static_cast<size_t>(h) * kBlockM] = -v;
      }
    }
  }
}

cudaError_t launch_delta(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st) {
  if (bf16)
    delta_kernel<__nv_bfloat16><<<num_sms * 8, 256, 0, st>>>(p);
  else
    delta_kernel<__half><<<num_sms * 8, 256, 0, st>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// e4m3 -> bf16 widening: dst[i] = bf16(float(src[i]) * scale), n % 16 == 0, both
// 16-byte aligned. Each e4m3 value is exact in fp16; the product is rounded once.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) widen_e4m3_kernel(const uint4* __restrict__ src,
                                                         uint4* __restrict__ dst, size_t n16,
                                                         float scale) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // two e4m3 bytes (lower one first) -> two floats
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((w[k] >> (16 * h)) & 0xffffu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
        o[2 * k + h] = *reinterpret_cast<const uint32_t*>(&b);
      }
    }
    dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

cudaError_t launch_widen_e4m3(const void* src, void* dst, size_t n, float scale, int num_sms,
                              cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  widen_e4m3_kernel<<<num_sms * 8, 256, 0, st>>>(static_cast<const uint4*>(src),
                                                  static_cast<uint4*>(dst), n / 16, scale);
  return cudaGetLastError();
}

}  // namespace teattn

// Forward attention, two query tiles per work item (head_dim <= 128).
//
// One work item = (sequence b, query head h, query rows [256u, 256u+256)): tile A
// holds the first 128 rows, tile B the next 128 (absent when the sequence ends
// before it). Both tiles read the same key/value tiles, so each K/V tile is loaded
// once for 256 query rows. Roles:
//   warps 0-3  softmax of tile A (one thread per query row / TMEM lane),
//   warps 4-7  softmax of tile B,
//   warp 8     TMA producer (Q_A, Q_B once per item; K_j, V_j rings),
//   warp 9     MMA issuer (the whole warp; one elected lane issues).
// TMEM: O_A [0, 128), O_B [128, 256), S_A [256, 384), S_B [384, 512). The issue
// order is  S_A0, S_B0 | PV_A0, S_A1 | PV_B0, S_B1 | PV_A1, S_A2 | ...  so while one
// softmax warpgroup turns S into P the tensor cores work on the other tile. Since
// S_X(j+1) is issued after PV_X(j), its completion also means PV_X(j) finished: the
// softmax may rescale O_X as soon as S_X(j+1) is ready. P_X(j) is written as 16-bit
// values over S_X(j) and read from TMEM by PV_X(j). The running max is rescaled
// lazily (only when it grows by more than 2^8); masks use the REAL lengths and are
// applied only on tiles that need them. A tile's normalized O rows go to a
// shared-memory O tile and leave with TMA stores issued by one thread, so the
// softmax warps do not wait for the global writes (tiles that reach past their
// sequence's padded rows store row by row instead).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "row_store.cuh"
#include "sm103_ptx.cuh"
#include "tmap.h"
#include "work_queue.cuh"

namespace teattn {

// kFP8: Q and K are e4m3 (one 128-byte column chunk per row for kD = 128) and
// S = Q K^T runs as kind::f8f6f4; V (a bf16 copy) and O stay 16-bit.
template <int kD, bool kFP8 = false>
struct FwdPairShape {
  static_assert(kD == 64 || kD == 128, "two-tile forward supports head_dim up to 128");
  static_assert(!kFP8 || kD == 128, "the e4m3 forward uses 128 columns of Q and K");
  static constexpr int kChunks = kD / 64;                      // 64-column chunks of V and O
  static constexpr int kQKChunks = kFP8 ? kD / 128 : kChunks;  // 128-byte chunks of Q, K rows
  static constexpr int kQKBytes = kQKChunks * 16384;           // one Q or K tile
  static constexpr int kVBytes = kChunks * 16384;              // one V tile (16-bit)
  static constexpr int kQKColsPerChunk = kFP8 ? 128 : 64;      // elements in 128 bytes
  static constexpr int kSKSteps = kFP8 ? kD / 32 : kD / 16;    // MMAs per S (32 bytes of K each)
  static constexpr int kStages = 2;                            // K and V rings
  static constexpr int kOBytes = kChunks * 16384;                // O tile staged for the TMA store
  static constexpr int kSmemUsed = kQKBytes * (2 + kStages) + kVBytes * kStages + kOBytes + 1024;
  static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  // TMEM columns of O_x and S_x for tile x (0: A, 1: B)
  __device__ static constexpr uint32_t col_o(int x) { return static_cast<uint32_t>(x) * 128u; }
  __device__ static constexpr uint32_t col_s(int x) { return 256u + static_cast<uint32_t>(x) * 128u; }
};

constexpr int kFwdPairThreads = 320;
constexpr int kFwdWarpProducer = 8, kFwdWarpMma = 9;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per-item geometry, identical in every role.
struct FwdItem {
  SeqInfo s;
  int h, g, u;
  int n[2];      // key tiles tile A / tile B visit (0: tile absent)
  int nmax;
  bool whole[2];  // tile rows lie inside the sequence's padded rows (TMA store allowed)
};

// Items are numbered pair-major: every query head of a pair before the next pair,
// pairs in list order (longest first). The blocks' last items are then the list's
// shortest, so they finish together, and a pair's heads share one sequence's K/V
// rows, which stay in L2 while they run. (The kernels with one query tile per item
// keep the group-major order of item_pair_head, which measured faster for them.)
__device__ __forceinline__ FwdItem fwd_item(const AttnParams& p, int item, bool causal) {
  FwdItem I;
  const PairHead ph{item / p.hq, item % p.hq};
  const int2 pr = p.f_pairs[ph.pair];
  I.h = ph.head;
  I.g = I.h / p.group;
  I.u = pr.y;
  I.s = load_seq(p, pr.x);
  const int ta = 2 * I.u, tb = 2 * I.u + 1;
  I.n[0] = (visible_keys(I.s, ta, causal) + kBlockN - 1) / kBlockN;
  I.n[1] = tb * kBlockM < I.s.len_q ? (visible_keys(I.s, tb, causal) + kBlockN - 1) / kBlockN : 0;
  I.nmax = I.n[0] > I.n[1] ? I.n[0] : I.n[1];
  // the store box may not reach into the next sequence's rows; sequence-major
  // tensors keep every sequence in its own batch entry (the box is clipped there)
  const int pad_q = p.sbhd ? p.total_q : p.cu_q_pad[pr.x + 1] - p.cu_q_pad[pr.x];
  I.whole[0] = ta * kBlockM + kBlockM <= pad_q;
  I.whole[1] = tb * kBlockM + kBlockM <= pad_q;
  return I;
}

template <int kD, bool kBF16, bool kFP8 = false>
__global__ void __launch_bounds__(kFwdPairThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmO) {
  using S = FwdPairShape<kD, kFP8>;
  static_assert(!kFP8 || kBF16, "the e4m3 forward writes bf16");
  constexpr int NS = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                          // tile A then tile B
  uint8_t* sK = sQ + 2 * S::kQKBytes;         // NS stages
  uint8_t* sV = sK + NS * S::kQKBytes;         // NS stages
  uint8_t* sO = sV + NS * S::kVBytes;         // one O tile, shared by both tiles in turn

  __shared__ uint64_t bar_q_full, bar_q_empty;
  __shared__ uint64_t bar_k_full[NS], bar_k_empty[NS], bar_v_full[NS], bar_v_empty[NS];
  __shared__ uint64_t bar_s_full[2], bar_p_ready[2], bar_o_full[2], bar_o_empty[2];
  __shared__ uint64_t bar_stage, bar_ostage[2];  // O staging free / a tile's rows staged
  __shared__ WorkRing ring;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* status = p.header + kHdrStatus;
  const int n_items = p.header[kHdrNumFPairs] * p.hq;
  const bool causal = p.causal != 0;

  if (tid == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_empty[i], 1);
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_v_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_s_full[x], 1);
      mbar_init(&bar_p_ready[x], 128);
      mbar_init(&bar_o_full[x], 1);
      mbar_init(&bar_o_empty[x], 128);
    }
    ring_init(ring, 1 + 256);
    mbar_init(&bar_stage, 1);
    mbar_init(&bar_ostage[0], 128);
    mbar_init(&bar_ostage[1], 128);
    fence_barrier_init();
  }
  if (warp == kFwdWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kFwdWarpProducer) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int it = 0, ii = 0;
      bool ok = true;
      int nxt = blockIdx.x;
      for (; ok; ++ii) {
        int item = nxt < n_items ? nxt : -1;
        FwdItem I;
        // Items whose two tiles see no key (rows before a lower-right causal
        // triangle) are left to the zero fill and never reach the ring.
        while (item >= 0) {
          I = fwd_item(p, item, causal);
          if (I.nmax > 0) break;
          nxt = next_item(p.header + kHdrNextFwd);
          item = nxt < n_items ? nxt : -1;
        }
        if (item < 0) {
          ok = ring_put(ring, ii, -1, status);
          break;
        }
        // both tiles' key-tile counts travel with the item: the MMA thread then
        // needs no global loads (which would queue behind the softmax warps' O stores)
        if (!(ok = ring_put(ring, ii, item, status, I.n[0] | (I.n[1] << 16)))) break;
        nxt = next_item(p.header + kHdrNextFwd);  // used at the next hand-over
        if (ii > 0 && !(ok = mbar_wait(&bar_q_empty, (ii - 1) & 1, status))) break;
        const int ntiles = I.n[1] > 0 ? 2 : 1;
        mbar_arrive_expect_tx(&bar_q_full, ntiles * S::kQKBytes);
        for (int x = 0; x < ntiles; ++x)
          for (int c = 0; c < S::kQKChunks; ++c)
            tma_load_4d(sQ + x * S::kQKBytes + c * 16384, &tmQ, &bar_q_full, c * S::kQKColsPerChunk, I.h, I.s.tb,
                        I.s.off_q + (2 * I.u + x) * kBlockM);
        for (int j = 0; j < I.nmax; ++j, ++it) {
          const int st = it % NS;
          if (it >= NS && !(ok = mbar_wait(&bar_k_empty[st], ((it / NS) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&bar_k_full[st], S::kQKBytes);
          for (int c = 0; c < S::kQKChunks; ++c)
            tma_load_4d(sK + st * S::kQKBytes + c * 16384, &tmK, &bar_k_full[st], c * S::kQKColsPerChunk, I.g, I.s.tb,
                        I.s.off_k + j * kBlockN);
          if (it >= NS && !(ok = mbar_wait(&bar_v_empty[st], ((it / NS) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&bar_v_full[st], S::kVBytes);
          for (int c = 0; c < S::kChunks; ++c)
            tma_load_4d(sV + st * S::kVBytes + c * 16384, &tmV, &bar_v_full[st], c * 64, I.g, I.s.tb,
                        I.s.off_k + j * kBlockN);
        }
      }
    }
  } else if (warp == kFwdWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t idS =
          kFP8 ? make_idesc_e4m3(128, kBlockN) : make_idesc_f16(kBF16, false, false, 128, kBlockN);
      constexpr uint32_t idPV = make_idesc_f16(kBF16, false, true, 128, kD);
      // Q and K K-major; V as the N-major (d-contiguous) B of P V.
      const SmemDesc dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
      const SmemDesc dk = smem_desc(smem_u32(sK), 16, 1024, kLayoutSW128);
      const SmemDesc dv = smem_desc(smem_u32(sV), 16384, 1024, kLayoutSW128);
      int it = 0;
      int np[2] = {0, 0};  // P hand-overs consumed per tile
      int no[2] = {0, 0};  // items in which the tile was present
      bool ok = true;
      // S_x = Q_x K^T for the key tile in ring stage st.
      auto issue_s = [&](int x, int st) {
        const SmemDesc qx{dq.lo + ((x * S::kQKBytes) >> 4), dq.hi};
        const SmemDesc kst{dk.lo + ((st * S::kQKBytes) >> 4), dk.hi};
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s = 0; s < S::kSKSteps; ++s) {
          // 32 bytes of K per MMA: 16 16-bit or 32 8-bit elements
          const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
          if constexpr (kFP8)
            mma_ss_f8(tmem + S::col_s(x), qx, off, kst, off, idS, s > 0 ? 1u : 0u);
          else
            mma_ss(tmem + S::col_s(x), qx, off, kst, off, idS, s > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s_full[x]);
      };
      struct {
        int n[2], nmax;
      } I;
      for (int ii = 0; ok; ++ii) {
        int counts = 0;
        const int item = ring_get_warp_once(ring, ii, status, &ok, &counts);
        if (!ok || item < 0) break;
        I.n[0] = counts & 0xffff;
        I.n[1] = counts >> 16;
        I.nmax = I.n[0] > I.n[1] ? I.n[0] : I.n[1];
        if (!(ok = mbar_wait_warp(&bar_q_full, ii & 1, status))) break;
        if (!(ok = mbar_wait_warp(&bar_k_full[it % NS], (it / NS) & 1, status))) break;
        tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if (I.n[x] > 0) issue_s(x, it % NS);
        mma_commit(&bar_k_empty[it % NS]);
        if (I.nmax == 1) mma_commit(&bar_q_empty);
        for (int j = 0; j < I.nmax && ok; ++j) {
          const int cur = it + j, st = cur % NS;
          bool v_ready = false, k_ready = false;
          for (int x = 0; x < 2 && ok; ++x) {
            if (j >= I.n[x]) continue;
            if (!(ok = mbar_wait_warp(&bar_p_ready[x], np[x] & 1, status))) break;
            ++np[x];
            if (j == 0 && no[x] > 0 && !(ok = mbar_wait_warp(&bar_o_empty[x], (no[x] - 1) & 1, status))) break;
            if (!v_ready) {
              if (!(ok = mbar_wait_warp(&bar_v_full[st], (cur / NS) & 1, status))) break;
              v_ready = true;
            }
            tc_fence_after();
            const SmemDesc vst{dv.lo + ((st * S::kVBytes) >> 4), dv.hi};
            const uint32_t acc0 = j > 0 ? 1u : 0u;
            __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
            for (int s = 0; s < kBlockN / 16; ++s)
              mma_ts(tmem + S::col_o(x), tmem + S::col_s(x) + s * 8, vst, s * 2048, idPV,
                     s > 0 ? 1u : acc0);
            if (j + 1 < I.n[x]) {
              const int nx = cur + 1;
              if (!k_ready) {
                if (!(ok = mbar_wait_warp(&bar_k_full[nx % NS], (nx / NS) & 1, status))) break;
                k_ready = true;
              }
              tc_fence_after();
              issue_s(x, nx % NS);
            } else {
              mma_commit(&bar_o_full[x]);
            }
          }
          if (!ok) break;
          mma_commit(&bar_v_empty[st]);
          if (j + 1 < I.nmax) mma_commit(&bar_k_empty[(cur + 1) % NS]);
          if (j + 2 == I.nmax) mma_commit(&bar_q_empty);
        }
        if (!ok) break;
        for (int x = 0; x < 2; ++x)
          if (I.n[x] > 0) ++no[x];
        it += I.nmax;
      }
    }
  } else {
    // ------------------------------------------------------------- softmax A / B
    const int x = warp >> 2;  // 0: tile A, 1: tile B
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + S::col_s(x) + lane_base;
    const uint32_t t_o = tmem + S::col_o(x) + lane_base;
    using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
    int ns = 0, no = 0;  // S hand-overs and items seen by this tile
    bool ok = true;
    // Per-item values of this thread's query row. The next item is decoded (its
    // global loads issued) before this item's O rows are stored: loads queued
    // behind those scattered row stores would otherwise wait for all of them.
    struct RowItem {
      int item, n, lim;
      bool row_valid;
      size_t out_row;  // token * hq + head of this row
      int stage_before;  // staging uses of this item before this tile's (0 or 1)
      int stage_item;    // staging uses of this item (both tiles)
      bool tma;          // this tile's O leaves through the staged TMA store
      int h, tb, tok0;   // store coordinates of this tile
    };
    auto decode = [&](int item) {
      RowItem r{item, 0, 0, false, 0, 0, 0, false, 0, 0, 0};
      if (item < 0) return r;
      const FwdItem I = fwd_item(p, item, causal);
      r.n = I.n[x];
      const bool ua = I.n[0] > 0 && I.whole[0], ub = I.n[1] > 0 && I.whole[1];
      r.tma = x == 0 ? ua : ub;
      r.stage_before = x == 1 && ua ? 1 : 0;
      r.stage_item = (ua ? 1 : 0) + (ub ? 1 : 0);
      r.h = I.h;
      r.tb = I.s.tb;
      r.tok0 = I.s.off_q + (2 * I.u + x) * kBlockM;
      const int row = (2 * I.u + x) * kBlockM + quarter * 32 + lane;
      // rows that see no key (before a lower-right triangle) are the zero fill's
      r.lim = row < I.s.len_q ? row_keys(I.s, row, causal) : 0;
      r.out_row = q_row(p, I.s, row) * p.hq + I.h;
      r.row_valid = r.lim > 0 &&
                    bounds_ok(r.out_row < static_cast<size_t>(p.total_q) * p.hq, p.header + kHdrStatus);
      return r;
    };
    int stage_uses = 0, ostage_uses = 0;  // O staging uses so far (block / this tile)
    RowItem cur = decode(ring_get_warp(ring, 0, status, &ok));
    for (int ii = 0; ok && cur.item >= 0; ++ii) {
      if (cur.n == 0) {
        stage_uses += cur.stage_item;
        cur = decode(ring_get_warp(ring, ii + 1, status, &ok));
        continue;
      }
      const int n = cur.n, lim = cur.lim;
      const bool row_valid = cur.row_valid;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s_full[x], ns & 1, status));
        if (!ok) break;
        ++ns;
        tc_fence_after();
        const int nvalid = min(max(lim - j * kBlockN, 0), kBlockN);
        const bool full = __all_sync(0xffffffffu, nvalid >= kBlockN);
        const float sl2 = p.scale_log2;
        // Row max of this tile's visible scores (log2 domain), from S in TMEM.
        auto tile_max = [&]() -> float {
          float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int k = 0; k < kBlockN / 32; ++k) {
            uint32_t sv[32];
            tmem_ld32(t_s + 32 * k, sv);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c)
              mp[c & 3] = max3(mp[c & 3], 32 * k + 2 * c < nvalid ? __uint_as_float(sv[2 * c]) : -INFINITY,
                               32 * k + 2 * c + 1 < nvalid ? __uint_as_float(sv[2 * c + 1]) : -INFINITY);
          }
          return fmaxf(max3(mp[0], mp[1], mp[2]), mp[3]) * sl2;
        };
        // A row's first tile with a visible key: its max, to start the offset m.
        if (__any_sync(0xffffffffu, m == -INFINITY && nvalid > 0)) {
          const float mxs = tile_max();
          if (m == -INFINITY && nvalid > 0) m = mxs;
        }
        // One pass over S: P = exp2(S * scale*log2e - m) and its row sum, P held in
        // registers until the pass is accepted. The offset is raised lazily: only
        // when a row's max exceeds m + 8 does that row take the new max, O and l are
        // scaled by exp2(m_old - m_new) (O is final for the tiles before this one:
        // S(j) was issued after P V(j-1)) and the pass is repeated; S is still intact
        // in TMEM then, as P is written only at the end. A row whose P sums to at
        // most 2^8 has no entry above 2^8 and cannot need a raise, so the max itself
        // is taken (in a second read of S) only for rows with a larger sum -- rare
        // once a row's offset is set, and no max instructions in the common pass.
        float alpha = 1.f;
        uint64_t sp[4];
        uint32_t pk[kBlockN / 32][16];
        // the pass, as straight-line code for full tiles and for masked ones
        auto pass = [&](auto full_tag) {
          constexpr bool kFull = decltype(full_tag)::value;
          const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(-m, -m);
#pragma unroll
          for (int k = 0; k < 4; ++k) sp[k] = f2_pack(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < kBlockN / 32; ++k) {
            uint32_t sv[32];
            tmem_ld32(t_s + 32 * k, sv);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float2 xx = f2_unpack(ffma2(f2_pack(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])),
                                                sl2x2, negm2));
              float p0 = ex2f(xx.x), p1 = ex2f(xx.y);
              if constexpr (!kFull) {
                p0 = 32 * k + 2 * c < nvalid ? p0 : 0.f;
                p1 = 32 * k + 2 * c + 1 < nvalid ? p1 : 0.f;
              }
              sp[c & 3] = fadd2(sp[c & 3], f2_pack(p0, p1));
              pk[k][c] = pack2<kBF16>(p0, p1);
            }
          }
        };
        for (;;) {
          if (full)
            pass(std::true_type{});
          else
            pass(std::false_type{});
          const float2 s01 = f2_unpack(fadd2(fadd2(sp[0], sp[1]), fadd2(sp[2], sp[3])));
          if (!__any_sync(0xffffffffu, s01.x + s01.y > 256.0f)) break;
          const float mxs = tile_max();
          const bool raise = nvalid > 0 && mxs > m + 8.0f;
          if (!__any_sync(0xffffffffu, raise)) break;
          // rare: a row's max grew by more than 2^8
          if (raise) {
            alpha = ex2f(m - mxs);
            m = mxs;
          }
#pragma unroll
          for (int c0 = 0; c0 < kD; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st16(t_o + c0, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
            tmem_st16(t_o + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&o[16]));
          }
        }
        // P (16-bit) over the first half of the S columns
#pragma unroll
        for (int k = 0; k < kBlockN / 32; ++k) tmem_st16(t_s + 16 * k, pk[k]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_p_ready[x]);
        const float2 s01 = f2_unpack(fadd2(fadd2(sp[0], sp[1]), fadd2(sp[2], sp[3])));
        l = l * alpha + (s01.x + s01.y);
      }
      if (!ok) break;
      const RowItem nxt = decode(ring_get_warp(ring, ii + 1, status, &ok));
      if (!ok) break;
      // epilogue: O / l and lse for this row once the tile's last P V has landed
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_o_full[x], no & 1, status));
      if (!ok) break;
      ++no;
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      if (cur.tma) {
        // The tile's rows go to a shared-memory O tile (128-byte swizzle, as the TMA
        // loads lay out Q) and leave with one TMA store per 64 columns, issued by one
        // thread; the warps go on as soon as their rows are in shared memory. The
        // buffer serves the block's tiles in turn: use u waits for use u-1's store
        // to have read it.
        const int u = stage_uses + cur.stage_before;
        if (u > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar_stage, (u - 1) & 1, status));
        if (!ok) break;
        const int r = quarter * 32 + lane;
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c0, o);
          tmem_ld_wait();
          uint8_t* row = sO + (c0 / 64) * 16384 + r * 128;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int piece = ((c0 % 64) / 8) + v;
            st_shared_v4(row + ((piece ^ (r & 7)) << 4),
                         pack2<kBF16>(__uint_as_float(o[8 * v]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                         pack2<kBF16>(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                         pack2<kBF16>(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                         pack2<kBF16>(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
          }
        }
        tc_fence_before();
        mbar_arrive(&bar_o_empty[x]);
        fence_proxy_async_smem();
        mbar_arrive(&bar_ostage[x]);
        if (quarter == 0 && lane == 0) {
          // every row of the tile is in shared memory: store, wait for the reads, release
          if (mbar_wait(&bar_ostage[x], ostage_uses & 1, status)) {
#pragma unroll
            for (int c = 0; c < S::kChunks; ++c) tma_store_4d(&tmO, sO + c * 16384, c * 64, cur.h, cur.tb, cur.tok0);
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&bar_stage);
        }
        ++ostage_uses;
      } else {
        const auto rows = make_row_pair(static_cast<T*>(p.out) + cur.out_row * static_cast<size_t>(p.d), row_valid);
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c0, o);
          tmem_ld_wait();
          store_pair16<kBF16>(rows, c0, p.d, *reinterpret_cast<uint32_t(*)[16]>(&o[0]), inv);
          store_pair16<kBF16>(rows, c0 + 16, p.d, *reinterpret_cast<uint32_t(*)[16]>(&o[16]), inv);
        }
        tc_fence_before();
        mbar_arrive(&bar_o_empty[x]);
      }
      if (row_valid) p.lse[cur.out_row] = m * 0.69314718055994531f + logf(l);
      stage_uses += cur.stage_item;
      cur = nxt;
    }
  }

  // the stores' global writes are complete before the block ends
  if (warp < 8 && (warp & 3) == 0 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == kFwdWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int kD, bool kBF16, bool kFP8 = false>
static cudaError_t launch_fwd_pair_impl(const AttnParams& p, int num_sms, cudaStream_t st) {
  using S = FwdPairShape<kD, kFP8>;
  CUtensorMap tq, tk, tv, to;
  const int nb = p.sbhd ? p.batch : 1;
  const bool qk_ok = kFP8 ? make_tmap_tokens_u8(&tq, p.q, p.total_q, nb, p.hq, p.d) &&
                                make_tmap_tokens_u8(&tk, p.k, p.total_kv, nb, p.hkv, p.d)
                          : make_tmap_tokens(&tq, p.q, p.total_q, nb, p.hq, p.d, kBF16) &&
                                make_tmap_tokens(&tk, p.k, p.total_kv, nb, p.hkv, p.d, kBF16);
  if (!qk_ok || !make_tmap_tokens(&tv, p.v, p.total_kv, nb, p.hkv, p.d, kBF16) ||
      !make_tmap_tokens(&to, p.out, p.total_q, nb, p.hq, p.d, kBF16))
    return cudaErrorInvalidValue;
  auto kern = attn_fwd_pair_kernel<kD, kBF16, kFP8>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long max_items = static_cast<long long>(p.pair_cap_f) * p.hq;
  const int grid = static_cast<int>(max_items < num_sms ? (max_items > 0 ? max_items : 1) : num_sms);
  kern<<<grid, kFwdPairThreads, S::kSmemBytes, st>>>(p, tq, tk, tv, to);
  return cudaGetLastError();
}

// e4m3 Q and K (p.q, p.k), bf16 V (p.v), bf16 out; head_dim <= 128.
cudaError_t launch_attn_fwd_pair_e4m3(const AttnParams& p, int num_sms, cudaStream_t st) {
  return launch_fwd_pair_impl<128, true, true>(p, num_sms, st);
}

cudaError_t launch_attn_fwd_pair(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st) {
  if (bf16) return p.d <= 64 ? launch_fwd_pair_impl<64, true>(p, num_sms, st)
                             : launch_fwd_pair_impl<128, true>(p, num_sms, st);
  return p.d <= 64 ? launch_fwd_pair_impl<64, false>(p, num_sms, st)
                   : launch_fwd_pair_impl<128, false>(p, num_sms, st);
}

}  // namespace teattn

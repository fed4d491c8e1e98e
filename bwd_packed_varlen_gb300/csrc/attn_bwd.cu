// Backward attention over packed variable-length sequences on sm_103a.
//
// Two persistent tensor-core kernels with the same role split: 16 compute warps
// (warp w owns TMEM lane quarter w % 4 and a quarter of the step's columns), one
// TMA producer warp and one MMA warp (the whole warp runs the issue loop; one
// elected lane issues every tcgen05.mma). Work items
// come from the scheduler's sorted lists through a per-kernel counter and a
// shared-memory ring (see work_queue.cuh).
//
// dK/dV kernel -- item = (sequence b, key/value head g, 128-row key tile).
//   K and V of the tile stay in shared memory for the whole item; the item sweeps
//   the G query heads of the group and, for each, the query tiles that can see
//   the key tile (causal: from the diagonal on), in a fixed order:
//     S^T  = K Q^T,  dP^T = V dO^T                      (tcgen05, into TMEM)
//     P^T  = exp(S^T - lse), dS^T = P^T (dP^T - D)      (one thread per key row;
//            masked entries are selected to exact 0, so pad-slot values never
//            leak; P^T and dS^T are written back over S^T / dP^T as 16-bit)
//     dV  += P^T dO,  dK += dS^T Q                      (A operands from TMEM)
//   dK/dV accumulate in TMEM over the whole group, so the GQA reduction happens
//   inside one block with no atomics: results are deterministic.
//   For head_dim > 128 the tile sweeps 64 query rows per step and each block
//   produces half of the output columns (two blocks per item).
//
// dQ kernel -- item = (sequence b, query head h, 128-row query tile); Q and dO stay
//   in shared memory, key tiles stream through separate K and V rings: S = Q K^T,
//   dP = dO V^T, dS = P (dP - D) into one of two 16-bit TMEM buffers, dQ += dS K
//   with dQ in TMEM.
//
// Both scale by attn_scale in the epilogue and store only rows that belong to
// real tokens (and, for dK/dV, that some real query sees); every other row is
// written as exact zero by the zero-fill kernel.
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


__device__ __forceinline__ float ex2b(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kBF16>
using elem_t = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;

// ===========================================================================
// dK / dV
// ===========================================================================
// Thread roles: 16 compute warps (warp w owns TMEM lanes 32*(w%4).. and the query
// columns [(kBM/4)*(w/4), +kBM/4) of each step), then one TMA warp and one MMA warp.
// TMEM: dK at columns [0, kDo), dV at [128, 128+kDo), S^T at [256, 256+kBM) and
// dP^T at [384, 384+kBM). Each step is one query tile of kBM rows; the MMA thread
// issues  S^T_t, dP^T_t, | dV_t, S^T_t+1, dK_t, dP^T_t+1 | ...  so the tensor cores
// compute dP^T_t while the compute warps turn S^T_t into P^T_t, and dV_t / S^T_t+1
// while they turn dP^T_t into dS^T_t. P^T and dS^T are written as 16-bit values
// over the first half of each warp's own column range of S^T / dP^T.
constexpr int kBwdComputeWarps = 16;
constexpr int kBwdThreads = (kBwdComputeWarps + 2) * 32;
constexpr int kBwdComputeThreads = kBwdComputeWarps * 32;
constexpr int kWarpProducer = kBwdComputeWarps, kWarpMma = kBwdComputeWarps + 1;
constexpr int kColGroups = kBwdComputeWarps / 4;  // warps sharing one TMEM lane quarter

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// TMEM column (relative to a score buffer) of the packed 16-bit operand for
// MMA k-step s (16 rows of the reduction dimension): group g = s / (G/16) of
// width G = step / 4 keeps its packed values in the first G/2 columns of its own
// range [g*G, g*G+G).
template <int kStep>
__device__ __forceinline__ constexpr uint32_t packed_col(int s) {
  constexpr int G = kStep / kColGroups;  // columns per group
  constexpr int per = G / 16;            // k-steps per group
  return static_cast<uint32_t>((s / per) * G + (s % per) * 8);
}

template <int kD>
struct DkdvShape {
  static constexpr int kBM = kD <= 128 ? 128 : 64;   // query rows per step
  static constexpr int kSplit = kD <= 128 ? 1 : 2;   // output column halves
  static constexpr int kDo = kD / kSplit;            // output columns per block (<= 128)
  static constexpr int kChunks = kD / 64;
  static constexpr int kKVBytes = kChunks * 16384;   // one 128-row K or V tile
  static constexpr int kQBytes = kChunks * kBM * 128; // one kBM-row Q or dO tile
  static constexpr int kStageBytes = 2 * kQBytes + 2 * kBM * 4;
  static constexpr int kFixed = 2 * kKVBytes + 1024 + 2048;
  static constexpr int kStages = cmin(4, (227 * 1024 - kFixed) / kStageBytes);
  static constexpr int kSmemUsed = 2 * kKVBytes + kStages * kStageBytes + 1024;
  static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  static constexpr int kG = kBM / kColGroups;        // query columns per compute warp
  static constexpr uint32_t kColDK = 0, kColDV = 128, kColST = 256, kColDPT = 384;
  static_assert(kStages >= 1, "shared memory budget");
};

template <int kD, bool kBF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV) {
  using S = DkdvShape<kD>;
  constexpr int kBM = S::kBM, NS = S::kStages, kG = S::kG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + S::kKVBytes;
  uint8_t* sQ = sV + S::kKVBytes;             // NS stages
  uint8_t* sDO = sQ + NS * S::kQBytes;        // NS stages
  float* sLse = reinterpret_cast<float*>(sDO + NS * S::kQBytes);  // NS x kBM (log2 domain)
  float* sDelta = sLse + NS * kBM;                                 // NS x kBM

  __shared__ uint64_t bar_kv_full, bar_kv_empty, bar_acc_full, bar_acc_empty;
  __shared__ uint64_t bar_q_full[NS], bar_q_empty[NS];
  __shared__ uint64_t bar_s_full, bar_dp_full, bar_p_ready, bar_ds_ready;
  __shared__ WorkRing ring;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* status = p.header + kHdrStatus;
  const int per_pair = p.hkv * S::kSplit;
  const int n_pairs = p.header[kHdrNumKPairs];
  const int n_items = n_pairs * per_pair;
  const bool causal = p.causal != 0;

  if (tid == 0) {
    mbar_init(&bar_kv_full, 1);
    mbar_init(&bar_kv_empty, 1);
    mbar_init(&bar_acc_full, 1);
    mbar_init(&bar_acc_empty, kBwdComputeThreads);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bar_q_full[i], 1);
      mbar_init(&bar_q_empty[i], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_p_ready, kBwdComputeThreads);
    mbar_init(&bar_ds_ready, kBwdComputeThreads);
    ring_init(ring, 1 + kBwdComputeThreads);
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Per-item geometry, identical in every role.
  struct Item {
    SeqInfo s;
    int b, kt, g, split, qt0, nq, steps;
  };
  auto decode = [&](int item) {
    Item it;
    const PairHead ph = item_pair_head_banded(item, n_pairs, per_pair);
    const int2 pr = p.k_pairs[ph.pair];
    it.g = ph.head / S::kSplit;
    it.split = ph.head % S::kSplit;
    it.kt = pr.y;
    it.b = pr.x;
    it.s = load_seq(p, pr.x);
    it.qt0 = first_query(it.s, it.kt * kBlockN, causal) / kBM;
    it.nq = (it.s.len_q + kBM - 1) / kBM;
    it.steps = p.group * (it.nq - it.qt0);
    return it;
  };

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int it = 0, ii = 0;
      bool ok = true;
      int nxt = blockIdx.x;
      for (; ok; ++ii) {
        const int item = nxt < n_items ? nxt : -1;
        if (item < 0) {
          ok = ring_put(ring, ii, -1, status);
          break;
        }
        const Item I = decode(item);
        // step count and column half travel with the item: the MMA thread then
        // needs no global loads (which would queue behind the dK/dV row stores)
        if (!(ok = ring_put(ring, ii, item, status, I.steps | (I.split << 24)))) break;
        nxt = next_item(p.header + kHdrNextDkdv);  // used at the next hand-over
        if (ii > 0 && !(ok = mbar_wait(&bar_kv_empty, (ii - 1) & 1, status))) break;
        mbar_arrive_expect_tx(&bar_kv_full, 2 * S::kKVBytes);
        for (int c = 0; c < S::kChunks; ++c) {
          tma_load_4d(sK + c * 16384, &tmK, &bar_kv_full, c * 64, I.g, I.s.tb, I.s.off_k + I.kt * kBlockN);
          tma_load_4d(sV + c * 16384, &tmV, &bar_kv_full, c * 64, I.g, I.s.tb, I.s.off_k + I.kt * kBlockN);
        }
        const int nqt = I.nq - I.qt0;
        for (int t = 0; t < I.steps; ++t, ++it) {
          const int h = I.g * p.group + t / nqt;
          const int qt = I.qt0 + t % nqt;
          const int st = it % NS;
          if (it >= NS && !(ok = mbar_wait(&bar_q_empty[st], ((it / NS) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&bar_q_full[st], 2 * S::kQBytes + 2 * kBM * 4);
          for (int c = 0; c < S::kChunks; ++c) {
            tma_load_4d(sQ + st * S::kQBytes + c * kBM * 128, &tmQ, &bar_q_full[st], c * 64, h, I.s.tb,
                        I.s.off_q + qt * kBM);
            tma_load_4d(sDO + st * S::kQBytes + c * kBM * 128, &tmDO, &bar_q_full[st], c * 64, h, I.s.tb,
                        I.s.off_q + qt * kBM);
          }
          size_t ti = tiled_index(p, I.b, qt * kBM, h);
          // a bad offset still completes the barrier's byte count, from row 0
          if (!bounds_ok(ti + kBM <= static_cast<size_t>(p.pair_cap_q) * p.hq * kBlockM, status)) ti = 0;
          bulk_load(sLse + st * kBM, p.lse_t + ti, kBM * 4, &bar_q_full[st]);
          bulk_load(sDelta + st * kBM, p.delta_t + ti, kBM * 4, &bar_q_full[st]);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t idS = make_idesc_f16(kBF16, false, false, 128, kBM);
      constexpr uint32_t idAcc = make_idesc_f16(kBF16, false, true, 128, S::kDo);
      const uint32_t t_dk = tmem + S::kColDK, t_dv = tmem + S::kColDV;
      const uint32_t t_st = tmem + S::kColST, t_dpt = tmem + S::kColDPT;
      // K, V, Q, dO K-major for S^T / dP^T; dO and Q N-major (d-contiguous) for dV / dK.
      const SmemDesc dk = smem_desc(smem_u32(sK), 16, 1024, kLayoutSW128);
      const SmemDesc dv = smem_desc(smem_u32(sV), 16, 1024, kLayoutSW128);
      const SmemDesc dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
      const SmemDesc ddo = smem_desc(smem_u32(sDO), 16, 1024, kLayoutSW128);
      const SmemDesc dq_mn = smem_desc(smem_u32(sQ), kBM * 128, 1024, kLayoutSW128);
      const SmemDesc ddo_mn = smem_desc(smem_u32(sDO), kBM * 128, 1024, kLayoutSW128);
      int it = 0, ii = 0;
      bool ok = true;
      auto wait_q = [&](int cur) { return mbar_wait_warp(&bar_q_full[cur % NS], (cur / NS) & 1, status); };
      // S^T = K Q^T (A: K tile, B: Q stage) or dP^T = V dO^T for global step `cur`.
      auto issue_st = [&](int cur, uint32_t d_tmem, SmemDesc a, SmemDesc b, uint64_t* done) {
        const SmemDesc bst{b.lo + ((cur % NS) * S::kQBytes >> 4), b.hi};
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)
          mma_ss(d_tmem, a, (s >> 2) * 16384 + (s & 3) * 32, bst, (s >> 2) * (kBM * 128) + (s & 3) * 32,
                 idS, s > 0 ? 1u : 0u);
        mma_commit(done);
      };
      // dV += P^T dO or dK += dS^T Q for global step `cur` (A from TMEM).
      auto issue_acc = [&](int cur, uint32_t d_tmem, uint32_t a_tmem, SmemDesc b, uint32_t split_off,
                           uint32_t acc0) {
        const SmemDesc bst{b.lo + (((cur % NS) * S::kQBytes + split_off) >> 4), b.hi};
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s = 0; s < kBM / 16; ++s)
          mma_ts(d_tmem, a_tmem + packed_col<kBM>(s), bst, s * 2048, idAcc, s > 0 ? 1u : acc0);
      };
      struct {
        int steps, split;
      } I;
      for (; ok; ++ii) {
        int aux = 0;
        const int item = ring_get_warp_once(ring, ii, status, &ok, &aux);
        if (!ok || item < 0) break;
        I.steps = aux & 0xffffff;
        I.split = aux >> 24;
        if (!(ok = mbar_wait_warp(&bar_kv_full, ii & 1, status))) break;
        const uint32_t split_off = I.split * (S::kDo / 64) * kBM * 128;
        if (!(ok = wait_q(it))) break;
        tc_fence_after();
        issue_st(it, t_st, dk, dq, &bar_s_full);
        issue_st(it, t_dpt, dv, ddo, &bar_dp_full);
        // K and V are free once the item's last S^T and dP^T are done, so the next
        // item's tiles load while its final dV/dK products still run.
        if (I.steps == 1) mma_commit(&bar_kv_empty);
        for (int t = 0; t < I.steps; ++t) {
          const int cur = it + t;
          const bool more = t + 1 < I.steps;
          if (!(ok = mbar_wait_warp(&bar_p_ready, cur & 1, status))) break;
          if (t == 0 && ii > 0 && !(ok = mbar_wait_warp(&bar_acc_empty, (ii - 1) & 1, status))) break;
          tc_fence_after();
          issue_acc(cur, t_dv, t_st, ddo_mn, split_off, t > 0 ? 1u : 0u);
          if (NS >= 2 && more) {
            if (!(ok = wait_q(cur + 1))) break;
            tc_fence_after();
            issue_st(cur + 1, t_st, dk, dq, &bar_s_full);
          }
          if (!(ok = mbar_wait_warp(&bar_ds_ready, cur & 1, status))) break;
          tc_fence_after();
          issue_acc(cur, t_dk, t_dpt, dq_mn, split_off, t > 0 ? 1u : 0u);
          mma_commit(&bar_q_empty[cur % NS]);
          if (more) {
            if (NS == 1) {
              if (!(ok = wait_q(cur + 1))) break;
              tc_fence_after();
              issue_st(cur + 1, t_st, dk, dq, &bar_s_full);
            }
            issue_st(cur + 1, t_dpt, dv, ddo, &bar_dp_full);
            if (t + 2 == I.steps) mma_commit(&bar_kv_empty);
          }
        }
        if (!ok) break;
        it += I.steps;
        mma_commit(&bar_acc_full);
      }
    }
  } else {
    // ------------------------------------------------------------- compute
    const int quarter = warp & 3, grp = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int col0 = grp * kG;
    const float sl2 = p.scale_log2;
    int it = 0, ii = 0;
    bool ok = true;
    for (; ok; ++ii) {
      const int item = ring_get_warp(ring, ii, status, &ok);
      if (!ok || item < 0) break;

      const Item I = decode(item);
      const int kv_row = I.kt * kBlockN + quarter * 32 + lane;
      const bool kv_valid = kv_row < I.s.len_k;
      const int nqt = I.nq - I.qt0;
      // tensor row of key token 0: the loop carries one value for the epilogue
      const int kv_row0 = I.s.off_k * p.rs + I.s.tb;
      for (int t = 0; t < I.steps; ++t, ++it) {
        const int qt = I.qt0 + t % nqt;
        const int st = it % NS;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_q_full[st], (it / NS) & 1, status));
        if (!ok) break;
        // query columns i of this warp with a nonzero P^T for this key row: [lo, hi)
        const int q_base = qt * kBM + col0;
        const int hi = kv_valid ? min(kG, I.s.len_q - q_base) : 0;
        const int lo = causal ? max(0, kv_row - I.s.diag - q_base) : 0;
        // Warp-uniform: only tiles on the causal diagonal or a length boundary pay
        // for per-element masking.
        const bool full = __all_sync(0xffffffffu, lo == 0 && hi >= kG);
        const float4* lse4 = reinterpret_cast<const float4*>(sLse + st * kBM + col0);
        const float4* dlt4 = reinterpret_cast<const float4*>(sDelta + st * kBM + col0);
        // ---- phase A: P^T = exp2(S^T * scale * log2e - lse2), masked entries 0
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s_full, it & 1, status));
        if (!ok) break;
        tc_fence_after();
        float pv[kG];
        {
          uint32_t sv[kG];
          if constexpr (kG == 32) tmem_ld32(tmem + S::kColST + lane_base + col0, sv);
          else tmem_ld16(tmem + S::kColST + lane_base + col0, *reinterpret_cast<uint32_t(*)[16]>(sv));
          tmem_ld_wait();
          if (full) {
            // paired fma: one instruction for two entries, same rounding as fmaf
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
            for (int k = 0; k < kG / 4; ++k) {
              const float4 l4 = lse4[k];
              const float2 x01 = f2_unpack(ffma2(f2_pack(__uint_as_float(sv[4 * k]), __uint_as_float(sv[4 * k + 1])),
                                                 sl2x2, f2_pack(l4.x, l4.y)));
              const float2 x23 = f2_unpack(ffma2(f2_pack(__uint_as_float(sv[4 * k + 2]), __uint_as_float(sv[4 * k + 3])),
                                                 sl2x2, f2_pack(l4.z, l4.w)));
              pv[4 * k] = ex2b(x01.x);
              pv[4 * k + 1] = ex2b(x01.y);
              pv[4 * k + 2] = ex2b(x23.x);
              pv[4 * k + 3] = ex2b(x23.y);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kG / 4; ++k) {
              const float4 l4 = lse4[k];
              const float l[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 4 * k + e;
                const float x = ex2b(fmaf(__uint_as_float(sv[i]), sl2, l[e]));
                pv[i] = (i >= lo && i < hi) ? x : 0.f;
              }
            }
          }
          uint32_t pk[kG / 2];
#pragma unroll
          for (int k = 0; k < kG / 2; ++k) pk[k] = pack2<kBF16>(pv[2 * k], pv[2 * k + 1]);
          if constexpr (kG == 32) tmem_st16(tmem + S::kColST + lane_base + col0, pk);
          else tmem_st8(tmem + S::kColST + lane_base + col0, *reinterpret_cast<uint32_t(*)[8]>(pk));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_p_ready);
        // ---- phase B: dS^T = P^T (dP^T - D)
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_dp_full, it & 1, status));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dv[kG];
          if constexpr (kG == 32) tmem_ld32(tmem + S::kColDPT + lane_base + col0, dv);
          else tmem_ld16(tmem + S::kColDPT + lane_base + col0, *reinterpret_cast<uint32_t(*)[16]>(dv));
          tmem_ld_wait();
          // Masked entries are selected to 0 (not multiplied): D of rows past the
          // query length is never written and may hold any bits.
          float r[kG];
          // paired subtract and multiply: the same two roundings per entry
#pragma unroll
          for (int k = 0; k < kG / 4; ++k) {
            const float4 d4 = dlt4[k];
            const float2 r01 = f2_unpack(fmul2(f2_pack(pv[4 * k], pv[4 * k + 1]),
                                               fadd2(f2_pack(__uint_as_float(dv[4 * k]), __uint_as_float(dv[4 * k + 1])),
                                                     f2_pack(d4.x, d4.y))));
            const float2 r23 = f2_unpack(fmul2(f2_pack(pv[4 * k + 2], pv[4 * k + 3]),
                                               fadd2(f2_pack(__uint_as_float(dv[4 * k + 2]), __uint_as_float(dv[4 * k + 3])),
                                                     f2_pack(d4.z, d4.w))));
            r[4 * k] = r01.x;
            r[4 * k + 1] = r01.y;
            r[4 * k + 2] = r23.x;
            r[4 * k + 3] = r23.y;
          }
          if (!full) {
#pragma unroll
            for (int i = 0; i < kG; ++i) r[i] = (i >= lo && i < hi) ? r[i] : 0.f;
          }
          uint32_t dk[kG / 2];
#pragma unroll
          for (int k = 0; k < kG / 2; ++k) dk[k] = pack2<kBF16>(r[2 * k], r[2 * k + 1]);
          if constexpr (kG == 32) tmem_st16(tmem + S::kColDPT + lane_base + col0, dk);
          else tmem_st8(tmem + S::kColDPT + lane_base + col0, *reinterpret_cast<uint32_t(*)[8]>(dk));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_ds_ready);
      }
      if (!ok) break;
      // Epilogue: scale * dK and dV for rows some real query sees; each column group
      // of the compute warps stores a quarter of the columns.
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc_full, ii & 1, status));
      if (!ok) break;
      tc_fence_after();
      const size_t kv_tok = static_cast<size_t>(kv_row0) + static_cast<size_t>(kv_row) * p.rs;
      const bool store = kv_row < seen_keys(I.s, causal) &&
                         bounds_ok(kv_tok < static_cast<size_t>(p.total_kv), status);
      const size_t kv_off = (kv_tok * p.hkv + I.g) * p.d;
      const auto dk_rows = make_row_pair(static_cast<elem_t<kBF16>*>(p.dk) + kv_off, store);
      const auto dv_rows = make_row_pair(static_cast<elem_t<kBF16>*>(p.dv) + kv_off, store);
      const int col_out = I.split * S::kDo;
      constexpr int kOutCols = S::kDo / kColGroups;
#pragma unroll
      for (int c = 0; c < kOutCols; c += 16) {
        const int c0 = grp * kOutCols + c;
        uint32_t a[16], b[16];
        tmem_ld16(tmem + S::kColDK + lane_base + c0, a);
        tmem_ld16(tmem + S::kColDV + lane_base + c0, b);
        tmem_ld_wait();
        store_pair16<kBF16>(dk_rows, col_out + c0, p.d, a, p.scale);
        store_pair16<kBF16>(dv_rows, col_out + c0, p.d, b, 1.0f);
      }
      tc_fence_before();
      mbar_arrive(&bar_acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// dQ
// ===========================================================================
// Same role split as dK/dV: compute warp w owns query rows 32*(w%4).. and key
// columns [(kBN/4)*(w/4), +kBN/4) of each step. TMEM: dQ at [0, kD), S at kColS,
// dP at kColDP and two packed 16-bit dS buffers at kColDS (step j uses buffer j%2).
// The MMA thread stops twice per step: it issues S_j+1 once the compute warps have
// read S_j, then dQ_j and dP_j+1 together once they have written dS_j. Every stop
// between MMA groups (a wait, even a commit) leaves the tensor pipe idle for about
// a hundred cycles, so the compute warps, which have slack, also do the K/V ring
// bookkeeping: they check that the next K and V tiles have landed before they
// arrive, and hand the stages back to the producer when the MMA commits show them
// read.
// K and V stream through separate rings: a K tile is read until dQ_j, late in
// step j, and S_j+1 wants the next one early, so the K ring is the deeper one;
// a V tile is free as soon as dP_j has read it.
template <int kD>
struct DqShape {
  static constexpr int kBN = kD <= 128 ? 128 : 64;     // key rows per step
  static constexpr int kChunks = kD / 64;
  static constexpr int kQBytes = kChunks * 16384;      // 128-row Q or dO tile
  static constexpr int kKVBytes = kChunks * kBN * 128; // kBN-row K or V tile
  static constexpr int kFixed = 2 * kQBytes + 1024 + 2048;
  static constexpr int kTiles = cmin(8, (227 * 1024 - kFixed) / kKVBytes);  // K + V stages
  static constexpr int kKStages = cmin(4, (kTiles + 1) / 2);
  static constexpr int kVStages = cmin(4, kTiles - kKStages);
  static constexpr int kSmemUsed = 2 * kQBytes + (kKStages + kVStages) * kKVBytes + 1024;
  static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  static constexpr int kG = kBN / kColGroups;          // key columns per compute warp
  static constexpr uint32_t kColDQ = 0, kColS = kD <= 128 ? 128 : 256, kColDP = kColS + kBN;
  static constexpr uint32_t kColDS = kColDP + kBN, kDsCols = kBN / 2;  // two dS buffers
  static_assert(kColDS + 2 * kDsCols <= 512, "TMEM budget");
  static_assert(kKStages >= 2 && kVStages >= 1, "shared memory budget");
};

template <int kD, bool kBF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
  using S = DqShape<kD>;
  constexpr int kBN = S::kBN, KS = S::kKStages, VS = S::kVStages, kG = S::kG;
  // With three or more K stages, K_j+1 can land while step j still holds K_j and
  // K_j-1, so S_j+1 is issued as soon as S_j has been read; with two, K_j+1 reuses
  // the stage of K_j-1, which dQ_j-1 frees only during step j, so S_j+1 goes out
  // with dQ_j.
  constexpr bool kEarlyS = KS >= 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = sQ + S::kQBytes;
  uint8_t* sK = sDO + S::kQBytes;          // KS stages
  uint8_t* sV = sK + KS * S::kKVBytes;     // VS stages

  __shared__ uint64_t bar_q_full, bar_q_empty, bar_acc_full, bar_acc_empty;
  __shared__ uint64_t bar_k_full[KS], bar_k_empty[KS], bar_v_full[VS], bar_v_empty[VS];
  __shared__ uint64_t bar_s_full, bar_dp_full, bar_s_free, bar_ds_ready;
  __shared__ WorkRing ring;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* status = p.header + kHdrStatus;
  const int n_pairs = p.header[kHdrNumQPairs];
  const int n_items = n_pairs * p.hq;
  const bool causal = p.causal != 0;

  if (tid == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 1);
    mbar_init(&bar_acc_full, 1);
    mbar_init(&bar_acc_empty, kBwdComputeThreads);
    for (int i = 0; i < KS; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_empty[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_v_empty[i], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_s_free, kBwdComputeThreads);
    mbar_init(&bar_ds_ready, kBwdComputeThreads);
    ring_init(ring, 1 + kBwdComputeThreads);
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int it = 0, ii = 0;
      bool ok = true;
      int nxt = blockIdx.x;
      for (; ok; ++ii) {
        int item = nxt < n_items ? nxt : -1;
        int2 pr;
        SeqInfo s;
        int n = 0;
        // Query tiles that see no key (rows before a lower-right causal triangle)
        // are left to the zero fill and never reach the ring.
        PairHead ph{0, 0};
        while (item >= 0) {
          ph = item_pair_head(item, n_pairs, p.group);
          pr = p.q_pairs[ph.pair];
          s = load_seq(p, pr.x);
          n = (visible_keys(s, pr.y, causal) + kBN - 1) / kBN;
          if (n > 0) break;
          nxt = next_item(p.header + kHdrNextDq);
          item = nxt < n_items ? nxt : -1;
        }
        if (item < 0) {
          ok = ring_put(ring, ii, -1, status);
          break;
        }
        const int h = ph.head, g = h / p.group;
        // the step count travels with the item: the MMA thread then needs no global loads
        if (!(ok = ring_put(ring, ii, item, status, n))) break;
        nxt = next_item(p.header + kHdrNextDq);  // used at the next hand-over
        if (ii > 0 && !(ok = mbar_wait(&bar_q_empty, (ii - 1) & 1, status))) break;
        mbar_arrive_expect_tx(&bar_q_full, 2 * S::kQBytes);
        for (int c = 0; c < S::kChunks; ++c) {
          tma_load_4d(sQ + c * 16384, &tmQ, &bar_q_full, c * 64, h, s.tb, s.off_q + pr.y * kBlockM);
          tma_load_4d(sDO + c * 16384, &tmDO, &bar_q_full, c * 64, h, s.tb, s.off_q + pr.y * kBlockM);
        }
        for (int j = 0; j < n; ++j, ++it) {
          const int sk = it % KS, sv = it % VS;
          if (it >= KS && !(ok = mbar_wait(&bar_k_empty[sk], ((it / KS) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&bar_k_full[sk], S::kKVBytes);
          for (int c = 0; c < S::kChunks; ++c)
            tma_load_4d(sK + sk * S::kKVBytes + c * kBN * 128, &tmK, &bar_k_full[sk], c * 64, g, s.tb,
                        s.off_k + j * kBN);
          if (it >= VS && !(ok = mbar_wait(&bar_v_empty[sv], ((it / VS) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&bar_v_full[sv], S::kKVBytes);
          for (int c = 0; c < S::kChunks; ++c)
            tma_load_4d(sV + sv * S::kKVBytes + c * kBN * 128, &tmV, &bar_v_full[sv], c * 64, g, s.tb,
                        s.off_k + j * kBN);
        }
      }
    }
  } else if (warp == kWarpMma) {
    {
      constexpr uint32_t idS = make_idesc_f16(kBF16, false, false, 128, kBN);
      constexpr uint32_t idDQ = make_idesc_f16(kBF16, false, true, 128, kD);
      const uint32_t t_dq = tmem + S::kColDQ, t_s = tmem + S::kColS, t_dp = tmem + S::kColDP;
      const uint32_t t_ds = tmem + S::kColDS;
      // Q, dO, K, V K-major for S / dP; K N-major (d-contiguous) for dS K.
      const SmemDesc dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
      const SmemDesc ddo = smem_desc(smem_u32(sDO), 16, 1024, kLayoutSW128);
      const SmemDesc dk = smem_desc(smem_u32(sK), 16, 1024, kLayoutSW128);
      const SmemDesc dv = smem_desc(smem_u32(sV), 16, 1024, kLayoutSW128);
      const SmemDesc dk_mn = smem_desc(smem_u32(sK), kBN * 128, 1024, kLayoutSW128);
      int it = 0, ii = 0;
      bool ok = true;
      auto wait_k = [&](int cur) { return mbar_wait_warp(&bar_k_full[cur % KS], (cur / KS) & 1, status); };
      auto wait_v = [&](int cur) { return mbar_wait_warp(&bar_v_full[cur % VS], (cur / VS) & 1, status); };
      // S = Q K^T (a = Q, b = K stage) or dP = dO V^T (a = dO, b = V stage).
      auto issue_s = [&](int stage, uint32_t d_tmem, SmemDesc a, SmemDesc b, uint64_t* done) {
        const SmemDesc bst{b.lo + (stage * S::kKVBytes >> 4), b.hi};
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s2 = 0; s2 < kD / 16; ++s2)
          mma_ss(d_tmem, a, (s2 >> 2) * 16384 + (s2 & 3) * 32, bst, (s2 >> 2) * (kBN * 128) + (s2 & 3) * 32,
                 idS, s2 > 0 ? 1u : 0u);
        mma_commit(done);
      };
      for (; ok; ++ii) {
        int n = 0;
        const int item = ring_get_warp_once(ring, ii, status, &ok, &n);
        if (!ok || item < 0) break;
        if (!(ok = mbar_wait_warp(&bar_q_full, ii & 1, status))) break;
        if (!(ok = wait_k(it))) break;
        if (!(ok = wait_v(it))) break;
        tc_fence_after();
        issue_s(it % KS, t_s, dq, dk, &bar_s_full);
        issue_s(it % VS, t_dp, ddo, dv, &bar_dp_full);
        // Q and dO are free once the item's last S and dP are done: the next item's
        // tiles then load while its final dQ steps still run.
        if (n == 1) mma_commit(&bar_q_empty);
        // Two hand-overs per step. The compute warps arrive on s_free once they
        // have read S_j and K_j+1 has landed, and on ds_ready once dS_j is written
        // (dP_j read) and V_j+1 has landed; they hand the V stages (and, without
        // early S, the K stages) back to the producer. With early S this thread
        // returns K stage j by a commit behind dQ_j, its last reader.
        for (int j = 0; j < n; ++j) {
          const int cur = it + j;
          const bool more = j + 1 < n;
          if (kEarlyS && more) {
            if (!(ok = mbar_wait_warp(&bar_s_free, cur & 1, status))) break;
            tc_fence_after();
            issue_s((cur + 1) % KS, t_s, dq, dk, &bar_s_full);
          }
          if (!(ok = mbar_wait_warp(&bar_ds_ready, cur & 1, status))) break;
          if (j == 0 && ii > 0 && !(ok = mbar_wait_warp(&bar_acc_empty, (ii - 1) & 1, status))) break;
          tc_fence_after();
          // Early-S order: dP_j+1 goes ahead of dQ_j (its region was read before
          // ds_ready_j), so the compute warps start on dS_j+1 while the tensor
          // cores run dQ_j; a commit after dQ_j hands K stage j back.
          if (kEarlyS && more) issue_s((cur + 1) % VS, t_dp, ddo, dv, &bar_dp_full);
          const SmemDesc kst{dk_mn.lo + ((cur % KS) * S::kKVBytes >> 4), dk_mn.hi};
          const uint32_t a_ds = t_ds + (cur & 1) * S::kDsCols;
          const uint32_t acc0 = j > 0 ? 1u : 0u;
          __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
          for (int s2 = 0; s2 < kBN / 16; ++s2)
            mma_ts(t_dq, a_ds + s2 * 8, kst, s2 * 2048, idDQ, s2 > 0 ? 1u : acc0);
          if (kEarlyS) mma_commit(&bar_k_empty[cur % KS]);
          if (!kEarlyS && more) issue_s((cur + 1) % KS, t_s, dq, dk, &bar_s_full);
          // here dp_full of step j+1 also covers dQ_j: K_j is free once it fires
          if (!kEarlyS && more) issue_s((cur + 1) % VS, t_dp, ddo, dv, &bar_dp_full);
          if (j + 2 == n) mma_commit(&bar_q_empty);
        }
        if (!ok) break;
        it += n;
        mma_commit(&bar_acc_full);
      }
    }
  } else {
    const int quarter = warp & 3, grp = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int col0 = grp * kG;
    const float sl2 = p.scale_log2;
    // The K/V ring bookkeeping of the compute warps (the readiness waits before
    // s_free and ds_ready, the V stage release) is done by lane 0 of the last
    // compute warp: warp 0 finishes its share of each phase last on its SM
    // sub-partition, and the waits there delayed both hand-overs (measured: dQ
    // -1.3 % with the bookkeeping in the last warp).
    constexpr int kRingThread = kBwdComputeThreads - 32;
    // Per-item values of this thread's query row. The next item is decoded (its
    // global loads issued) before this item's dQ rows are stored: loads queued
    // behind those scattered row stores would otherwise wait for all of them.
    struct RowItem {
      int item, n, lim;
      bool row_valid;
      size_t gi;
      float nlse2, ndlt;  // -lse * log2(e) and -D of this row
    };
    auto decode = [&](int item) {
      RowItem r{item, 0, 0, false, 0, 0.f, 0.f};
      if (item < 0) return r;
      const PairHead ph = item_pair_head(item, n_pairs, p.group);
      const int2 pr = p.q_pairs[ph.pair];
      const int h = ph.head;
      const SeqInfo s = load_seq(p, pr.x);
      r.n = (visible_keys(s, pr.y, causal) + kBN - 1) / kBN;
      const int row = pr.y * kBlockM + quarter * 32 + lane;
      // rows that see no key (before a lower-right triangle) are the zero fill's
      r.lim = row < s.len_q ? row_keys(s, row, causal) : 0;
      r.gi = q_row(p, s, row) * p.hq + h;
      const size_t ti = tiled_index(p, pr.x, row, h);
      r.row_valid = r.lim > 0 &&
                    bounds_ok(r.gi < static_cast<size_t>(p.total_q) * p.hq &&
                                  ti < static_cast<size_t>(p.pair_cap_q) * p.hq * kBlockM,
                              status);
      r.nlse2 = r.row_valid ? p.lse_t[ti] : 0.f;
      r.ndlt = r.row_valid ? p.delta_t[ti] : 0.f;
      return r;
    };
    int it = 0, ii = 0;
    bool ok = true;
    RowItem cur = decode(ring_get_warp(ring, 0, status, &ok));
    for (; ok && cur.item >= 0; ++ii) {
      const int n = cur.n, lim = cur.lim;
      const float nlse2 = cur.nlse2, ndlt = cur.ndlt;
      for (int j = 0; j < n; ++j, ++it) {
        const int nvalid = lim - (j * kBN + col0);
        // ---- phase A: P = exp2(S * scale * log2e - nlse2) into registers, then free S
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s_full, it & 1, status));
        if (!ok) break;
        tc_fence_after();
        float pv[kG];
        {
          uint32_t sv[kG];
          if constexpr (kG == 32) tmem_ld32(tmem + S::kColS + lane_base + col0, sv);
          else tmem_ld16(tmem + S::kColS + lane_base + col0, *reinterpret_cast<uint32_t(*)[16]>(sv));
          tmem_ld_wait();
          if (kEarlyS && tid == kRingThread && j + 1 < n)
            ok = mbar_wait(&bar_k_full[(it + 1) % KS], ((it + 1) / KS) & 1, status);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_before();
          mbar_arrive(&bar_s_free);
          if (__all_sync(0xffffffffu, nvalid >= kG)) {
            // paired fma: one instruction for two entries, same rounding as fmaf
            const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(nlse2, nlse2);
#pragma unroll
            for (int i = 0; i < kG; i += 2) {
              const float2 xx = f2_unpack(ffma2(f2_pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])),
                                                sl2x2, nl2));
              pv[i] = ex2b(xx.x);
              pv[i + 1] = ex2b(xx.y);
            }
          } else {
#pragma unroll
            for (int i = 0; i < kG; ++i) {
              const float x = ex2b(fmaf(__uint_as_float(sv[i]), sl2, nlse2));
              pv[i] = i < nvalid ? x : 0.f;
            }
          }
        }
        // ---- phase B: dS = P (dP - D), packed into dS buffer it % 2
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_dp_full, it & 1, status));
        if (!ok) break;
        tc_fence_after();
        if (tid == kRingThread) {
          // dP_it is done, so V stage it is free; without early S, past an item's
          // first step the commit also covered dQ_(it-1), the last reader of K
          // stage it-1 (with early S the MMA thread commits K stages itself).
          mbar_arrive(&bar_v_empty[it % VS]);
          if (!kEarlyS && j > 0) mbar_arrive(&bar_k_empty[(it - 1) % KS]);
        }
        {
          uint32_t dv[kG];
          if constexpr (kG == 32) tmem_ld32(tmem + S::kColDP + lane_base + col0, dv);
          else tmem_ld16(tmem + S::kColDP + lane_base + col0, *reinterpret_cast<uint32_t(*)[16]>(dv));
          tmem_ld_wait();
          // paired subtract and multiply: the same two roundings per entry
          uint32_t dd[kG / 2];
          const uint64_t nd2 = f2_pack(ndlt, ndlt);
#pragma unroll
          for (int k = 0; k < kG / 2; ++k) {
            const float2 r = f2_unpack(fmul2(f2_pack(pv[2 * k], pv[2 * k + 1]),
                                             fadd2(f2_pack(__uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1])), nd2)));
            dd[k] = pack2<kBF16>(r.x, r.y);
          }
          const uint32_t ds_col = S::kColDS + (it & 1) * S::kDsCols + grp * (kG / 2);
          if constexpr (kG == 32) tmem_st16(tmem + ds_col + lane_base, dd);
          else tmem_st8(tmem + ds_col + lane_base, *reinterpret_cast<uint32_t(*)[8]>(dd));
        }
        tmem_st_wait();
        if (!kEarlyS && tid == kRingThread && j + 1 < n)
          ok = mbar_wait(&bar_k_full[(it + 1) % KS], ((it + 1) / KS) & 1, status);
        if (tid == kRingThread && j + 1 < n)
          ok = ok && mbar_wait(&bar_v_full[(it + 1) % VS], ((it + 1) / VS) & 1, status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_before();
        mbar_arrive(&bar_ds_ready);
      }
      if (!ok) break;
      const RowItem nxt = decode(ring_get_warp(ring, ii + 1, status, &ok));
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc_full, ii & 1, status));
      if (!ok) break;
      tc_fence_after();
      if (!kEarlyS && tid == kRingThread) mbar_arrive(&bar_k_empty[(it - 1) % KS]);  // the item's last dQ
      const auto rows = make_row_pair(static_cast<elem_t<kBF16>*>(p.dq) + cur.gi * p.d, cur.row_valid);
      constexpr int kOutCols = kD / kColGroups;
#pragma unroll
      for (int c = 0; c < kOutCols; c += 16) {
        const int c0 = grp * kOutCols + c;
        uint32_t a[16];
        tmem_ld16(tmem + S::kColDQ + lane_base + c0, a);
        tmem_ld_wait();
        store_pair16<kBF16>(rows, c0, p.d, a, p.scale);
      }
      tc_fence_before();
      mbar_arrive(&bar_acc_empty);
      cur = nxt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// Launchers
// ===========================================================================
template <int kD, bool kBF16>
static cudaError_t launch_dkdv_impl(const AttnParams& p, int num_sms, cudaStream_t st) {
  using S = DkdvShape<kD>;
  CUtensorMap tq, tdo, tk, tv;
  const int nb = p.sbhd ? p.batch : 1;
  if (!make_tmap_tokens(&tq, p.q, p.total_q, nb, p.hq, p.d, kBF16, S::kBM) ||
      !make_tmap_tokens(&tdo, p.dout, p.total_q, nb, p.hq, p.d, kBF16, S::kBM) ||
      !make_tmap_tokens(&tk, p.k, p.total_kv, nb, p.hkv, p.d, kBF16, 128) ||
      !make_tmap_tokens(&tv, p.v, p.total_kv, nb, p.hkv, p.d, kBF16, 128))
    return cudaErrorInvalidValue;
  auto kern = attn_bwd_dkdv_kernel<kD, kBF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long max_items = static_cast<long long>(p.pair_cap_k) * p.hkv * S::kSplit;
  const int grid = static_cast<int>(max_items < num_sms ? (max_items > 0 ? max_items : 1) : num_sms);
  kern<<<grid, kBwdThreads, S::kSmemBytes, st>>>(p, tq, tdo, tk, tv);
  return cudaGetLastError();
}

template <int kD, bool kBF16>
static cudaError_t launch_dq_impl(const AttnParams& p, int num_sms, cudaStream_t st) {
  using S = DqShape<kD>;
  CUtensorMap tq, tdo, tk, tv;
  const int nb = p.sbhd ? p.batch : 1;
  if (!make_tmap_tokens(&tq, p.q, p.total_q, nb, p.hq, p.d, kBF16, 128) ||
      !make_tmap_tokens(&tdo, p.dout, p.total_q, nb, p.hq, p.d, kBF16, 128) ||
      !make_tmap_tokens(&tk, p.k, p.total_kv, nb, p.hkv, p.d, kBF16, S::kBN) ||
      !make_tmap_tokens(&tv, p.v, p.total_kv, nb, p.hkv, p.d, kBF16, S::kBN))
    return cudaErrorInvalidValue;
  auto kern = attn_bwd_dq_kernel<kD, kBF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long max_items = static_cast<long long>(p.pair_cap_q) * p.hq;
  const int grid = static_cast<int>(max_items < num_sms ? (max_items > 0 ? max_items : 1) : num_sms);
  kern<<<grid, kBwdThreads, S::kSmemBytes, st>>>(p, tq, tdo, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dkdv(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st) {
  const int d = p.d;
  if (bf16) {
    if (d <= 64) return launch_dkdv_impl<64, true>(p, num_sms, st);
    if (d <= 128) return launch_dkdv_impl<128, true>(p, num_sms, st);
    return launch_dkdv_impl<256, true>(p, num_sms, st);
  }
  if (d <= 64) return launch_dkdv_impl<64, false>(p, num_sms, st);
  if (d <= 128) return launch_dkdv_impl<128, false>(p, num_sms, st);
  return launch_dkdv_impl<256, false>(p, num_sms, st);
}

cudaError_t launch_attn_bwd_dq(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st) {
  const int d = p.d;
  if (bf16) {
    if (d <= 64) return launch_dq_impl<64, true>(p, num_sms, st);
    if (d <= 128) return launch_dq_impl<128, true>(p, num_sms, st);
    return launch_dq_impl<256, true>(p, num_sms, st);
  }
  if (d <= 64) return launch_dq_impl<64, false>(p, num_sms, st);
  if (d <= 128) return launch_dq_impl<128, false>(p, num_sms, st);
  return launch_dq_impl<256, false>(p, num_sms, st);
}

}  // namespace teattn

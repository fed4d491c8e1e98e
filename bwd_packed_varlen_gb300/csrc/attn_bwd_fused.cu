// Fused backward (head_dim <= 128): dK, dV and dQ in one persistent kernel, with a
// deterministic dQ.
//
// Item = (sequence b, key/value head g, 128-row key tile kt), as in the dK/dV
// kernel: K and V stay in shared memory, the item sweeps the query tiles that see
// the key tile and, inside each, the G query heads of the group (step t: query tile
// qt0 + t / G, head g*G + t % G). Per step, on the tensor cores:
//   S^T  = K Q^T           -> TMEM X   (fp32)      P^T, dS^T written back into X
//   dP^T = V dO^T          -> TMEM Y   (fp32)
//   dV  += P^T dO          (A = P^T from X)
//   dK  += dS^T Q          (A = dS^T from X)
//   dQ_t = dS K            -> TMEM Y   (A = dS from a shared-memory tile)
// so the backward runs its five products once each: no recomputation of S and dP
// for dQ. dK and dV accumulate in TMEM over the whole item (the GQA reduction
// stays inside the block, no atomics); dQ_t is this key tile's share of one
// (query tile, head) dQ tile, which several key tiles -- several blocks -- add to.
//
// Deterministic dQ: every (query tile, head) tile has an fp32 accumulator in the
// workspace and an int semaphore counting the key tiles that have added to it. The
// key tiles that see query tile qt are exactly kt = 0 .. last(qt) (the masks are
// prefix masks), and they add in descending order: key tile kt waits until the
// count equals last(qt) - kt, then adds (the first one stores), then increments the
// count. The order is fixed, so every element is the same fp32 sum in the same
// order on every call.
//
// Why no wait can starve: items are claimed in list order from one counter
// (every claim, including each block's first, is an atomic increment), and the
// scheduler lists, within each (sequence, head group) chain, key tile kt + 1
// before kt (chain-major: a chain's key tiles are consecutive items, so they run
// together and the dQ tiles they add to stay in L2). A block waits only on contributions of key tile kt + 1 of its own
// chain, i.e. on items claimed before its own. Take the earliest-claimed item that
// has not finished: the block that claimed it is working on it (its own earlier
// items are finished, by the choice of item), and every item it waits on was
// claimed earlier and has finished, so it runs to completion; by induction every
// item does. Waits are bounded anyway (4 s, then TE_STATUS_TIMEOUT and unwinding).
// The same order puts each dependency G steps ahead: key tile kt + 1 reaches query
// tile qt one query tile (G steps) earlier in its sweep than key tile kt does.
//
// Roles (768 threads, six warpgroups): 16 compute warps (warp w owns TMEM lanes
// 32*(w%4).. and query columns [32*(w/4), +32) of S^T and dP^T, output columns
// [kD/4*(w/4), +kD/4) of dK and dV); a TMA producer warp; an MMA warp (one elected
// lane issues every tcgen05.mma); two reducer warps (lane 0) that add the staged dQ tiles of
// even and odd steps to the accumulator with bulk reductions; and four drain warps
// (one per TMEM lane quarter) that read dQ_t out of TMEM and stage it, so neither
// the compute warps nor the MMA warp ever wait on dQ's way to global memory. dQ_t
// is staged in the step's Q and dO buffers (columns [0, kD/2) and [kD/2, kD) in
// fp32), which are free once dQ_t is done: their last readers, dK_t and dV_t, ran
// before it. The producer refills the stage once the reducer has read the staged
// tile, so a reducer has a whole step to take its tile. Registers: launched at 80
// a thread, the compute warpgroups take 96 and the others give up to 48
// (512 * 96 + 256 * 48 = 768 * 80).
// A block claims its next item only once it has issued the loads of its current
// item's last step, so items start about in the order they are claimed and the key
// tile a block waits on is normally already ahead of it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "row_store.cuh"
#include "sm103_ptx.cuh"
#include "tmap.h"
#include "work_queue.cuh"

namespace teattn {

namespace {

__device__ __forceinline__ float ex2_fused(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kBF16>
using fused_elem_t = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;

constexpr int kFusedComputeWarps = 16;
constexpr int kFusedComputeThreads = kFusedComputeWarps * 32;
constexpr int kFusedWarpProducer = 16, kFusedWarpMma = 17, kFusedWarpReducer = 18;
constexpr int kFusedWarpDrain = 20, kFusedDrainThreads = 4 * 32;
constexpr int kFusedThreads = 24 * 32;
// per-thread registers after the split (launch: 65536 / 768 rounded down to 80)
constexpr int kFusedRegsCompute = 96, kFusedRegsOther = 48;
static_assert(16 * 32 * kFusedRegsCompute + 8 * 32 * kFusedRegsOther == kFusedThreads * 80,
              "register split must equal the launch allocation");

// Barriers and the work ring live at the end of dynamic shared memory (the kernel
// has no static shared memory, so the dynamic base keeps its 1024-byte alignment).
struct FusedBars {
  uint64_t kv_full, kv_empty, acc_full, acc_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, dq_full, y_free;
  uint64_t stage_full[2];
  WorkRing ring;
  uint32_t tmem_slot;
};

}  // namespace

template <int kD>
struct FusedShape {
  static_assert(kD == 64 || kD == 128, "fused backward: head_dim up to 128");
  static constexpr int kBM = 128;                      // query rows per step
  static constexpr int kChunks = kD / 64;              // 64-column chunks of a row
  static constexpr int kTileBytes = kChunks * 16384;   // one 128-row K, V, Q or dO tile
  static constexpr int kStages = 2;                    // Q / dO stages
  static constexpr int kDSBytes = 32768;               // dS: 128 keys x 128 queries, 16-bit
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;
  static constexpr int kOffLse = kOffDS + kDSBytes;
  static constexpr int kOffDelta = kOffLse + kStages * kBM * 4;
  static constexpr int kOffBar = kOffDelta + kStages * kBM * 4;
  static constexpr int kSmemBytes = kOffBar + 1024;
  // dQ staging: two halves of kD/2 fp32 columns, each exactly one Q or dO buffer
  static constexpr int kHalfBytes = kBM * (kD / 2) * 4;
  static constexpr int kHalfRowBytes = (kD / 2) * 4;
  static_assert(kHalfBytes == kTileBytes, "a staging half fills one Q or dO buffer");
  static constexpr int kG = 32;                        // query columns per compute warp
  static constexpr int kOutCols = kD / 4;              // output columns per compute warp
  static constexpr uint32_t kColDK = 0, kColDV = 128, kColX = 256, kColY = 384;
  static_assert(sizeof(FusedBars) <= 1024, "barrier area");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// TMEM column (relative to X) of the packed 16-bit operand for MMA k-step s (16
// query rows): the compute warps of column group c keep their 32 columns' packed
// values in [32c, 32c+16) (P^T) and [32c+16, 32c+32) (dS^T).
__device__ __forceinline__ constexpr uint32_t fused_packed_col(int s) {
  return static_cast<uint32_t>((s >> 1) * 32 + (s & 1) * 8);
}

template <int kD, bool kBF16>
__global__ void __launch_bounds__(kFusedThreads, 1)
    attn_bwd_fused_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV) {
  using S = FusedShape<kD>;
  constexpr int kBM = S::kBM, kG = S::kG;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sK = smem + S::kOffK;
  uint8_t* sV = smem + S::kOffV;
  uint8_t* sQ = smem + S::kOffQ;
  uint8_t* sDO = smem + S::kOffDO;
  uint8_t* sDS = smem + S::kOffDS;
  float* sLse = reinterpret_cast<float*>(smem + S::kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + S::kOffDelta);
  FusedBars& B = *reinterpret_cast<FusedBars*>(smem + S::kOffBar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* status = p.header + kHdrStatus;
  // Every 128-byte-swizzled tile assumes a 1024-byte aligned base.
  if (smem_u32(smem) & 1023u) {
    if (tid == 0) atomicOr(status, kStatusInternal);
    return;
  }
  const int n_items = p.header[kHdrNumKPairs] * p.hkv;
  const bool causal = p.causal != 0;
  const int G = p.group;

  if (tid == 0) {
    mbar_init(&B.kv_full, 1);
    mbar_init(&B.kv_empty, 1);
    mbar_init(&B.acc_full, 1);
    mbar_init(&B.acc_empty, kFusedComputeThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.q_full[i], 1);
      mbar_init(&B.q_empty[i], 1);
      mbar_init(&B.stage_full[i], 4);
    }
    mbar_init(&B.s_full, 1);
    mbar_init(&B.dp_full, 1);
    mbar_init(&B.p_ready, kFusedComputeThreads);
    mbar_init(&B.ds_ready, kFusedComputeThreads);
    mbar_init(&B.dq_full, 1);
    mbar_init(&B.y_free, kFusedDrainThreads);
    ring_init(B.ring, 1 + kFusedComputeThreads + 2 + kFusedDrainThreads);
    fence_barrier_init();
  }
  if (warp == kFusedWarpMma) {
    tmem_alloc(&B.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_slot;

  struct Item {
    SeqInfo s;
    int b, kt, g, qt0, nq, steps;
  };
  auto decode = [&](int item) {
    Item it;
    const int4 e = p.k_items[item];
    it.b = e.x;
    it.kt = e.y;
    it.g = e.z;
    it.s = load_seq(p, e.x);
    it.qt0 = first_query(it.s, it.kt * kBlockN, causal) / kBM;
    it.nq = (it.s.len_q + kBM - 1) / kBM;
    it.steps = G * (it.nq - it.qt0);
    return it;
  };

  if (warp >= kFusedComputeWarps) {
  // Warpgroups 4 and 5 (producer, MMA, reducers, drain) give registers back; each
  // warpgroup executes the same setmaxnreg before splitting into its roles.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFusedRegsOther));
  if (warp == kFusedWarpProducer) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int it = 0, ii = 0;
      bool ok = true;
      int nxt = atomicAdd(p.header + kHdrNextFused, 1);
      for (; ok; ++ii) {
        int item = nxt < n_items ? nxt : -1;
        Item I;
        // The scheduler lists only key tiles some query sees, so every item has
        // steps; one without (an inconsistent list) is passed over, never handed on.
        while (item >= 0) {
          I = decode(item);
          if (I.steps > 0 && I.kt >= 0) break;
          bounds_ok(false, status);  // recorded by the debug build
          nxt = atomicAdd(p.header + kHdrNextFused, 1);
          item = nxt < n_items ? nxt : -1;
        }
        if (item < 0) {
          ok = ring_put(B.ring, ii, -1, status);
          break;
        }
        if (!(ok = ring_put(B.ring, ii, item, status, I.steps))) break;
        if (ii > 0 && !(ok = mbar_wait(&B.kv_empty, (ii - 1) & 1, status))) break;
        mbar_arrive_expect_tx(&B.kv_full, 2 * S::kTileBytes);
        for (int c = 0; c < S::kChunks; ++c) {
          tma_load_4d(sK + c * 16384, &tmK, &B.kv_full, c * 64, I.g, I.s.tb, I.s.off_k + I.kt * kBlockN);
          tma_load_4d(sV + c * 16384, &tmV, &B.kv_full, c * 64, I.g, I.s.tb, I.s.off_k + I.kt * kBlockN);
        }
        for (int t = 0; t < I.steps; ++t, ++it) {
          const int qt = I.qt0 + t / G;
          const int h = I.g * G + t % G;
          const int st = it & 1;
          if (it >= 2 && !(ok = mbar_wait(&B.q_empty[st], ((it >> 1) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&B.q_full[st], 2 * S::kTileBytes + 2 * kBM * 4);
          for (int c = 0; c < S::kChunks; ++c) {
            tma_load_4d(sQ + st * S::kTileBytes + c * 16384, &tmQ, &B.q_full[st], c * 64, h, I.s.tb,
                        I.s.off_q + qt * kBM);
            tma_load_4d(sDO + st * S::kTileBytes + c * 16384, &tmDO, &B.q_full[st], c * 64, h, I.s.tb,
                        I.s.off_q + qt * kBM);
          }
          size_t ti = tiled_index(p, I.b, qt * kBM, h);
          if (!bounds_ok(ti + kBM <= static_cast<size_t>(p.pair_cap_q) * p.hq * kBlockM, status)) ti = 0;
          bulk_load(sLse + st * kBM, p.lse_t + ti, kBM * 4, &B.q_full[st]);
          bulk_load(sDelta + st * kBM, p.delta_t + ti, kBM * 4, &B.q_full[st]);
        }
        if (!ok) break;
        // claim the next item only now, close to when this block can start it
        nxt = atomicAdd(p.header + kHdrNextFused, 1);
      }
    }
  } else if (warp == kFusedWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t idS = make_idesc_f16(kBF16, false, false, 128, kBM);
      constexpr uint32_t idAcc = make_idesc_f16(kBF16, false, true, 128, kD);
      constexpr uint32_t idDQ = make_idesc_f16(kBF16, true, true, 128, kD);
      const uint32_t t_dk = tmem + S::kColDK, t_dv = tmem + S::kColDV;
      const uint32_t t_x = tmem + S::kColX, t_y = tmem + S::kColY;
      // K, V, Q, dO K-major for S^T / dP^T; dO and Q MN-major (d contiguous) for
      // dV / dK; dS MN-major (queries contiguous) and K MN-major for dQ.
      const SmemDesc dk = smem_desc(smem_u32(sK), 16, 1024, kLayoutSW128);
      const SmemDesc dv = smem_desc(smem_u32(sV), 16, 1024, kLayoutSW128);
      const SmemDesc dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
      const SmemDesc ddo = smem_desc(smem_u32(sDO), 16, 1024, kLayoutSW128);
      const SmemDesc dq_mn = smem_desc(smem_u32(sQ), 16384, 1024, kLayoutSW128);
      const SmemDesc ddo_mn = smem_desc(smem_u32(sDO), 16384, 1024, kLayoutSW128);
      const SmemDesc dds_mn = smem_desc(smem_u32(sDS), 16384, 1024, kLayoutSW128);
      const SmemDesc dk_mn = smem_desc(smem_u32(sK), 16384, 1024, kLayoutSW128);
      int it = 0, ii = 0;
      bool ok = true;
      auto wait_q = [&](int cur) { return mbar_wait_warp(&B.q_full[cur & 1], (cur >> 1) & 1, status); };
      // S^T = K Q^T or dP^T = V dO^T of step `cur` (B from the step's stage).
      auto issue_st = [&](int cur, uint32_t d_tmem, SmemDesc a, SmemDesc b, uint64_t* done) {
        const SmemDesc bst{b.lo + (((cur & 1) * S::kTileBytes) >> 4), b.hi};
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)
          mma_ss(d_tmem, a, (s >> 2) * 16384 + (s & 3) * 32, bst, (s >> 2) * 16384 + (s & 3) * 32, idS,
                 s > 0 ? 1u : 0u);
        mma_commit(done);
      };
      // dV += P^T dO (a_off 0) or dK += dS^T Q (a_off 16) of step `cur`.
      auto issue_acc = [&](int cur, uint32_t d_tmem, uint32_t a_off, SmemDesc b, uint32_t acc0) {
        const SmemDesc bst{b.lo + (((cur & 1) * S::kTileBytes) >> 4), b.hi};
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s = 0; s < kBM / 16; ++s)
          mma_ts(d_tmem, t_x + a_off + fused_packed_col(s), bst, s * 2048, idAcc, s > 0 ? 1u : acc0);
      };
      // dQ_t = dS K into Y.
      auto issue_dq = [&]() {
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s = 0; s < kBlockN / 16; ++s)
          mma_ss(t_y, dds_mn, s * 2048, dk_mn, s * 2048, idDQ, s > 0 ? 1u : 0u);
        mma_commit(&B.dq_full);
      };
      for (; ok; ++ii) {
        int steps = 0;
        const int item = ring_get_warp_once(B.ring, ii, status, &ok, &steps);
        if (!ok || item < 0) break;
        if (!(ok = mbar_wait_warp(&B.kv_full, ii & 1, status))) break;
        if (!(ok = wait_q(it))) break;
        tc_fence_after();
        issue_st(it, t_x, dk, dq, &B.s_full);
        // Y holds the previous step's dQ until the compute warps have read it
        if (it > 0 && !(ok = mbar_wait_warp(&B.y_free, (it - 1) & 1, status))) break;
        tc_fence_after();
        issue_st(it, t_y, dv, ddo, &B.dp_full);
        for (int t = 0; t < steps; ++t) {
          const int cur = it + t;
          if (!(ok = mbar_wait_warp(&B.p_ready, cur & 1, status))) break;
          if (t == 0 && ii > 0 && !(ok = mbar_wait_warp(&B.acc_empty, (ii - 1) & 1, status))) break;
          tc_fence_after();
          issue_acc(cur, t_dv, 0, ddo_mn, t > 0 ? 1u : 0u);
          if (!(ok = mbar_wait_warp(&B.ds_ready, cur & 1, status))) break;
          tc_fence_after();
          issue_acc(cur, t_dk, 16, dq_mn, t > 0 ? 1u : 0u);
          issue_dq();
          if (t + 1 == steps) {
            mma_commit(&B.kv_empty);  // the item's last readers of K (dQ) and V (dP^T)
            break;
          }
          if (!(ok = wait_q(cur + 1))) break;
          tc_fence_after();
          issue_st(cur + 1, t_x, dk, dq, &B.s_full);
          if (!(ok = mbar_wait_warp(&B.y_free, cur & 1, status))) break;
          tc_fence_after();
          issue_st(cur + 1, t_y, dv, ddo, &B.dp_full);
        }
        if (!ok) break;
        it += steps;
        mma_commit(&B.acc_full);
      }
    }
  } else if (warp >= kFusedWarpDrain) {
    // ------------------------------------------------------------- drain
    // dQ_t out of Y in 16-column chunks into the fp32 staging of the step (Q buffer:
    // columns [0, kD/2), dO buffer: the rest; [128 rows][kD/2] per half, 16-byte
    // unit u of a row at (u ^ row % 8): the accumulator's layout). Y is handed back
    // after the last chunk has been read, before its stores.
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int row_in_tile = quarter * 32 + lane;
    const int sw = row_in_tile & 7;
    int it = 0, ii = 0;
    bool ok = true;
    for (; ok; ++ii) {
      const int item = ring_get_warp(B.ring, ii, status, &ok);
      if (!ok || item < 0) break;
      const Item I = decode(item);
      for (int t = 0; t < I.steps; ++t, ++it) {
        const int st = it & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&B.dq_full, it & 1, status));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD / 16; ++c) {
          uint32_t o[16];
          tmem_ld16(tmem + S::kColY + lane_base + c * 16, o);
          tmem_ld_wait();
          if (c == kD / 16 - 1) {
            tc_fence_before();
            mbar_arrive(&B.y_free);
          }
          const int col = c * 16;  // first column of the chunk
          uint8_t* row = (col < kD / 2 ? sQ : sDO) + st * S::kTileBytes + row_in_tile * S::kHalfRowBytes;
          const int u0 = (col % (kD / 2)) / 4;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_shared_v4(row + (((u0 + v) ^ sw) << 4), o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.stage_full[it & 1]);
      }
    }
  } else if (warp >= kFusedWarpReducer) {
    // ------------------------------------------------------------- reducers
    // Reducer r adds the dQ tiles of the steps with (step & 1) == r.
    const int r = warp - kFusedWarpReducer;
    if (lane == 0) {
      int it = 0, ii = 0;
      bool ok = true;
      constexpr uint32_t kHalfBytes = S::kHalfBytes;
      for (; ok; ++ii) {
        int steps = 0;
        const int item = ring_get(B.ring, ii, status, &ok, &steps);
        if (!ok || item < 0) break;
        const Item I = decode(item);
        for (int t = 0; t < I.steps; ++t, ++it) {
          if ((it & 1) != r) continue;
          const int qt = I.qt0 + t / G;
          const int h = I.g * G + t % G;
          // key tiles 0 .. last see query tile qt; they add in descending order
          const int last = (visible_keys(I.s, qt, causal) + kBlockN - 1) / kBlockN - 1;
          const int rank = last - I.kt;
          const size_t tile = static_cast<size_t>(p.pref_q[I.b] + qt) * p.hq + h;
          const bool in_bounds = bounds_ok(
              rank >= 0 && tile < static_cast<size_t>(p.pair_cap_q) * p.hq, status);
          int* sem = p.dq_sem + (in_bounds ? tile : 0);
          uint8_t* acc = reinterpret_cast<uint8_t*>(p.dq_acc) + (in_bounds ? tile : 0) * (2 * kHalfBytes);
          if (in_bounds && rank > 0 && !(ok = sem_wait_eq(sem, rank, status))) break;
          fence_proxy_async_global();
          if (!(ok = mbar_wait(&B.stage_full[r], (it >> 1) & 1, status))) break;
          const uint8_t* half0 = sQ + (it & 1) * S::kTileBytes;
          const uint8_t* half1 = sDO + (it & 1) * S::kTileBytes;
          if (in_bounds) {
            if (rank == 0) {
              bulk_store(acc, half0, kHalfBytes);
              bulk_store(acc + kHalfBytes, half1, kHalfBytes);
            } else {
              bulk_reduce_add_f32(acc, half0, kHalfBytes);
              bulk_reduce_add_f32(acc + kHalfBytes, half1, kHalfBytes);
            }
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&B.q_empty[it & 1]);  // the stage may take step it + 2
          if (in_bounds) {
            bulk_wait_all();
            fence_proxy_async_global();
            red_release_gpu_add(sem, 1);
          }
        }
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kFusedRegsCompute));
    // ------------------------------------------------------------- compute
    const int quarter = warp & 3, grp = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int col0 = grp * kG;
    const float sl2 = p.scale_log2;
    const int row_in_tile = quarter * 32 + lane;  // key row (S^T, dS^T), query row (dQ)
    const int sw = row_in_tile & 7;               // 128-byte swizzle phase of this row
    int it = 0, ii = 0;
    bool ok = true;
    for (; ok; ++ii) {
      const int item = ring_get_warp(B.ring, ii, status, &ok);
      if (!ok || item < 0) break;
      const Item I = decode(item);
      const int kv_row = I.kt * kBlockN + row_in_tile;
      const bool kv_valid = kv_row < I.s.len_k;
      const int kv_row0 = I.s.off_k * p.rs + I.s.tb;
      for (int t = 0; t < I.steps; ++t, ++it) {
        const int qt = I.qt0 + t / G;
        const int st = it & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&B.q_full[st], (it >> 1) & 1, status));
        if (!ok) break;
        // query columns i of this warp with a nonzero P^T for this key row: [lo, hi)
        const int q_base = qt * kBM + col0;
        const int hi = kv_valid ? min(kG, I.s.len_q - q_base) : 0;
        const int lo = causal ? max(0, kv_row - I.s.diag - q_base) : 0;
        const bool full = __all_sync(0xffffffffu, lo == 0 && hi >= kG);
        const float4* lse4 = reinterpret_cast<const float4*>(sLse + st * kBM + col0);
        const float4* dlt4 = reinterpret_cast<const float4*>(sDelta + st * kBM + col0);
        // ---- A: P^T = exp2(S^T * scale * log2e - lse2) into X[32c, 32c+16)
        ok = __all_sync(0xffffffffu, mbar_wait(&B.s_full, it & 1, status));
        if (!ok) break;
        tc_fence_after();
        float pv[kG];
        {
          uint32_t sv[kG];
          tmem_ld32(tmem + S::kColX + lane_base + col0, sv);
          tmem_ld_wait();
          if (full) {
            // paired fma (-lse * log2e arrives negated): same rounding as fmaf
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
            for (int k = 0; k < kG / 4; ++k) {
              const float4 l4 = lse4[k];
              const float2 x01 = f2_unpack(ffma2(f2_pack(__uint_as_float(sv[4 * k]), __uint_as_float(sv[4 * k + 1])),
                                                 sl2x2, f2_pack(l4.x, l4.y)));
              const float2 x23 = f2_unpack(ffma2(f2_pack(__uint_as_float(sv[4 * k + 2]), __uint_as_float(sv[4 * k + 3])),
                                                 sl2x2, f2_pack(l4.z, l4.w)));
              pv[4 * k] = ex2_fused(x01.x);
              pv[4 * k + 1] = ex2_fused(x01.y);
              pv[4 * k + 2] = ex2_fused(x23.x);
              pv[4 * k + 3] = ex2_fused(x23.y);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kG / 4; ++k) {
              const float4 l4 = lse4[k];
              const float l[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 4 * k + e;
                const float x = ex2_fused(fmaf(__uint_as_float(sv[i]), sl2, l[e]));
                pv[i] = (i >= lo && i < hi) ? x : 0.f;
              }
            }
          }
          uint32_t pk[kG / 2];
#pragma unroll
          for (int k = 0; k < kG / 2; ++k) pk[k] = pack2<kBF16>(pv[2 * k], pv[2 * k + 1]);
          tmem_st16(tmem + S::kColX + lane_base + col0, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&B.p_ready);
        // ---- B: dS^T = P^T (dP^T - D) into X[32c+16, 32c+32) and the dS tile
        ok = __all_sync(0xffffffffu, mbar_wait(&B.dp_full, it & 1, status));
        if (!ok) break;
        tc_fence_after();
        uint32_t dd[kG / 2];
        {
          uint32_t dv[kG];
          tmem_ld32(tmem + S::kColY + lane_base + col0, dv);
          tmem_ld_wait();
          // Masked entries are selected to 0 (not multiplied): D of rows past the
          // query length is never written and may hold any bits.
          float rr[kG];
          // paired add (-D arrives negated) and multiply: the same two roundings
#pragma unroll
          for (int k = 0; k < kG / 4; ++k) {
            const float4 d4 = dlt4[k];
            const float2 r01 = f2_unpack(fmul2(f2_pack(pv[4 * k], pv[4 * k + 1]),
                                               fadd2(f2_pack(__uint_as_float(dv[4 * k]), __uint_as_float(dv[4 * k + 1])),
                                                     f2_pack(d4.x, d4.y))));
            const float2 r23 = f2_unpack(fmul2(f2_pack(pv[4 * k + 2], pv[4 * k + 3]),
                                               fadd2(f2_pack(__uint_as_float(dv[4 * k + 2]), __uint_as_float(dv[4 * k + 3])),
                                                     f2_pack(d4.z, d4.w))));
            rr[4 * k] = r01.x;
            rr[4 * k + 1] = r01.y;
            rr[4 * k + 2] = r23.x;
            rr[4 * k + 3] = r23.y;
          }
          if (!full) {
#pragma unroll
            for (int i = 0; i < kG; ++i) rr[i] = (i >= lo && i < hi) ? rr[i] : 0.f;
          }
#pragma unroll
          for (int k = 0; k < kG / 2; ++k) dd[k] = pack2<kBF16>(rr[2 * k], rr[2 * k + 1]);
        }
        tmem_st16(tmem + S::kColX + lane_base + col0 + 16, dd);
        {
          // dS tile (its last reader, dQ_t-1, finished before dP^T_t, which this
          // phase waited for): row = key,
          // 16-byte unit u of queries [8u, 8u+8) in 64-query chunks, 128-byte
          // swizzled (unit ^ row % 8) -- dQ's A operand, MN-major (queries contiguous).
          uint8_t* row = sDS + (grp >> 1) * 16384 + row_in_tile * 128;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int u = 4 * (grp & 1) + v;
            st_shared_v4(row + ((u ^ sw) << 4), dd[4 * v], dd[4 * v + 1], dd[4 * v + 2], dd[4 * v + 3]);
          }
        }
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&B.ds_ready);
      }
      if (!ok) break;
      // Epilogue: scale * dK and dV for key rows some real query sees.
      ok = __all_sync(0xffffffffu, mbar_wait(&B.acc_full, ii & 1, status));
      if (!ok) break;
      tc_fence_after();
      const size_t kv_tok = static_cast<size_t>(kv_row0) + static_cast<size_t>(kv_row) * p.rs;
      const bool store = kv_row < seen_keys(I.s, causal) &&
                         bounds_ok(kv_tok < static_cast<size_t>(p.total_kv), status);
      const size_t kv_off = (kv_tok * p.hkv + I.g) * p.d;
      const auto dk_rows = make_row_pair(static_cast<fused_elem_t<kBF16>*>(p.dk) + kv_off, store);
      const auto dv_rows = make_row_pair(static_cast<fused_elem_t<kBF16>*>(p.dv) + kv_off, store);
#pragma unroll
      for (int c = 0; c < S::kOutCols; c += 16) {
        const int c0 = grp * S::kOutCols + c;
        uint32_t a[16], b[16];
        tmem_ld16(tmem + S::kColDK + lane_base + c0, a);
        tmem_ld16(tmem + S::kColDV + lane_base + c0, b);
        tmem_ld_wait();
        store_pair16<kBF16>(dk_rows, c0, p.d, a, p.scale);
        store_pair16<kBF16>(dv_rows, c0, p.d, b, 1.0f);
      }
      tc_fence_before();
      mbar_arrive(&B.acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kFusedWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// dQ conversion: the fp32 accumulator (scaled by attn_scale) to 16-bit dq, for
// every real query row that sees a key; one warp per row, all heads, 16-byte
// reads of the swizzled tiles and 8-byte stores.
// ===========================================================================
template <bool kBF16>
__global__ void __launch_bounds__(256) dq_convert_kernel(AttnParams p) {
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const bool causal = p.causal != 0;
  // tile: two halves of 128 rows x dq_cols/2 fp32 columns (dq_cols = 64 or 128)
  const int half_units = p.dq_cols / 8;  // 16-byte units per row of a half
  const size_t half_bytes = static_cast<size_t>(kBlockM) * half_units * 16;
  const size_t tile_bytes = 2 * half_bytes;
  const int units = p.d / 4;  // 16-byte units of 4 fp32 per row and head
  using T = fused_elem_t<kBF16>;
  for (int r = gw; r < p.total_q; r += warps) {
    int i = 0;
    const int b = locate_row(p, p.cu_q_pad, r, &i);
    if (b < 0) continue;
    const SeqInfo s = load_seq(p, b);
    if (i >= s.len_q || row_keys(s, i, causal) == 0) continue;
    const size_t pair = static_cast<size_t>(p.pref_q[b] + i / kBlockM);
    const int ii = i % kBlockM;
    if (!bounds_ok(pair < static_cast<size_t>(p.pair_cap_q), p.header + kHdrStatus)) continue;
    for (int e = lane; e < p.hq * units; e += 32) {
      const int h = e / units, u = e % units;  // columns [4u, 4u+4) of head h
      const int half = u / half_units, uu = u % half_units;
      const uint8_t* tile = reinterpret_cast<const uint8_t*>(p.dq_acc) + (pair * p.hq + h) * tile_bytes;
      const float4 v = *reinterpret_cast<const float4*>(tile + half * half_bytes +
                                                        static_cast<size_t>(ii) * half_units * 16 +
                                                        ((uu ^ (ii & 7)) << 4));
      uint2 w;
      w.x = pack2<kBF16>(v.x * p.scale, v.y * p.scale);
      w.y = pack2<kBF16>(v.z * p.scale, v.w * p.scale);
      *reinterpret_cast<uint2*>(static_cast<T*>(p.dq) + (static_cast<size_t>(r) * p.hq + h) * p.d + 4 * u) = w;
    }
  }
}

// ===========================================================================
// Launchers
// ===========================================================================
template <int kD, bool kBF16>
static cudaError_t launch_fused_impl(const AttnParams& p, int num_sms, cudaStream_t st) {
  using S = FusedShape<kD>;
  CUtensorMap tq, tdo, tk, tv;
  const int nb = p.sbhd ? p.batch : 1;
  if (!make_tmap_tokens(&tq, p.q, p.total_q, nb, p.hq, p.d, kBF16, 128) ||
      !make_tmap_tokens(&tdo, p.dout, p.total_q, nb, p.hq, p.d, kBF16, 128) ||
      !make_tmap_tokens(&tk, p.k, p.total_kv, nb, p.hkv, p.d, kBF16, 128) ||
      !make_tmap_tokens(&tv, p.v, p.total_kv, nb, p.hkv, p.d, kBF16, 128))
    return cudaErrorInvalidValue;
  auto kern = attn_bwd_fused_kernel<kD, kBF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long max_items = static_cast<long long>(p.pair_cap_k) * p.hkv;
  const int grid = static_cast<int>(max_items < num_sms ? (max_items > 0 ? max_items : 1) : num_sms);
  kern<<<grid, kFusedThreads, S::kSmemBytes, st>>>(p, tq, tdo, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_fused(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st) {
  if (bf16) return p.d <= 64 ? launch_fused_impl<64, true>(p, num_sms, st)
                             : launch_fused_impl<128, true>(p, num_sms, st);
  return p.d <= 64 ? launch_fused_impl<64, false>(p, num_sms, st)
                   : launch_fused_impl<128, false>(p, num_sms, st);
}

cudaError_t launch_dq_convert(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st) {
  if (bf16)
    dq_convert_kernel<true><<<num_sms * 8, 256, 0, st>>>(p);
  else
    dq_convert_kernel<false><<<num_sms * 8, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace teattn

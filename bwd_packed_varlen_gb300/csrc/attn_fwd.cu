// Forward attention over packed variable-length sequences on sm_103a, one query
// tile per work item (used for head_dim 256; head_dim <= 128 runs the two-tile
// kernel in attn_fwd_pair.cu).
//
// One work item = (sequence b, query head h, 128-row query tile). A persistent
// grid walks the scheduler's sorted item list with a static stride. Inside a
// thread block three roles run concurrently and hand tiles over through
// mbarriers:
//   warp 4  (TMA)     loads the Q tile once per item and K/V tiles of 128 key
//                     rows into multi-stage shared-memory rings (128-byte swizzle,
//                     rows at the PADDED offsets, rows past the tensor read as 0);
//   warp 5  (MMA)     one elected lane issues tcgen05 MMAs: S_j = Q K_j^T into one of two
//                     TMEM score buffers, then O += P_j V_j with P_j read from TMEM;
//   warps 0-3 (softmax) one thread per query row: masks by the REAL lengths
//                     (key j visible iff j < Lk, and j <= i when causal), runs the
//                     online softmax in fp32 in the log2 domain, writes P_j as
//                     16-bit values over S_j in TMEM, rescales O only when the
//                     running max grows by more than 2^8, and finally writes
//                     O / l and lse = m ln2 + ln l for its row.
// Issue order of the MMA thread is S_0, S_1, PV_0, S_2, PV_1, ... so the tensor
// cores compute the next scores while the softmax warps work on the current
// ones.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "launch.h"
#include "sm103_ptx.cuh"
#include "tmap.h"

namespace teattn {

template <int kD>
struct FwdShape {
  static constexpr int kChunks = kD / 64;            // 64-column swizzle atoms
  static constexpr int kTileBytes = kChunks * 16384; // 128 rows x kD cols x 2 B
  static constexpr int kStagesK = (kD <= 128) ? 2 : 1;
  static constexpr int kStagesV = (kD <= 128) ? 2 : 1;
  static constexpr int kSmemUsed = kTileBytes * (1 + kStagesK + kStagesV) + 1024;
  // Request at least 120 KB so that one block owns an SM (and all of TMEM).
  static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = kD;  // S buffers follow O (kD columns)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int kD, bool kBF16>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using S = FwdShape<kD>;
  constexpr int SK = S::kStagesK, SV = S::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + S::kTileBytes;
  uint8_t* sV = sK + SK * S::kTileBytes;

  __shared__ uint64_t bar_q_full, bar_q_empty, bar_o_empty;
  __shared__ uint64_t bar_k_full[SK], bar_k_empty[SK], bar_v_full[SV], bar_v_empty[SV];
  __shared__ uint64_t bar_s_full[2], bar_p_ready[2], bar_o_ready[2];
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* status = p.header + kHdrStatus;
  const int n_pairs = p.header[kHdrNumQPairs];
  const int n_items = n_pairs * p.hq;
  const bool causal = p.causal != 0;

  if (tid == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 1);
    mbar_init(&bar_o_empty, 128);
    for (int i = 0; i < SK; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_empty[i], 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_ready[i], 128);
      mbar_init(&bar_o_ready[i], 1);
    }
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&tmem_slot, S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_o = tmem;

  if (warp == 4) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int it = 0, ii = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const PairHead ph = item_pair_head(item, n_pairs, p.group);
        const int2 pr = p.q_pairs[ph.pair];
        const int h = ph.head, g = h / p.group;
        const SeqInfo s = load_seq(p, pr.x);
        const int qt = pr.y;
        const int n = (visible_keys(s, qt, causal) + kBlockN - 1) / kBlockN;
        // a tile that sees no key (before a lower-right causal triangle) is the
        // zero fill's; every role skips it without touching a barrier
        if (n == 0) continue;
        const int k = ii++;  // index of this item among the block's processed ones
        if (k > 0 && !(ok = mbar_wait(&bar_q_empty, (k - 1) & 1, status))) break;
        mbar_arrive_expect_tx(&bar_q_full, S::kTileBytes);
        for (int c = 0; c < S::kChunks; ++c)
          tma_load_4d(sQ + c * 16384, &tmQ, &bar_q_full, c * 64, h, s.tb, s.off_q + qt * kBlockM);
        for (int j = 0; j < n; ++j, ++it) {
          const int sk = it % SK;
          if (it >= SK && !(ok = mbar_wait(&bar_k_empty[sk], ((it / SK) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&bar_k_full[sk], S::kTileBytes);
          for (int c = 0; c < S::kChunks; ++c)
            tma_load_4d(sK + sk * S::kTileBytes + c * 16384, &tmK, &bar_k_full[sk], c * 64, g, s.tb,
                        s.off_k + j * kBlockN);
          const int sv = it % SV;
          if (it >= SV && !(ok = mbar_wait(&bar_v_empty[sv], ((it / SV) - 1) & 1, status))) break;
          mbar_arrive_expect_tx(&bar_v_full[sv], S::kTileBytes);
          for (int c = 0; c < S::kChunks; ++c)
            tma_load_4d(sV + sv * S::kTileBytes + c * 16384, &tmV, &bar_v_full[sv], c * 64, g, s.tb,
                        s.off_k + j * kBlockN);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t idS = make_idesc_f16(kBF16, false, false, 128, kBlockN);
      constexpr uint32_t idPV = make_idesc_f16(kBF16, false, true, 128, kD);
      // Operand descriptors: Q and K K-major; V as the N-major (d-contiguous) B of P V.
      const SmemDesc dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
      const SmemDesc dk = smem_desc(smem_u32(sK), 16, 1024, kLayoutSW128);
      const SmemDesc dv = smem_desc(smem_u32(sV), 16384, 1024, kLayoutSW128);
      int it = 0, ii = 0;
      bool ok = true;
      auto issue_s = [&](int t) -> bool {
        const int sk = t % SK;
        if (!mbar_wait_warp(&bar_k_full[sk], (t / SK) & 1, status)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem + S::kColS0 + (t & 1) * kBlockN;
        const SmemDesc kst{dk.lo + ((sk * S::kTileBytes) >> 4), dk.hi};
        __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
        for (int s = 0; s < kD / 16; ++s) {
          const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
          mma_ss(d_tmem, dq, off, kst, off, idS, s > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s_full[t & 1]);
        mma_commit(&bar_k_empty[sk]);
        return true;
      };
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int2 pr = p.q_pairs[item_pair_head(item, n_pairs, p.group).pair];
        const SeqInfo s = load_seq(p, pr.x);
        const int n = (visible_keys(s, pr.y, causal) + kBlockN - 1) / kBlockN;
        if (n == 0) continue;
        const int k = ii++;  // index of this item among the block's processed ones
        if (!(ok = mbar_wait_warp(&bar_q_full, k & 1, status))) break;
        if (!(ok = issue_s(it))) break;
        for (int j = 0; j < n && ok; ++j) {
          const int cur = it + j;
          if (j + 1 < n) {
            if (!(ok = issue_s(cur + 1))) break;
          } else {
            mma_commit(&bar_q_empty);
          }
          if (!(ok = mbar_wait_warp(&bar_p_ready[cur & 1], (cur >> 1) & 1, status))) break;
          const int sv = cur % SV;
          if (!(ok = mbar_wait_warp(&bar_v_full[sv], (cur / SV) & 1, status))) break;
          if (j == 0 && k > 0 && !(ok = mbar_wait_warp(&bar_o_empty, (k - 1) & 1, status))) break;
          tc_fence_after();
          const uint32_t a_tmem = tmem + S::kColS0 + (cur & 1) * kBlockN;
          const SmemDesc vst{dv.lo + ((sv * S::kTileBytes) >> 4), dv.hi};
          const uint32_t acc0 = j > 0 ? 1u : 0u;
          __syncwarp();  // elect.sync in the MMA wrappers needs a converged warp
#pragma unroll
          for (int s = 0; s < kBlockN / 16; ++s)
            mma_ts(t_o, a_tmem + s * 8, vst, s * 2048, idPV, s > 0 ? 1u : acc0);
          mma_commit(&bar_v_empty[sv]);
          mma_commit(&bar_o_ready[cur & 1]);
        }
        it += n;
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const PairHead ph = item_pair_head(item, n_pairs, p.group);
      const int2 pr = p.q_pairs[ph.pair];
      const int h = ph.head;
      const SeqInfo s = load_seq(p, pr.x);
      const int qt = pr.y;
      const int n = (visible_keys(s, qt, causal) + kBlockN - 1) / kBlockN;
      if (n == 0) continue;
      const int row = qt * kBlockM + tid;
      // rows that see no key (before a lower-right triangle) are the zero fill's
      const int lim = row < s.len_q ? row_keys(s, row, causal) : 0;
      const bool row_valid = lim > 0 && bounds_ok(q_row(p, s, row) < static_cast<size_t>(p.total_q),
                                                  p.header + kHdrStatus);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        const int cur = it + j;
        const uint32_t t_s = tmem + S::kColS0 + (cur & 1) * kBlockN;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s_full[cur & 1], (cur >> 1) & 1, status));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld32(t_s + lane_base + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(t_s + lane_base + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(t_s + lane_base + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        tmem_ld32(t_s + lane_base + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        tmem_ld_wait();
        const int nvalid = min(max(lim - j * kBlockN, 0), kBlockN);
        // Warp-uniform: only tiles on the causal diagonal or a length boundary pay
        // for per-element masking. Max and sum use 8 independent partials so the
        // dependent chains stay short.
        const bool full = __all_sync(0xffffffffu, nvalid >= kBlockN);
        float mp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = -INFINITY;
        if (full) {
#pragma unroll
          for (int c = 0; c < kBlockN; ++c) mp[c & 7] = fmaxf(mp[c & 7], __uint_as_float(sr[c]));
        } else {
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            mp[c & 7] = fmaxf(mp[c & 7], c < nvalid ? __uint_as_float(sr[c]) : -INFINITY);
        }
        const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        const float mxs = mx * sl2;
        float m_new = m;
        bool rescale = false;
        if (nvalid > 0) {
          if (m == -INFINITY) {
            m_new = mxs;
          } else if (mxs > m + 8.0f) {
            m_new = mxs;
            rescale = true;
          }
        }
        float sp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sp[k] = 0.f;
        uint32_t pk[64];
        if (full) {
#pragma unroll
          for (int c = 0; c < kBlockN / 2; ++c) {
            const float p0 = ex2(fmaf(__uint_as_float(sr[2 * c]), sl2, -m_new));
            const float p1 = ex2(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -m_new));
            sp[c & 7] += p0 + p1;
            pk[c] = pack2<kBF16>(p0, p1);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kBlockN / 2; ++c) {
            const float x0 = ex2(fmaf(__uint_as_float(sr[2 * c]), sl2, -m_new));
            const float x1 = ex2(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -m_new));
            const float p0 = 2 * c < nvalid ? x0 : 0.f;
            const float p1 = 2 * c + 1 < nvalid ? x1 : 0.f;
            sp[c & 7] += p0 + p1;
            pk[c] = pack2<kBF16>(p0, p1);
          }
        }
        const float rs = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        if (__any_sync(0xffffffffu, rescale)) {
          const int prev = cur - 1;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bar_o_ready[prev & 1], (prev >> 1) & 1, status));
          if (!ok) break;
          tc_fence_after();
          const float alpha = rescale ? ex2(m - m_new) : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < kD; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + lane_base + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st16(t_o + lane_base + c0, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
            tmem_st16(t_o + lane_base + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&o[16]));
          }
          l *= alpha;
        }
        tmem_st16(t_s + lane_base + 0, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        tmem_st16(t_s + lane_base + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
        tmem_st16(t_s + lane_base + 32, *reinterpret_cast<uint32_t(*)[16]>(&pk[32]));
        tmem_st16(t_s + lane_base + 48, *reinterpret_cast<uint32_t(*)[16]>(&pk[48]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_p_ready[cur & 1]);
        l += rs;
        m = m_new;
      }
      if (!ok) break;
      // Epilogue: O / l and lse for this row once the last PV has landed.
      const int last = it + n - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_o_ready[last & 1], (last >> 1) & 1, status));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
      T* orow = static_cast<T*>(p.out) +
                (q_row(p, s, row) * p.hq + h) * static_cast<size_t>(p.d);
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(t_o + lane_base + c0, o);
        tmem_ld_wait();
        if (row_valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int col = c0 + v * 8;
            if (col + 8 <= p.d) {
              uint4 w;
              w.x = pack2<kBF16>(__uint_as_float(o[v * 8 + 0]) * inv, __uint_as_float(o[v * 8 + 1]) * inv);
              w.y = pack2<kBF16>(__uint_as_float(o[v * 8 + 2]) * inv, __uint_as_float(o[v * 8 + 3]) * inv);
              w.z = pack2<kBF16>(__uint_as_float(o[v * 8 + 4]) * inv, __uint_as_float(o[v * 8 + 5]) * inv);
              w.w = pack2<kBF16>(__uint_as_float(o[v * 8 + 6]) * inv, __uint_as_float(o[v * 8 + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + col) = w;
            }
          }
        }
      }
      if (row_valid)
        p.lse[q_row(p, s, row) * p.hq + h] = m * 0.69314718055994531f + logf(l);
      tc_fence_before();
      mbar_arrive(&bar_o_empty);
      it += n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, S::kTmemCols);
  }
}

template <int kD, bool kBF16>
static cudaError_t launch_fwd_impl(const AttnParams& p, int num_sms, cudaStream_t st) {
  using S = FwdShape<kD>;
  CUtensorMap tq, tk, tv;
  const bool bf16 = kBF16;
  const int nb = p.sbhd ? p.batch : 1;
  if (!make_tmap_tokens(&tq, p.q, p.total_q, nb, p.hq, p.d, bf16) ||
      !make_tmap_tokens(&tk, p.k, p.total_kv, nb, p.hkv, p.d, bf16) ||
      !make_tmap_tokens(&tv, p.v, p.total_kv, nb, p.hkv, p.d, bf16))
    return cudaErrorInvalidValue;
  auto kern = attn_fwd_kernel<kD, kBF16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long max_items = static_cast<long long>(p.pair_cap_q) * p.hq;
  const int grid = static_cast<int>(max_items < num_sms ? (max_items > 0 ? max_items : 1) : num_sms);
  kern<<<grid, 192, S::kSmemBytes, st>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st) {
  const int d = p.d;
  if (bf16) {
    if (d <= 64) return launch_fwd_impl<64, true>(p, num_sms, st);
    if (d <= 128) return launch_fwd_impl<128, true>(p, num_sms, st);
    return launch_fwd_impl<256, true>(p, num_sms, st);
  }
  if (d <= 64) return launch_fwd_impl<64, false>(p, num_sms, st);
  if (d <= 128) return launch_fwd_impl<128, false>(p, num_sms, st);
  return launch_fwd_impl<256, false>(p, num_sms, st);
}

}  // namespace teattn

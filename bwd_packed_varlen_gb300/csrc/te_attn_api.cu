// C ABI of libteattn.so (declared in include/te_attn.h): argument checks,
// workspace layout and the launch sequence of each call.
//
//   forward : schedule -> attention forward -> zero fill of rows no tile writes
//   backward: schedule -> zero fill -> D = rowsum(dO * O) -> dQ -> dK/dV
//   fused backward (te_attn_bwd_thd_fused, head_dim <= 128): schedule -> zero fill
//             -> D -> dK/dV with an ordered dQ accumulation -> dQ conversion
//
// All launches go to the caller's stream; nothing is allocated and nothing is
// kept between calls except per-device constants (SM count).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/te_attn.h"
#include "common.cuh"
#include "launch.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int ok_status() {
  g_last_error.clear();
  return TE_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t header, pref_q, pref_k, pref_f, q_pairs, k_pairs, f_pairs, lse_t, delta_t, dq_acc, dq_sem,
      k_items, total;
  int cap_q, cap_k, cap_f;
};

// Workspace layout (256-byte aligned sections):
//   header  int32[64]        status word and pair counts of this call
//   pref_q  int32[batch+1]   prefix sums of query tiles per sequence
//   pref_k  int32[batch+1]   prefix sums of key tiles per sequence
//   pref_f  int32[batch+1]   prefix sums of 256-row query tile pairs per sequence
//   q_pairs int2[cap_q]      sorted (sequence, query tile)
//   k_pairs int2[cap_k]      sorted (sequence, key tile)
//   f_pairs int2[cap_f]      sorted (sequence, 256-row query tile pair)
//   lse_t   fp32[cap_q*hq*128] backward only: -lse * log2(e), tile-major
//   delta_t fp32[cap_q*hq*128] backward only: -rowsum(dO * O), tile-major (both
//           negated so that the consumers add them without a negation)
//   dq_acc  fp32[cap_q*hq*128*dq_cols] fused backward only: the ordered dQ
//           accumulator, one 128-row tile per (query tile pair, head)
//   dq_sem  int32[cap_q*hq]  fused backward only: key tiles added to each dQ tile
//   k_items int4[cap_k*hkv]  fused backward only: work items, chain-major
// dq_cols: 0 (no fused backward), 64 (head_dim <= 64) or 128 (head_dim <= 128).
bool make_layout(int batch, int total_q, int total_kv, int hq, bool backward, Layout* L,
                 int dq_cols = 0, int hkv = 0) {
  if (batch < 1 || total_q < 0 || total_kv < 0 || hq < 1) return false;
  // sum_b ceil(L_b / 128) <= total / 128 + batch when sum_b L_b <= total
  const long long cq = static_cast<long long>(total_q) / teattn::kBlockM + batch + 1;
  const long long ck = static_cast<long long>(total_kv) / teattn::kBlockN + batch + 1;
  const long long cf = static_cast<long long>(total_q) / teattn::kBlockF + batch + 1;
  if (cq > INT32_MAX / 64 || ck > INT32_MAX / 64) return false;
  L->cap_q = static_cast<int>(cq);
  L->cap_k = static_cast<int>(ck);
  L->cap_f = static_cast<int>(cf);
  size_t off = 0;
  L->header = off;
  off = align_up(off + teattn::kHdrWords * sizeof(int), 256);
  L->pref_q = off;
  off = align_up(off + (static_cast<size_t>(batch) + 1) * sizeof(int), 256);
  L->pref_k = off;
  off = align_up(off + (static_cast<size_t>(batch) + 1) * sizeof(int), 256);
  L->pref_f = off;
  off = align_up(off + (static_cast<size_t>(batch) + 1) * sizeof(int), 256);
  L->q_pairs = off;
  off = align_up(off + static_cast<size_t>(cq) * sizeof(int2), 256);
  L->k_pairs = off;
  off = align_up(off + static_cast<size_t>(ck) * sizeof(int2), 256);
  L->f_pairs = off;
  off = align_up(off + static_cast<size_t>(cf) * sizeof(int2), 256);
  const size_t tiled = static_cast<size_t>(cq) * hq * teattn::kBlockM * sizeof(float);
  L->lse_t = off;
  if (backward) off = align_up(off + tiled, 256);
  L->delta_t = off;
  if (backward) off = align_up(off + tiled, 256);
  L->dq_acc = off;
  off += static_cast<size_t>(cq) * hq * teattn::kBlockM * dq_cols * sizeof(float);
  L->dq_sem = off;
  if (dq_cols > 0) off = align_up(off + static_cast<size_t>(cq) * hq * sizeof(int), 256);
  L->k_items = off;
  if (dq_cols > 0) off = align_up(off + static_cast<size_t>(ck) * hkv * 4 * sizeof(int), 256);
  L->total = off;
  return true;
}

// Columns of a dQ accumulator tile in the fused backward (0: no fused path).
int fused_cols(int d) { return d <= 64 ? 64 : (d <= 128 ? 128 : 0); }

int num_sms_of_current_device() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared argument checks of both entry points. Returns TE_OK or an error code.
int check_common(int batch, int total_q, int total_kv, int hq, int hkv, int d, float attn_scale,
                 int mask_type, int dtype, const int32_t* cu_q, const int32_t* cu_kv,
                 const int32_t* cu_q_pad, const int32_t* cu_kv_pad) {
  if (!cu_q || !cu_kv || !cu_q_pad || !cu_kv_pad)
    return fail(TE_ERR_INVALID_ARG, "cu_seqlens pointers must not be NULL");
  if (batch < 1) return fail(TE_ERR_INVALID_ARG, "batch must be >= 1");
  if (total_q < 0 || total_kv < 0) return fail(TE_ERR_INVALID_ARG, "total_q/total_kv must be >= 0");
  if (hq < 1 || hkv < 1) return fail(TE_ERR_INVALID_ARG, "hq and hkv must be >= 1");
  if (hq % hkv != 0) return fail(TE_ERR_INVALID_ARG, "hq must be a multiple of hkv");
  if (d < 8 || d > 256 || d % 8 != 0)
    return fail(TE_ERR_UNSUPPORTED, "head dim must be a multiple of 8 in [8, 256]");
  if (mask_type != TE_MASK_PADDING && mask_type != TE_MASK_PADDING_CAUSAL &&
      mask_type != TE_MASK_PADDING_CAUSAL_BOTTOM_RIGHT)
    return fail(TE_ERR_UNSUPPORTED,
                "mask_type must be TE_MASK_PADDING, TE_MASK_PADDING_CAUSAL or "
                "TE_MASK_PADDING_CAUSAL_BOTTOM_RIGHT");
  if (dtype != TE_DTYPE_FP16 && dtype != TE_DTYPE_BF16)
    return fail(TE_ERR_UNSUPPORTED, "dtype must be TE_DTYPE_FP16 or TE_DTYPE_BF16");
  if (!std::isfinite(attn_scale)) return fail(TE_ERR_INVALID_ARG, "attn_scale must be finite");
  if (static_cast<long long>(total_q) * hq * d >= (1ll << 40) ||
      static_cast<long long>(total_kv) * hkv * d >= (1ll << 40))
    return fail(TE_ERR_UNSUPPORTED, "tensor too large");
  return TE_OK;
}

teattn::AttnParams base_params(const int32_t* cu_q, const int32_t* cu_kv, const int32_t* cu_q_pad,
                               const int32_t* cu_kv_pad, int batch, int total_q, int total_kv, int hq,
                               int hkv, int d, float attn_scale, int mask_type, void* workspace,
                               const Layout& L) {
  teattn::AttnParams p{};
  p.cu_q = cu_q;
  p.cu_kv = cu_kv;
  p.cu_q_pad = cu_q_pad;
  p.cu_kv_pad = cu_kv_pad;
  p.batch = batch;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.hq = hq;
  p.hkv = hkv;
  p.d = d;
  p.group = hq / hkv;
  p.sbhd = 0;
  p.rs = 1;
  p.causal = mask_type == TE_MASK_PADDING_CAUSAL ? 1
             : mask_type == TE_MASK_PADDING_CAUSAL_BOTTOM_RIGHT ? 2 : 0;
  p.scale = attn_scale;
  p.scale_log2 = attn_scale * 1.4426950408889634f;
  char* ws = static_cast<char*>(workspace);
  p.header = reinterpret_cast<int*>(ws + L.header);
  p.q_pairs = reinterpret_cast<int2*>(ws + L.q_pairs);
  p.k_pairs = reinterpret_cast<int2*>(ws + L.k_pairs);
  p.f_pairs = reinterpret_cast<int2*>(ws + L.f_pairs);
  p.pair_cap_q = L.cap_q;
  p.pair_cap_k = L.cap_k;
  p.pair_cap_f = L.cap_f;
  return p;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(TE_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

// Optional per-launch event timing (te_attn_profile_enable / _read).
struct ProfRecord {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof;

const char* const kKernelNames[TE_NUM_KERNELS] = {"teattn schedule", "teattn forward",
                                                   "teattn zero fill", "teattn delta",
                                                   "teattn dK/dV", "teattn dQ",
                                                   "teattn widen e4m3", "teattn fused backward",
                                                   "teattn dQ conversion"};

// Runs `launch` between two events on `st` when profiling is enabled, inside an
// NVTX range named after the kernel (visible to Nsight tools; a no-op without one).
template <typename F>
cudaError_t timed(int kernel, cudaStream_t st, F&& launch) {
  if (!g_prof_on) return launch();
  struct Range {
    explicit Range(const char* n) { nvtxRangePushA(n); }
    ~Range() { nvtxRangePop(); }
  } range(kKernelNames[kernel]);
  ProfRecord r{kernel, nullptr, nullptr};
  cudaError_t e = cudaEventCreate(&r.start);
  if (e == cudaSuccess) e = cudaEventCreate(&r.stop);
  if (e == cudaSuccess) e = cudaEventRecord(r.start, st);
  if (e != cudaSuccess) return e;
  e = launch();
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(r.stop, st);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.push_back(r);
  return cudaSuccess;
}

}  // namespace

namespace teattn {
// Lets other entry points of the library report through te_attn_last_error().
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace teattn

extern "C" {

int te_attn_version(void) { return 10100; }

size_t te_attn_fwd_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv, int d) {
  (void)hkv;
  (void)d;
  Layout L;
  return make_layout(batch, total_q, total_kv, hq, false, &L) ? L.total : 0;
}

size_t te_attn_bwd_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv, int d) {
  (void)hkv;
  (void)d;
  Layout L;
  return make_layout(batch, total_q, total_kv, hq, true, &L) ? L.total : 0;
}

size_t te_attn_bwd_fused_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv,
                                        int d) {
  Layout L;
  const int cols = fused_cols(d);
  return cols > 0 && make_layout(batch, total_q, total_kv, hq, true, &L, cols, hkv) ? L.total : 0;
}

// Per-tensor dequantisation factors of an e4m3 forward (real value = stored
// value * descale); `on` false for 16-bit inputs.
struct E4m3Scales {
  bool on;
  float q, k, v;
};

// Bytes of the widened (bf16) V copy an e4m3 forward keeps after the layout.
size_t widened_v_bytes(int total_kv, int hkv, int d) {
  return align_up(static_cast<size_t>(total_kv > 0 ? total_kv : 0) * hkv * d * 2, 256);
}

// Forward of either layout: sbhd = false packs sequences by cu_seqlens_*_padded,
// sbhd = true puts token i of sequence b at row i * batch + b.
static int fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                    const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int batch,
                    int total_q, int total_kv, int hq, int hkv, int d, float attn_scale, int mask_type,
                    int dtype, void* workspace, size_t workspace_bytes, void* stream, bool sbhd,
                    E4m3Scales e4m3 = E4m3Scales{false, 1.f, 1.f, 1.f}) {
  int rc = check_common(batch, total_q, total_kv, hq, hkv, d, attn_scale, mask_type, dtype,
                        cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded);
  if (rc != TE_OK) return rc;
  if (!workspace) return fail(TE_ERR_INVALID_ARG, "workspace must not be NULL");
  if (total_q > 0 && (!q || !out || !lse))
    return fail(TE_ERR_INVALID_ARG, "q, out and lse must not be NULL");
  if (total_kv > 0 && (!k || !v)) return fail(TE_ERR_INVALID_ARG, "k and v must not be NULL");
  if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) || (out && !aligned16(out)))
    return fail(TE_ERR_INVALID_ARG, "q, k, v, out must be 16-byte aligned");
  if (e4m3.on) {
    if (d % 16 != 0 || d > 128)
      return fail(TE_ERR_UNSUPPORTED, "the e4m3 forward needs head dim a multiple of 16, <= 128");
    if (!(e4m3.q > 0.f) || !(e4m3.k > 0.f) || !(e4m3.v > 0.f) || !std::isfinite(e4m3.q) ||
        !std::isfinite(e4m3.k) || !std::isfinite(e4m3.v))
      return fail(TE_ERR_INVALID_ARG, "descale factors must be finite and > 0");
  }
  Layout L;
  if (!make_layout(batch, total_q, total_kv, hq, false, &L))
    return fail(TE_ERR_INVALID_ARG, "sizes out of range");
  const size_t need = L.total + (e4m3.on ? widened_v_bytes(total_kv, hkv, d) : 0);
  if (workspace_bytes < need)
    return fail(TE_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than the *_workspace_size() answer");
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return fail(TE_ERR_CUDA, "no CUDA device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // e4m3: the softmax sees attn_scale * q_descale * k_descale times the e4m3 dot product
  const float scale = e4m3.on ? attn_scale * e4m3.q * e4m3.k : attn_scale;
  teattn::AttnParams p = base_params(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                                     cu_seqlens_kv_padded, batch, total_q, total_kv, hq, hkv, d,
                                     scale, mask_type, workspace, L);
  if (sbhd) {
    p.sbhd = 1;
    p.rs = batch;
  }
  char* ws = static_cast<char*>(workspace);
  p.q = q;
  p.k = k;
  p.v = e4m3.on ? static_cast<const void*>(ws + L.total) : v;
  p.out = out;
  p.lse = lse;
  p.sched_lists = d <= 128 ? teattn::kListF : teattn::kListQ;
  int* pref_q = reinterpret_cast<int*>(ws + L.pref_q);
  int* pref_k = reinterpret_cast<int*>(ws + L.pref_k);
  const bool bf16 = dtype == TE_DTYPE_BF16;
  cudaError_t e = timed(TE_KERNEL_SCHEDULE, st, [&] { return teattn::launch_schedule(p, pref_q, pref_k, reinterpret_cast<int*>(ws + L.pref_f), st); });
  if (e != cudaSuccess) return cuda_fail(e, "schedule");
  if (e4m3.on && total_kv > 0) {
    // every row of V, pad slots included (they are finite e4m3 values)
    e = timed(TE_KERNEL_WIDEN, st, [&] {
      return teattn::launch_widen_e4m3(v, ws + L.total, static_cast<size_t>(total_kv) * hkv * d,
                                       e4m3.v, sms, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "widen V");
  }
  if (total_q > 0 && total_kv > 0) {
    e = timed(TE_KERNEL_FWD, st, [&] {
      if (e4m3.on) return teattn::launch_attn_fwd_pair_e4m3(p, sms, st);
      return d <= 128 ? teattn::launch_attn_fwd_pair(p, bf16, sms, st)
                      : teattn::launch_attn_fwd(p, bf16, sms, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "attention forward");
  }
  if (total_q > 0) {
    e = timed(TE_KERNEL_ZERO_FILL, st, [&] { return teattn::launch_zero_fill(p, 0, sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "zero fill");
  }
  return ok_status();
}

int te_attn_fwd_thd(const void* q, const void* k, const void* v, void* out, float* lse,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                    const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int batch,
                    int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv, int hq, int hkv,
                    int d, float attn_scale, int mask_type, int dtype, void* workspace,
                    size_t workspace_bytes, void* stream) {
  (void)max_seqlen_q;
  (void)max_seqlen_kv;
  return fwd_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                  cu_seqlens_kv_padded, batch, total_q, total_kv, hq, hkv, d, attn_scale, mask_type,
                  dtype, workspace, workspace_bytes, stream, false);
}

// Rows of a [seq, batch, heads, d] tensor; -1 (an error) for bad sizes or int overflow.
static int sbhd_rows(int batch, int seq) {
  if (batch < 1 || seq < 0) return -1;
  const long long rows = static_cast<long long>(batch) * seq;
  return rows > INT32_MAX ? -1 : static_cast<int>(rows);
}

int te_attn_fwd_sbhd(const void* q, const void* k, const void* v, void* out, float* lse,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch, int seq_q,
                     int seq_kv, int hq, int hkv, int d, float attn_scale, int mask_type, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream) {
  const int tq = sbhd_rows(batch, seq_q), tk = sbhd_rows(batch, seq_kv);
  if (tq < 0 || tk < 0) return fail(TE_ERR_INVALID_ARG, "batch >= 1, seq_q/seq_kv >= 0, rows < 2^31");
  // the real prefix sums stand in for the padded ones, which this layout does not use
  return fwd_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q, cu_seqlens_kv,
                  batch, tq, tk, hq, hkv, d, attn_scale, mask_type, dtype, workspace,
                  workspace_bytes, stream, true);
}

size_t te_attn_fwd_e4m3_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv,
                                       int d) {
  Layout L;
  if (!make_layout(batch, total_q, total_kv, hq, false, &L)) return 0;
  return L.total + widened_v_bytes(total_kv, hkv, d);
}

int te_attn_fwd_thd_e4m3(const void* q, const void* k, const void* v, void* out, float* lse,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                         const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                         int batch, int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                         int hq, int hkv, int d, float attn_scale, float q_descale, float k_descale,
                         float v_descale, int mask_type, void* workspace, size_t workspace_bytes,
                         void* stream) {
  (void)max_seqlen_q;
  (void)max_seqlen_kv;
  return fwd_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                  cu_seqlens_kv_padded, batch, total_q, total_kv, hq, hkv, d, attn_scale, mask_type,
                  TE_DTYPE_BF16, workspace, workspace_bytes, stream, false,
                  E4m3Scales{true, q_descale, k_descale, v_descale});
}

}  // extern "C"

namespace teattn {
// Every host-side check of a backward call except the workspace ones: TE_OK or the
// error code (with the message for te_attn_last_error()).
int bwd_check_args(const void* q, const void* k, const void* v, const void* out, const void* dout,
                   const float* lse, const void* dq, const void* dk, const void* dv,
                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                   const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                   int batch, int total_q, int total_kv, int hq, int hkv, int d, float attn_scale,
                   int mask_type, int dtype) {
  int rc = check_common(batch, total_q, total_kv, hq, hkv, d, attn_scale, mask_type, dtype,
                        cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded);
  if (rc != TE_OK) return rc;
  if (total_q > 0 && (!q || !out || !dout || !lse || !dq))
    return fail(TE_ERR_INVALID_ARG, "q, out, dout, lse and dq must not be NULL");
  if (total_kv > 0 && (!k || !v || !dk || !dv))
    return fail(TE_ERR_INVALID_ARG, "k, v, dk and dv must not be NULL");
  const void* ptrs[] = {q, k, v, out, dout, dq, dk, dv};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return fail(TE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  Layout L;
  if (!make_layout(batch, total_q, total_kv, hq, true, &L))
    return fail(TE_ERR_INVALID_ARG, "sizes out of range");
  return TE_OK;
}
}  // namespace teattn

extern "C" {

static int bwd_impl(const void* q, const void* k, const void* v, const void* out, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                    const int32_t* cu_seqlens_kv_padded, int batch, int total_q, int total_kv,
                    int hq, int hkv, int d, float attn_scale, int mask_type, int dtype,
                    void* workspace, size_t workspace_bytes, void* stream, cudaEvent_t dq_done,
                    bool sbhd, bool fused = false) {
  int rc = teattn::bwd_check_args(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv,
                                  cu_seqlens_q_padded, cu_seqlens_kv_padded, batch, total_q,
                                  total_kv, hq, hkv, d, attn_scale, mask_type, dtype);
  if (rc != TE_OK) return rc;
  if (!workspace) return fail(TE_ERR_INVALID_ARG, "workspace must not be NULL");
  const int cols = fused ? fused_cols(d) : 0;
  if (fused && cols == 0) return fail(TE_ERR_UNSUPPORTED, "the fused backward needs head dim <= 128");
  Layout L;
  if (!make_layout(batch, total_q, total_kv, hq, true, &L, cols, hkv))
    return fail(TE_ERR_INVALID_ARG, "sizes out of range");
  if (workspace_bytes < L.total)
    return fail(TE_ERR_WORKSPACE_TOO_SMALL,
                fused ? "workspace smaller than te_attn_bwd_fused_workspace_size()"
                      : "workspace smaller than te_attn_bwd_workspace_size()");
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return fail(TE_ERR_CUDA, "no CUDA device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  teattn::AttnParams p = base_params(cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                                     cu_seqlens_kv_padded, batch, total_q, total_kv, hq, hkv, d,
                                     attn_scale, mask_type, workspace, L);
  if (sbhd) {
    p.sbhd = 1;
    p.rs = batch;
  }
  p.q = q;
  p.k = k;
  p.v = v;
  p.sched_lists = fused ? teattn::kListKChain : (teattn::kListQ | teattn::kListK);
  p.out_in = out;
  p.dout = dout;
  p.lse_in = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  char* ws = static_cast<char*>(workspace);
  p.lse_t = reinterpret_cast<float*>(ws + L.lse_t);
  p.delta_t = reinterpret_cast<float*>(ws + L.delta_t);
  if (fused) {
    p.dq_acc = reinterpret_cast<float*>(ws + L.dq_acc);
    p.dq_sem = reinterpret_cast<int*>(ws + L.dq_sem);
    p.dq_cols = cols;
    p.k_items = reinterpret_cast<int4*>(ws + L.k_items);
  }
  int* pref_q = reinterpret_cast<int*>(ws + L.pref_q);
  p.pref_q = pref_q;
  int* pref_k = reinterpret_cast<int*>(ws + L.pref_k);
  const bool bf16 = dtype == TE_DTYPE_BF16;
  cudaError_t e = timed(TE_KERNEL_SCHEDULE, st, [&] { return teattn::launch_schedule(p, pref_q, pref_k, reinterpret_cast<int*>(ws + L.pref_f), st); });
  if (e != cudaSuccess) return cuda_fail(e, "schedule");
  // Rows no tile writes are zeroed first (they depend on the lengths only), so dq
  // is final as soon as the dQ kernel ends and dk/dv when the dK/dV kernel does.
  e = timed(TE_KERNEL_ZERO_FILL, st, [&] { return teattn::launch_zero_fill(p, 1, sms, st); });
  if (e != cudaSuccess) return cuda_fail(e, "zero fill");
  if (total_q > 0) {
    e = timed(TE_KERNEL_DELTA, st, [&] { return teattn::launch_delta(p, bf16, sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "delta");
  }
  if (fused) {
    if (total_q > 0 && total_kv > 0) {
      e = timed(TE_KERNEL_BWD_FUSED, st, [&] { return teattn::launch_attn_bwd_fused(p, bf16, sms, st); });
      if (e != cudaSuccess) return cuda_fail(e, "fused backward");
      e = timed(TE_KERNEL_DQ_CONVERT, st, [&] { return teattn::launch_dq_convert(p, bf16, sms, st); });
      if (e != cudaSuccess) return cuda_fail(e, "dQ conversion");
    }
    if (dq_done) {
      e = cudaEventRecord(dq_done, st);
      if (e != cudaSuccess) return cuda_fail(e, "dq event record");
    }
    return ok_status();
  }
  if (total_q > 0 && total_kv > 0) {
    e = timed(TE_KERNEL_DQ, st, [&] { return teattn::launch_attn_bwd_dq(p, bf16, sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "dQ");
  }
  if (dq_done) {
    e = cudaEventRecord(dq_done, st);
    if (e != cudaSuccess) return cuda_fail(e, "dq event record");
  }
  if (total_q > 0 && total_kv > 0) {
    e = timed(TE_KERNEL_DKDV, st, [&] { return teattn::launch_attn_bwd_dkdv(p, bf16, sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "dK/dV");
  }
  return ok_status();
}

int te_attn_bwd_thd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                    const int32_t* cu_seqlens_kv_padded, int batch, int total_q, int total_kv,
                    int max_seqlen_q, int max_seqlen_kv, int hq, int hkv, int d, float attn_scale,
                    int mask_type, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  (void)max_seqlen_q;
  (void)max_seqlen_kv;
  return bwd_impl(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                  cu_seqlens_kv_padded, batch, total_q, total_kv, hq, hkv, d, attn_scale, mask_type,
                  dtype, workspace, workspace_bytes, stream, nullptr, false);
}

int te_attn_bwd_thd_fused(const void* q, const void* k, const void* v, const void* out,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                          const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                          int batch, int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                          int hq, int hkv, int d, float attn_scale, int mask_type, int dtype,
                          void* workspace, size_t workspace_bytes, void* stream) {
  (void)max_seqlen_q;
  (void)max_seqlen_kv;
  return bwd_impl(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                  cu_seqlens_kv_padded, batch, total_q, total_kv, hq, hkv, d, attn_scale, mask_type,
                  dtype, workspace, workspace_bytes, stream, nullptr, false, true);
}

int te_attn_bwd_thd_ev(const void* q, const void* k, const void* v, const void* out, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                       const int32_t* cu_seqlens_kv_padded, int batch, int total_q, int total_kv,
                       int max_seqlen_q, int max_seqlen_kv, int hq, int hkv, int d, float attn_scale,
                       int mask_type, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                       void* dq_done) {
  (void)max_seqlen_q;
  (void)max_seqlen_kv;
  return bwd_impl(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                  cu_seqlens_kv_padded, batch, total_q, total_kv, hq, hkv, d, attn_scale, mask_type,
                  dtype, workspace, workspace_bytes, stream, static_cast<cudaEvent_t>(dq_done), false);
}

int te_attn_bwd_sbhd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens_q,
                     const int32_t* cu_seqlens_kv, int batch, int seq_q, int seq_kv, int hq, int hkv,
                     int d, float attn_scale, int mask_type, int dtype, void* workspace,
                     size_t workspace_bytes, void* stream) {
  const int tq = sbhd_rows(batch, seq_q), tk = sbhd_rows(batch, seq_kv);
  if (tq < 0 || tk < 0) return fail(TE_ERR_INVALID_ARG, "batch >= 1, seq_q/seq_kv >= 0, rows < 2^31");
  return bwd_impl(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q,
                  cu_seqlens_kv, batch, tq, tk, hq, hkv, d, attn_scale, mask_type, dtype, workspace,
                  workspace_bytes, stream, nullptr, true);
}

int te_attn_read_status(const void* workspace, int* status, void* stream) {
  if (!workspace || !status) return fail(TE_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  e = cudaMemcpy(status, static_cast<const char*>(workspace), sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status copy");
  return ok_status();
}

int te_attn_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = enable != 0;
  return ok_status();
}

int te_attn_profile_read(double* total_ms, int* launches) {
  if (!total_ms || !launches) return fail(TE_ERR_INVALID_ARG, "NULL argument");
  std::vector<ProfRecord> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  for (int k = 0; k < TE_NUM_KERNELS; ++k) {
    total_ms[k] = 0.0;
    launches[k] = 0;
  }
  int rc = TE_OK;
  for (ProfRecord& r : recs) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) rc = cuda_fail(e, "profile read");
    if (r.kernel >= 0 && r.kernel < TE_NUM_KERNELS) {
      total_ms[r.kernel] += ms;
      launches[r.kernel] += 1;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  return rc == TE_OK ? ok_status() : rc;
}

const char* te_attn_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"

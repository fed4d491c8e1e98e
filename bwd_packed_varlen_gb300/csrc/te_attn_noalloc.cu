// te_attn_bwd_thd_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain scratch memory for a call: plugin hosts and
// inference servers that own every device allocation and hand a custom operator only
// its input and output buffers, runtimes that forbid allocation after
// initialisation, and foreign-language callers with no CUDA allocator of their own.
// For them this entry point uses a fixed scratch area compiled into the library
// instead of a caller-provided workspace.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes. Every GPU
// that loads it keeps it until the process exits. In host code the array's name is
// only a host-side stand-in, so the device address is looked up with
// cudaGetSymbolAddress (with the device current) the first time a device is used,
// and cached together with the identity of the CUDA context it belongs to; a call
// in a different context (after cudaDeviceReset, say) looks it up again. That first
// call on a device should therefore come before any stream capture. All calls on a
// device share the one array, which keeps the previous call's contents: nothing in
// it has to start at zero (every call rewrites what it reads), but calls that
// overlap on the GPU race on it, so callers must order them (same stream or
// events). No cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/te_attn.h"

namespace teattn {
void set_last_error(const std::string& msg);  // te_attn_api.cu
int bwd_check_args(const void* q, const void* k, const void* v, const void* out, const void* dout,
                   const float* lse, const void* dq, const void* dk, const void* dv,
                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                   const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                   int batch, int total_q, int total_kv, int hq, int hkv, int d, float attn_scale,
                   int mask_type, int dtype);  // te_attn_api.cu
}  // namespace teattn

namespace {

constexpr size_t kNoAllocScratchBytes = TE_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct Cached {
  void* ptr;
  unsigned long long ctx_id;  // 0: not set up
};
Cached g_noalloc[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (0 when it cannot be
// read), through driver entry points resolved by the runtime (no -lcuda).
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = []() -> GetCurrent {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<GetCurrent>(f);
  }();
  static GetId get_id = []() -> GetId {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<GetId>(f);
  }();
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device, set up once per
// device and context. Returns nullptr and fills `err` on failure.
void* scratch_for_current_device(std::string* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *err = "device ordinal out of range";
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  Cached& c = g_noalloc[dev];
  const unsigned long long id = current_context_id();
  if (c.ptr == nullptr || id == 0 || id != c.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *err = std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
      return nullptr;
    }
    c.ptr = p;
    // the lookup made the device's primary context current if none was
    c.ctx_id = id != 0 ? id : current_context_id();
  }
  return c.ptr;
}

}  // namespace

extern "C" {

int te_attn_bwd_thd_noalloc(const void* q, const void* k, const void* v, const void* out,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                            const int32_t* cu_seqlens_q_padded,
                            const int32_t* cu_seqlens_kv_padded, int batch, int total_q,
                            int total_kv, int max_seqlen_q, int max_seqlen_kv, int hq, int hkv,
                            int d, float attn_scale, int mask_type, int dtype, void* stream) {
  // the same argument checks, codes and messages as te_attn_bwd_thd, first
  const int rc = teattn::bwd_check_args(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q,
                                        cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                                        batch, total_q, total_kv, hq, hkv, d, attn_scale,
                                        mask_type, dtype);
  if (rc != TE_OK) return rc;
  const size_t need = te_attn_bwd_workspace_size(batch, total_q, total_kv, hq, hkv, d);
  if (need > kNoAllocScratchBytes) {
    teattn::set_last_error("problem needs " + std::to_string(need) +
                           " bytes of scratch, more than the built-in " +
                           std::to_string(kNoAllocScratchBytes) +
                           " bytes; call te_attn_bwd_thd with a workspace instead");
    return TE_ERR_WORKSPACE_TOO_SMALL;
  }
  std::string err;
  void* scratch = scratch_for_current_device(&err);
  if (scratch == nullptr) {
    teattn::set_last_error(err);
    return TE_ERR_CUDA;
  }
  return te_attn_bwd_thd(q, k, v, out, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv,
                         cu_seqlens_q_padded, cu_seqlens_kv_padded, batch, total_q, total_kv,
                         max_seqlen_q, max_seqlen_kv, hq, hkv, d, attn_scale, mask_type, dtype,
                         scratch, kNoAllocScratchBytes, stream);
}

int te_attn_read_status_noalloc(int* status, void* stream) {
  if (!status) {
    teattn::set_last_error("NULL argument");
    return TE_ERR_INVALID_ARG;
  }
  std::string err;
  void* scratch = scratch_for_current_device(&err);
  if (scratch == nullptr) {
    teattn::set_last_error(err);
    return TE_ERR_CUDA;
  }
  // the status word is the first word of the scratch array, as of any workspace
  return te_attn_read_status(scratch, status, stream);
}

}  // extern "C"

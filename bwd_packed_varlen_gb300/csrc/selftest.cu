// te_attn_selftest_wait_timeout: runs the library's bounded-wait unwind path on
// purpose, without any copy or tensor-core work in flight, so that a test can check
// that a wait which can never finish gives up, records TE_STATUS_TIMEOUT, lets the
// other roles of the block give up too, frees the block's tensor memory and
// returns with the GPU context intact.
//
// One block of two warps, laid out like the attention kernels' roles:
//   warp 1 allocates all 512 TMEM columns (as every tensor-core kernel here does)
//          and frees them at the end;
//   warp 0, lane 0 waits with the caller's short limit on an mbarrier that no
//          thread ever arrives on -- the wait runs out and sets the timeout bit;
//   warp 1, lane 0 waits with the library's default limit (4 s) on a second
//          mbarrier that warp 0 would only arrive on after a normal first wait --
//          it sees the timeout bit and gives up early, as every other wait of a
//          kernel does once one of them has timed out.
// Header words kHdrSelftest.. record what happened (see the header file).
#include <cuda_runtime.h>

#include <string>

#include "../../include/te_attn.h"
#include "common.cuh"
#include "sm103_ptx.cuh"

namespace teattn {

void set_last_error(const std::string& msg);  // te_attn_api.cu

__global__ void __launch_bounds__(64, 1)
    selftest_wait_kernel(int* header, unsigned long long limit_ns) {
  __shared__ uint64_t bar_never, bar_after;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  int* status = header + kHdrStatus;
  if (tid == 0) {
    *status = 0;
    for (int i = 0; i < 4; ++i) header[kHdrSelftest + i] = 0;
    mbar_init(&bar_never, 1);
    mbar_init(&bar_after, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const unsigned long long t0 = global_ns();
    const bool ok = mbar_wait_limit(&bar_never, 0, status, limit_ns);
    if (ok) mbar_arrive(&bar_after);
    header[kHdrSelftest + 0] = ok ? 1 : 0;
    header[kHdrSelftest + 1] = static_cast<int>((global_ns() - t0) / 1000ull);  // microseconds
  } else if (tid == 32) {
    const unsigned long long t0 = global_ns();
    const bool ok = mbar_wait(&bar_after, 0, status);
    header[kHdrSelftest + 2] = static_cast<int>((global_ns() - t0) / 1000ull);
    (void)ok;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_slot, 512);
  }
  __syncthreads();
  if (tid == 0) header[kHdrSelftest + 3] = 1;  // reached the end, TMEM freed
}

}  // namespace teattn

extern "C" int te_attn_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                             unsigned int limit_us, void* stream) {
  if (!workspace) {
    teattn::set_last_error("workspace must not be NULL");
    return TE_ERR_INVALID_ARG;
  }
  if (workspace_bytes < teattn::kHdrWords * sizeof(int)) {
    teattn::set_last_error("workspace smaller than its 256-byte header");
    return TE_ERR_WORKSPACE_TOO_SMALL;
  }
  if (limit_us < 1 || limit_us > 1000000) {
    teattn::set_last_error("limit_us must lie in [1, 1000000]");
    return TE_ERR_INVALID_ARG;
  }
  teattn::selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int*>(workspace), static_cast<unsigned long long>(limit_us) * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    teattn::set_last_error(std::string("selftest launch: ") + cudaGetErrorString(e));
    return TE_ERR_CUDA;
  }
  teattn::set_last_error("");
  return TE_OK;
}

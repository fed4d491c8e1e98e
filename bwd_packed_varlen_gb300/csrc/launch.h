// Host-side launchers of the library's kernels (internal; the public surface is
// include/te_attn.h).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace teattn {

cudaError_t launch_schedule(const AttnParams& p, int* pref_q, int* pref_k, int* pref_f,
                            cudaStream_t st);
cudaError_t launch_zero_fill(const AttnParams& p, int mode, int num_sms, cudaStream_t st);
cudaError_t launch_delta(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st);
cudaError_t launch_widen_e4m3(const void* src, void* dst, size_t n, float scale, int num_sms,
                              cudaStream_t st);

cudaError_t launch_attn_fwd(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st);
cudaError_t launch_attn_fwd_pair(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st);
cudaError_t launch_attn_fwd_pair_e4m3(const AttnParams& p, int num_sms, cudaStream_t st);
cudaError_t launch_attn_bwd_dkdv(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st);
cudaError_t launch_attn_bwd_dq(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st);
cudaError_t launch_attn_bwd_fused(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st);
cudaError_t launch_dq_convert(const AttnParams& p, bool bf16, int num_sms, cudaStream_t st);

}  // namespace teattn

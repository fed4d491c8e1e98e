/*
 * te_attn.h -- C ABI of libteattn.so: scaled-dot-product attention forward and
 * backward over packed variable-length (THD) sequences, for NVIDIA GB300 (sm_103a).
 *
 * Pages cited, by title (keys are the pages' issue numbers):
 *   [2448] "Inconsistent fused_attn_bwd results of dk, dv under THD layout + GQA on multiple calls"
 *   [3333] "[Bug] FusedAttention (cuDNN) THD backward produces wrong gradients on sm_120 (RTX 5090); forward is correct, Unfused is correct"
 *   [3216] "flash-attn-4 4.0.0b11: DotProductAttention batched backward returns wrong dQ/dK/dV at head_dim=256 on Blackwell (sm_100)"
 *   [2892] "[BUG] SIGSEGV in fused_attn_fwd when cu_seqlens_q != cu_seqlens_q_padded with FP8 blockwise"
 *
 * What is computed (the TransformerEngine issues this library answers):
 *   For each sequence b and query head h (key/value head g = h / (hq / hkv)):
 *     S   = attn_scale * Q_b,h K_b,g^T        masked by the REAL lengths
 *     P   = softmax(S) row-wise,  LSE = log(sum_j exp(S_ij))  (natural log)
 *     O   = P V_b,g
 *   and the gradient of sum(dO * O):
 *     dV  = sum_{h in group} P^T dO,   dP = dO V^T,   D = rowsum(dO * O)
 *     dS  = P * (dP - D),  dQ = attn_scale dS K,  dK = attn_scale sum_{h in group} dS^T Q
 *   -- [2448] (THD + GQA fused_attn_bwd, "Expected behavior": rows of an empty
 *      query sequence give exactly-zero dk/dv, results must not depend on earlier
 *      calls), [3333] (THD padding_causal backward vs a per-sequence SDPA
 *      reference), [3216] (GQA via repeat_interleave, causal = upper-left
 *      triangle, head_dim 256 with batch >= 2), [2892] ("Expected Behavior":
 *      cu_seqlens_* mask, cu_seqlens_*_padded index memory, output keeps the padded
 *      layout).
 *
 * Layout (all tensors contiguous, row-major, device memory owned by the caller):
 *   q, out, dout, dq : [total_q,  hq,  d]   16-bit (fp16 or bf16, all the same)
 *   k, v, dk, dv     : [total_kv, hkv, d]   same dtype
 *   lse              : [total_q,  hq]       fp32
 *   cu_seqlens_q/kv          : int32 [batch+1] prefix sums of REAL lengths
 *   cu_seqlens_q/kv_padded   : int32 [batch+1] prefix sums of PADDED lengths;
 *       sequence b occupies rows cu_*_padded[b] .. cu_*_padded[b+1]-1 and its real
 *       tokens are the first (cu_*[b+1]-cu_*[b]) of those rows.
 *   Rows that are not real tokens (pad slots, tails after cu_*_padded[batch], rows
 *   of empty sequences) are written as exact zeros in out/dq/dk/dv and 0 in lse;
 *   key/value rows no real query sees are exact zeros in dk/dv. A real query that
 *   sees no key (its sequence has no real key, or it precedes a lower-right
 *   causal triangle) gets out = 0, lse = -inf, dq = 0.
 *   Pad slots may hold any finite values; they never reach a real output.
 *   q, k, v, out, dout, dq, dk and dv must start on a 16-byte boundary (tiles are
 *   moved with 16-byte vector and bulk-tensor copies); a pointer that does not is
 *   answered with TE_ERR_INVALID_ARG before anything is launched. lse and the
 *   cu_seqlens arrays need their natural 4-byte alignment.
 *
 * Supported: d a multiple of 8 with 8 <= d <= 256; hq a positive multiple of hkv;
 *   mask TE_MASK_PADDING, TE_MASK_PADDING_CAUSAL (key j visible to query i iff
 *   j <= i, upper-left aligned, the alignment [3216] uses) or
 *   TE_MASK_PADDING_CAUSAL_BOTTOM_RIGHT (key j visible iff j <= i + Lk - Lq, the
 *   triangle aligned to the last query and key; TransformerEngine's
 *   "padding_causal_bottom_right" -- the pages use equal lengths only, where the
 *   two causal masks agree); dtype TE_DTYPE_FP16 or TE_DTYPE_BF16.
 *
 * Determinism: no floating-point atomics; every output element is produced by one
 *   thread block in a fixed order, so repeated calls on identical inputs give
 *   bit-identical results regardless of call order, earlier calls, or the contents
 *   of the output and workspace buffers on entry.
 *
 * Workspace: caller-allocated device memory of at least the size returned by the
 *   matching *_workspace_size function. Its contents on entry are irrelevant: every
 *   call rewrites what it reads. The library allocates no device memory and keeps no
 *   state between calls. max_seqlen_q/kv are accepted for interface parity with
 *   TransformerEngine and ignored (lengths come from the cu_seqlens arrays).
 *
 * Streams: every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *   default stream); no host synchronisation. Calls that share a workspace must be
 *   ordered (same stream or explicit events).
 * CUDA graphs: the compute entry points neither allocate nor synchronise, so a
 *   sequence of calls can be captured into a graph and replayed; each replay reads
 *   the buffers' contents at replay time and gives the bits an eager call would.
 *   Make one eager call of each entry point before capturing (the first call sets
 *   kernel attributes). Not capturable: te_attn_read_status*, te_attn_profile_read
 *   (they synchronise) and profiling itself.
 *
 * Errors: functions return TE_OK (0) or a negative TE_ERR_* code, and
 *   te_attn_last_error() gives a thread-local message. Host-detectable argument
 *   errors launch nothing. Errors that need device data (inconsistent cu_seqlens, a
 *   pipeline wait that timed out) are recorded in a status word in the workspace;
 *   te_attn_read_status() reads it after synchronising the stream.
 */
#ifndef TE_ATTN_H_
#define TE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TE_MASK_PADDING 1
#define TE_MASK_PADDING_CAUSAL 2
#define TE_MASK_PADDING_CAUSAL_BOTTOM_RIGHT 3

#define TE_DTYPE_FP16 0
#define TE_DTYPE_BF16 1

#define TE_OK 0
#define TE_ERR_INVALID_ARG (-1)
#define TE_ERR_UNSUPPORTED (-2)
#define TE_ERR_WORKSPACE_TOO_SMALL (-3)
#define TE_ERR_CUDA (-4)
#define TE_ERR_BAD_SEQLENS (-5)
#define TE_ERR_TIMEOUT (-6)

/*
 * Device status bits reported by te_attn_read_status():
 *   TE_STATUS_BAD_SEQLENS   cu_seqlens inconsistent with the tensor extents (a real
 *                           length above its padded one, offsets past the tensor);
 *                           the offending sequences are treated as empty.
 *   TE_STATUS_TIMEOUT       a pipeline wait inside a kernel ran past its limit (4 s);
 *                           every other wait of that kernel then gave up too, the
 *                           kernel freed its tensor memory and returned, and the
 *                           outputs of the call are undefined.
 *   TE_STATUS_OUT_OF_BOUNDS only in the debug build of the library (compiled with
 *                           TEATTN_DEBUG_BOUNDS, libteattn_debug.so): a computed
 *                           global offset fell outside its buffer; the access was
 *                           skipped. The release build does not check.
 */
#define TE_STATUS_BAD_SEQLENS 1
#define TE_STATUS_TIMEOUT 2
#define TE_STATUS_OUT_OF_BOUNDS 4
/* A kernel found its launch unusable (shared memory not 1024-byte aligned); it
   returned without computing and the outputs of the call are undefined. */
#define TE_STATUS_INTERNAL 8

/* Library version, major * 10000 + minor * 100 + patch. */
int te_attn_version(void);

/* Bytes of workspace te_attn_fwd_thd needs for these sizes (0 on invalid sizes). */
size_t te_attn_fwd_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv,
                                  int d);

/* Bytes of workspace te_attn_bwd_thd needs for these sizes (0 on invalid sizes). */
size_t te_attn_bwd_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv,
                                  int d);

/*
 * Forward: writes out [total_q, hq, d] and lse [total_q, hq] (natural-log softmax
 * denominator of the scaled scores, fp32). [2892] "Expected Behavior" fixes the
 * real/padded split; [2448] passes lse to the backward as the aux tensor.
 */
int te_attn_fwd_thd(const void* q, const void* k, const void* v, void* out, float* lse,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                    const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                    int batch, int total_q, int total_kv, int max_seqlen_q,
                    int max_seqlen_kv, int hq, int hkv, int d, float attn_scale,
                    int mask_type, int dtype, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Backward: from q, k, v, out, dout and lse, writes dq [total_q, hq, d],
 * dk and dv [total_kv, hkv, d]. dk/dv of a key/value head sum over the hq/hkv query
 * heads of its group inside one thread block (no atomics). The arguments mirror
 * TransformerEngine's fused_attn_bwd as [2448] calls it (out and lse are
 * inputs; dropout 0; no bias; deterministic). dq comes from a separate kernel that
 * owns each query tile and recomputes its scores, so no partial sums of dq ever
 * meet in global memory.
 */
int te_attn_bwd_thd(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                    const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                    int batch, int total_q, int total_kv, int max_seqlen_q,
                    int max_seqlen_kv, int hq, int hkv, int d, float attn_scale,
                    int mask_type, int dtype, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Backward with a hand-over point (no counterpart in the pages): identical results
 * to te_attn_bwd_thd, plus `dq_done`, a cudaEvent_t created by the caller (or NULL),
 * is recorded on `stream` as soon as dq is final -- the backward computes dq before
 * dk and dv -- so that the caller can start consuming dq (a copy to the host, a
 * collective) on another stream while dk/dv are still being computed. Returns what
 * te_attn_bwd_thd returns, or TE_ERR_CUDA if the event cannot be recorded.
 */
int te_attn_bwd_thd_ev(const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                       const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                       int batch, int total_q, int total_kv, int max_seqlen_q,
                       int max_seqlen_kv, int hq, int hkv, int d, float attn_scale,
                       int mask_type, int dtype, void* workspace, size_t workspace_bytes,
                       void* stream, void* dq_done);

/*
 * Fused backward (no counterpart in the pages' code; the deterministic fused dQ of
 * the FlashAttention line of backward kernels, done without atomics in any varying
 * order): the same arguments and results, within the same tolerances, as
 * te_attn_bwd_thd, for head dims up to 128 (TE_ERR_UNSUPPORTED above). One kernel
 * computes dK, dV and each key tile's share of dQ from a single pass over the
 * scores -- five products instead of seven -- and adds the shares of every
 * (query tile, head) into an fp32 accumulator in the workspace in a fixed order
 * (descending key tiles, ordered by a counter per tile); a conversion kernel then
 * writes dq. Repeated calls are bit-identical; the results are not bit-identical to
 * te_attn_bwd_thd's (dq is summed in another order). The workspace, of
 * te_attn_bwd_fused_workspace_size() bytes, holds the accumulator (4 bytes per
 * padded query row, head and column, the head dim rounded up to 64 or 128).
 * On GB300 this path is slower than te_attn_bwd_thd at the sizes measured here:
 * moving each key tile's 64 KB fp32 share out of the SM costs more than the two
 * recomputed products save.
 */
size_t te_attn_bwd_fused_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv,
                                        int d);
int te_attn_bwd_thd_fused(const void* q, const void* k, const void* v, const void* out,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                          const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                          int batch, int total_q, int total_kv, int max_seqlen_q,
                          int max_seqlen_kv, int hq, int hkv, int d, float attn_scale,
                          int mask_type, int dtype, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * Sequence-major layout ("sbhd", the layout of [3216]'s reproduction: q, k, v of
 * shape [s, b, h, d], its fp32_reference indexing q[s, b, hq, d]):
 *   q, out, dout, dq : [seq_q,  batch, hq,  d]   16-bit, contiguous
 *   k, v, dk, dv     : [seq_kv, batch, hkv, d]
 *   lse              : [seq_q,  batch, hq]       fp32
 * Token i of sequence b is row i * batch + b of the flattened [seq * batch, h, d]
 * tensor. cu_seqlens_q/kv (int32 [batch+1]) are the prefix sums of the REAL
 * lengths, each at most seq_q / seq_kv: tokens 0 .. len-1 of batch entry b are
 * real and the rest are pad slots, written as exact zeros like the packed
 * layout's (there are no padded prefix sums: every entry spans seq_* tokens).
 * Same masks, numerics, determinism and errors as te_attn_fwd_thd /
 * te_attn_bwd_thd; the workspace sizes are those functions' for total_q =
 * batch * seq_q and total_kv = batch * seq_kv. Returns TE_ERR_INVALID_ARG when
 * batch < 1, a seq_* < 0 or batch * seq_* overflows int.
 */
int te_attn_fwd_sbhd(const void* q, const void* k, const void* v, void* out, float* lse,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                     int seq_q, int seq_kv, int hq, int hkv, int d, float attn_scale,
                     int mask_type, int dtype, void* workspace, size_t workspace_bytes,
                     void* stream);

int te_attn_bwd_sbhd(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                     int seq_q, int seq_kv, int hq, int hkv, int d, float attn_scale,
                     int mask_type, int dtype, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * e4m3 forward (no counterpart in the pages' code; [2892] is the report of TE's
 * FP8 forward failing when cu_seqlens_q != cu_seqlens_q_padded -- out of bounds
 * and an unpadded output -- and this entry keeps that case exact): q, k, v hold
 * FP8 e4m3 bytes in the packed layout ([total_q, hq, d], [total_kv, hkv, d]) with
 * per-tensor dequantisation factors (real value = stored value * descale), out is
 * bf16 [total_q, hq, d] and lse fp32 [total_q, hq], both in the padded layout with
 * the same exact-zero rows as te_attn_fwd_thd. Scores are formed on the e4m3
 * tensor-core path (attn_scale * q_descale * k_descale times the e4m3 dot
 * products, fp32 accumulation); V is widened once to bf16 (times v_descale) in
 * the workspace and P V runs in bf16 like te_attn_fwd_thd. Needs d a multiple of
 * 16 with d <= 128, descale factors finite and > 0, and a workspace of
 * te_attn_fwd_e4m3_workspace_size() bytes. Same masks, determinism and errors as
 * te_attn_fwd_thd otherwise.
 */
size_t te_attn_fwd_e4m3_workspace_size(int batch, int total_q, int total_kv, int hq, int hkv,
                                       int d);

int te_attn_fwd_thd_e4m3(const void* q, const void* k, const void* v, void* out, float* lse,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                         const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded,
                         int batch, int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                         int hq, int hkv, int d, float attn_scale, float q_descale, float k_descale,
                         float v_descale, int mask_type, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Synchronises `stream`, then copies the device status word of the last call that
 * used `workspace` into *status (0 = clean, else TE_STATUS_* bits). Returns TE_OK or
 * TE_ERR_CUDA. Intended for tests and debugging; it blocks the host.
 */
int te_attn_read_status(const void* workspace, int* status, void* stream);

/*
 * Self-test of the bounded-wait unwind path (no counterpart in the pages; a test and
 * debugging aid). Launches one block on `stream` that allocates all of its SM's
 * tensor memory, waits with a limit of `limit_us` microseconds (1 .. 1000000) on a
 * barrier no thread ever arrives on, while a second warp waits with the library's
 * default limit on a barrier the first would release. The first wait runs out and
 * records TE_STATUS_TIMEOUT in the status word of `workspace` (at least 256 bytes);
 * the second sees the bit and gives up early; the block frees its tensor memory and
 * returns. Afterwards te_attn_read_status(workspace) reports TE_STATUS_TIMEOUT and
 * header words 8..11 of the workspace hold: the first wait's result (0 = timed out),
 * its duration and the second wait's duration in microseconds, and 1 once the block
 * reached its end. The GPU context stays usable; a later call that uses the same
 * workspace rewrites the status word. Returns TE_OK, TE_ERR_INVALID_ARG,
 * TE_ERR_WORKSPACE_TOO_SMALL or TE_ERR_CUDA (launch failure).
 */
int te_attn_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                  unsigned int limit_us, void* stream);

/*
 * Kernel timing (profiling aid). te_attn_profile_enable(1) makes every later call
 * bracket each of its kernel launches with a pair of CUDA events recorded on the
 * call's stream; te_attn_profile_read() synchronises on those events, adds each
 * kernel's elapsed time and launch count into total_ms[k] / launches[k] for
 * k = TE_KERNEL_* (arrays of at least TE_NUM_KERNELS entries), and clears the
 * record. Disabled by default; while enabled, each launch costs two event
 * records. Returns TE_OK or TE_ERR_CUDA. The record is process-wide (guarded by a
 * mutex): calls from several threads land in the same totals.
 */
#define TE_KERNEL_SCHEDULE 0
#define TE_KERNEL_FWD 1
#define TE_KERNEL_ZERO_FILL 2
#define TE_KERNEL_DELTA 3
#define TE_KERNEL_DKDV 4
#define TE_KERNEL_DQ 5
#define TE_KERNEL_WIDEN 6
#define TE_KERNEL_BWD_FUSED 7
#define TE_KERNEL_DQ_CONVERT 8
#define TE_NUM_KERNELS 9
int te_attn_profile_enable(int enable);
int te_attn_profile_read(double* total_ms, int* launches);

/*
 * Backward pass for callers that cannot allocate device memory (no counterpart in
 * the pages this library follows; it is an interface addition). Some callers have
 * no way to get scratch memory for a call: plugin hosts and inference servers that
 * own every device allocation and give an operator only its inputs and outputs,
 * runtimes that forbid allocation after start-up, foreign-language callers without
 * a CUDA allocator. This variant of te_attn_bwd_thd takes the same arguments minus
 * the workspace and uses a scratch array of TE_NOALLOC_SCRATCH_BYTES compiled into
 * the library (a __device__ array: every GPU that loads it keeps it until the
 * process exits). It calls no cudaMalloc, cudaFree or other allocating routine.
 * - The first call on a device looks up the array's device address with that
 *   device current and caches it with the identity of the current CUDA context (a
 *   call in another context, e.g. after cudaDeviceReset, looks it up again); make
 *   that first call before any stream capture.
 * - All calls on a device share the one array and it keeps the last call's
 *   contents; nothing in it needs to start at zero (each call rewrites what it
 *   reads), but calls that overlap on the GPU race on it: order them (one stream,
 *   or events).
 * - Arguments are checked first, with the codes and messages of te_attn_bwd_thd;
 *   then TE_ERR_WORKSPACE_TOO_SMALL (and a message naming the size needed) is
 *   returned when te_attn_bwd_workspace_size() of the problem exceeds the array.
 *   Otherwise the results are those of te_attn_bwd_thd, bit for bit.
 * - Device-side errors (TE_STATUS_* bits) land in the array's status word:
 *   te_attn_read_status_noalloc() reads them for the current device.
 */
#define TE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int te_attn_bwd_thd_noalloc(const void* q, const void* k, const void* v, const void* out,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                            const int32_t* cu_seqlens_q_padded,
                            const int32_t* cu_seqlens_kv_padded, int batch, int total_q,
                            int total_kv, int max_seqlen_q, int max_seqlen_kv, int hq, int hkv,
                            int d, float attn_scale, int mask_type, int dtype, void* stream);

/*
 * The status word of the last te_attn_bwd_thd_noalloc call on the current device
 * (as te_attn_read_status() gives it for a workspace): synchronises `stream`, then
 * copies the word into *status. Returns TE_OK, TE_ERR_INVALID_ARG or TE_ERR_CUDA.
 */
int te_attn_read_status_noalloc(int* status, void* stream);

/* Thread-local description of the last error returned on this thread. */
const char* te_attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TE_ATTN_H_ */

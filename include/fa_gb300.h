/*
 * fa_gb300.h - C ABI of the exact IO-aware attention library for GB300 (sm_103a).
 *
 * The operation (forward):
 *     O = softmax(scale * Q K^T + M) V,   LSE_r = log sum_c exp(scale * Q_r . K_c + M_rc)
 * per (batch b, head h), where M is 0 for visible keys and -inf for masked
 * ones. Defined in "FlashAttention算法详解：从IO瓶颈到Triton实现", §先说结论
 * (the definition), §Causal Mask怎么处理 (the causal mask c <= r) and
 * §Backward为什么更复杂 (the saved row statistic LSE = m + log l); also
 * "FlashAttention 完整解析：从原理到 CUDA/Triton 实现", §1.1.
 * The backward computes the gradients of L = sum(O * dO) by the formulas of
 * §Backward为什么更复杂 (dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(dP o P)),
 * dQ = scale * dS K, dK = scale * dS^T Q), recomputing P from the saved LSE.
 *
 * Layout of every tensor: contiguous, row-major [B, H, N, d] (d fastest);
 * Q/K/V/O/dO/dQ/dK/dV are bf16, LSE is fp32 [B, H, N] in natural-log units.
 * Masks: causal (key c visible to query r iff c <= r, top-left aligned) and
 * key padding (key c visible iff c < kv_lens[b]); both may be combined.
 * A query row with no visible key gets O = 0, LSE = -inf and contributes
 * nothing to the backward.
 *
 * Ownership: the caller owns every buffer. The library allocates no device
 * memory and keeps no per-call state; all calls are asynchronous on `stream`
 * (a cudaStream_t, NULL = legacy default stream) and return after the launch.
 * Pointers named "device" must be device (or managed) memory of the current
 * device, 16-byte aligned. Inputs must not alias outputs.
 *
 * Threads: any host thread may call any entry point, also concurrently on
 * different streams. The TMA descriptors that a call encodes are cached on the
 * host (keyed by address, extents, strides and box; behind a mutex), and a
 * thread's first call binds the current device's primary context.
 *
 * Errors: every entry point returns an fa_status. Argument errors are found on
 * the host before any launch. FA_ERR_TIMEOUT is reported only in check mode
 * (environment FA_CHECK=1, or fa_check_status()): every wait inside the
 * kernels is bounded, and a wait that runs out records the timeout in a
 * device status word instead of hanging.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = -1,     /* null pointer, B/H/N < 1, scale not finite or <= 0, bad kv_lens */
  FA_ERR_UNSUPPORTED = -2, /* d not in {64, 128}, pointer not 16-byte aligned, size overflow */
  FA_ERR_LAUNCH = -3,      /* CUDA error at launch (message via fa_last_cuda_error) */
  FA_ERR_TIMEOUT = -4,     /* a bounded device wait ran out (check mode only) */
  FA_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than fa_bwd_workspace_size() */
  FA_ERR_SCRATCH_LIMIT = -6 /* fa_bwd_noalloc: problem larger than FA_NOALLOC_SCRATCH_BYTES */
} fa_status;

/*
 * Forward pass.
 *   q, k, v   device bf16 [B, H, N, d], read only.
 *   o         device bf16 [B, H, N, d], written.
 *   lse       device fp32 [B, H, N], written (natural log; -inf for empty rows).
 *   B, H, N   batch, heads, sequence length (>= 1); d in {64, 128}.
 *   scale     softmax scale (> 0, finite), usually 1/sqrt(d).
 *   causal    0 or 1.
 *   kv_lens   device int32 [B] of valid key counts, or NULL for N. Values are
 *             clamped to [0, N] on the device (check mode rejects them on the
 *             host after a copy).
 *   stream    cudaStream_t.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, const int* kv_lens, void* stream);

/*
 * Forward pass over a packed batch of variable-length sequences.
 * Sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key
 * rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 (lengths Lq_b, Lk_b may differ;
 * 0 allowed). With causal = 1 the mask is bottom-right aligned: query i of a
 * sequence sees key c iff c <= i + Lk_b - Lq_b, so the last query sees every
 * key (for Lq = Lk this is the ordinary causal mask); queries that see no key
 * get O = 0 and LSE = -inf. This generalises the per-batch key lengths of
 * the forward loop's "apply mask if causal or padding" ("FlashAttention算法详解：
 * 从IO瓶颈到Triton实现", §FlashAttention Forward流程) to packed batches.
 *   q, o         device bf16 [total_q, H, d] (row-major, d fastest).
 *   k, v         device bf16 [total_k, H, d].
 *   lse          device fp32 [H, total_q], natural log.
 *   cu_seqlens_* device int32 [batch + 1], non-decreasing, [0] = 0, [batch] =
 *                total; check mode (FA_CHECK=1) validates them on the host.
 *   max_seqlen_* bounds of the sequence lengths (the grid is sized by
 *                max_seqlen_q; a larger value only adds idle CTAs).
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int batch, int H, int d, int total_q, int total_k, int max_seqlen_q,
                  int max_seqlen_k, float scale, int causal, void* stream);

/*
 * Bytes of device workspace every backward entry point needs: rowsum(dO o O)
 * and -LSE*log2(e) as fp32 [B, H, Np] each, an fp32 [B, H, Np, d] dQ
 * accumulator and, for the deterministic order, one 32-bit counter per
 * 128-row block and a ticket counter, where Np is N rounded up to a multiple
 * of 128. 0 on bad sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass (same shapes, masks and scale as the forward that produced
 * o and lse).
 *   q, k, v, o, dO   device bf16 [B, H, N, d], read only.
 *   lse              device fp32 [B, H, N] from fa_fwd, read only.
 *   dq, dk, dv       device bf16 [B, H, N, d], written.
 *   workspace        device, >= fa_bwd_workspace_size(B, H, N, d) bytes,
 *                    16-byte aligned, caller-owned; contents on entry are
 *                    ignored (it is cleared on the stream).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
           const int* kv_lens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass that allocates nothing, for callers that cannot allocate
 * device memory when they need the backward (for example code running inside
 * a memory-pool or allocator callback, or a framework whose device memory is
 * owned by another component, so that neither cudaMalloc nor a caching
 * allocator may be called). The pages have no counterpart: this is a service
 * of the library, not part of the method.
 *
 * Same arguments and results as fa_bwd, minus the workspace: the workspace is
 * a fixed array of FA_NOALLOC_SCRATCH_BYTES (64 MiB) in the library's own
 * static device memory, which every GPU that loads the library reserves until
 * the process exits. Problems with fa_bwd_workspace_size(B, H, N, d) above
 * that size are rejected with FA_ERR_SCRATCH_LIMIT before anything runs
 * (d = 128: B*H*ceil(N/128)*128 up to about 129,000 rows; d = 64: about 254,000).
 * The first call on a device is a set-up: with that device current it looks
 * up the array's device address (cached per device and context; a context
 * torn down and recreated, e.g. by cudaDeviceReset, repeats the set-up).
 * Under lazy module loading that first call may also load the library's
 * kernels on that device, and loading reserves the array's
 * FA_NOALLOC_SCRATCH_BYTES of device memory then: make the first call on
 * each device outside any allocator callback and before any stream capture.
 * Later calls allocate nothing. Every call uses the same array and leaves its
 * contents behind; each call clears what must start at zero itself. Calls
 * that overlap on the GPU (for example on two streams) race on the array:
 * serialise them, e.g. by issuing them on one stream.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                   int causal, const int* kv_lens, void* stream);

/*
 * Backward pass over a packed batch of variable-length sequences: the
 * gradients of sum(O * dO) for the forward of fa_fwd_varlen with the same
 * arguments (same packing, bottom-right causal mask and scale).
 *   q, o, dO, dq   device bf16 [total_q, H, d];  k, v, dk, dv  [total_k, H, d].
 *   lse            device fp32 [H, total_q] from fa_fwd_varlen.
 *   workspace      >= fa_bwd_workspace_size(batch, H, max_seqlen_q, d) bytes.
 * dK and dV rows of keys that no query sees are written as zero.
 */
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int H,
                  int d, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, float scale, int causal,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Deterministic backward ("FlashAttention算法详解", 实际使用建议: a
 * deterministic backward may cost speed). fa_bwd and fa_bwd_varlen add the
 * per-key-block shares of each dQ block into an fp32 accumulator in whatever
 * order the blocks finish, so dQ can differ in its last bits from run to
 * run. These entry points add the shares of every dQ block in ascending
 * key-block order instead, so dQ, dK and dV are bitwise the same on every
 * run with the same inputs, shapes and GPU model (they may differ in the last
 * bits from fa_bwd's results, which are equally accurate). Arguments, layout,
 * workspace (same size), ownership and errors are those of fa_bwd and
 * fa_bwd_varlen. Two calls must not share a workspace at the same time.
 */
int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, const int* kv_lens, void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_varlen_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dO, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                                const int* cu_seqlens_k, int batch, int H, int d, int total_q, int total_k,
                                int max_seqlen_q, int max_seqlen_k, float scale, int causal, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * One decoding step over a paged KV cache ("FlashAttention 完整解析", §7.2-7.4:
 * KV cache pages found through a block table). Sequence b has seq_lens[b]
 * cached tokens; token t sits in slot t % block_size of physical block
 * block_table[b * max_blocks_per_seq + t / block_size]. The one new query of
 * each (sequence, head) attends to all seq_lens[b] cached keys (its own K/V
 * is expected to be in the cache already):
 *   O[b,h] = softmax(scale * q[b,h] . K^T) V,  LSE[b,h] = log-sum-exp (natural log).
 *   q, o           device bf16 [B, H, d].
 *   k_cache, v_cache  device bf16 [num_blocks, block_size, H, d] (the pool).
 *   lse            device fp32 [B, H]; -inf and O = 0 for a sequence with no keys.
 *   block_table    device int32 [B, max_blocks_per_seq]; entries past a
 *                  sequence's last page are not read.
 *   seq_lens       device int32 [B], each in [0, max_seq_len].
 *   block_size     a multiple of 64; max_seq_len <= max_blocks_per_seq * block_size.
 *   workspace      >= fa_decode_workspace_size(B, H, d, max_seq_len) bytes
 *                  (may be NULL when that size's split count is 1), caller-owned.
 * Scores, softmax and the weighted sum of V run in fp32. seq_lens and the
 * table are checked on the host only in check mode (FA_CHECK=1); otherwise
 * lengths are clamped to [0, max_seq_len] on the device and block ids outside
 * [0, num_blocks) read as zero keys and values. Errors as for fa_fwd, plus
 * FA_ERR_UNSUPPORTED for a block size that is not a multiple of 64 or a pool
 * of 2^31 or more token slots, FA_ERR_WORKSPACE for a missing workspace.
 */
size_t fa_decode_workspace_size(int B, int H, int d, int max_seq_len);
int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    const int* block_table, const int* seq_lens, int B, int H, int d, int num_blocks,
                    int block_size, int max_blocks_per_seq, int max_seq_len, float scale, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * FP8 (E4M3) block quantisation ("flash_attention.zh" §9.2: block
 * quantisation, one scale factor per block; "FlashAttention 完整解析" §5.5:
 * E4M3, range +-448). For every 128-row block of every (b, h) slice of the
 * bf16 tensor x [B, H, N, d]: s = amax / 448 (fp32; 0 for an all-zero block)
 * and codes e4m3(x * (448 / amax)) (fp32 product, round to nearest even,
 * saturating at +-448), so x ~ code * s.
 *   out          device uint8: [B, H, N, d], or [B, H, d, Np] with
 *                Np = N rounded up to 128 when `transpose` (keys contiguous,
 *                padding columns 0: the layout fa_fwd_fp8 takes for V).
 *   block_scale  device fp32 [B, H, ceil(N / 128)].
 * Errors: FA_ERR_INVALID / FA_ERR_UNSUPPORTED as for fa_fwd (B * H <= 65535).
 */
int fa_quantize_fp8(const void* x, void* out, float* block_scale, int B, int H, int N, int d, int transpose,
                    void* stream);

/*
 * FP8 forward: the attention of the dequantised inputs (code * block scale),
 * computed with E4M3 tensor-core products ("flash_attention.zh" §9.2;
 * "FlashAttention 完整解析" §5.5). The probabilities are rounded to E4M3 for
 * the P.V product after scaling by 2^7 * sV_block / max sV (no underflow of
 * the largest terms, no saturation); softmax statistics, accumulators and O's
 * normalisation stay in fp32.
 *   q8, k8          device uint8 E4M3 [B, H, N, d] (fa_quantize_fp8, transpose 0).
 *   v8t             device uint8 E4M3 [B, H, d, Np] (fa_quantize_fp8, transpose 1).
 *   q/k/v_scale     device fp32 [B, H, ceil(N / 128)].
 *   o, lse, kv_lens, scale, causal: as for fa_fwd (O bf16, LSE natural log).
 * Only d = 128 (FA_ERR_UNSUPPORTED otherwise).
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
               const int* kv_lens, void* stream);

/* Synchronise `stream`, then read and clear the kernels' device status word:
 * FA_OK, FA_ERR_TIMEOUT, or FA_ERR_LAUNCH for a CUDA error. */
int fa_check_status(void* stream);

/* Static string for an fa_status value. */
const char* fa_status_string(int status);

/* Static string of the last CUDA error seen by this library in this thread. */
const char* fa_last_cuda_error(void);

/*
 * Kernel timing, for benchmarks. Not part of the attention operation itself.
 * fa_timing_begin(n) creates CUDA events (host objects, no device memory) for
 * up to n calls of each kernel; while it is active, fa_fwd and fa_bwd record
 * an event pair on the call's stream around each kernel they launch.
 * fa_timing_read(kind, &ms, &count) waits for the recorded events and returns
 * the summed elapsed time (ms) and the number of timed launches of one kernel:
 * kind 0 = forward, 1 = backward pre-pass, 2 = backward main kernel,
 * 3 = backward dQ conversion. fa_timing_end() releases the events; calls made
 * after n launches of a kind are no longer timed. Returns fa_status.
 */
int fa_timing_begin(int max_calls);
int fa_timing_read(int kind, double* total_ms, int* count);
int fa_timing_end(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

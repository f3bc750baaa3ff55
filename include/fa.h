/*
 * fa.h - exact attention (forward and backward) for NVIDIA GB300 (sm_103).
 *
 * Computes O = softmax(scale * Q K^T [+ causal mask]) V by streaming key/value
 * tiles through shared memory with an online softmax (running row max m and
 * running row sum l), so the N x N score matrix never reaches device memory.
 * The forward stores O and the per-row logsumexp; the backward recomputes the
 * scores from that logsumexp to produce dQ, dK and dV.
 *
 * Sources: the definition softmax(Q K^T / sqrt(d_k)) V ("FlashAttention v2相比
 * 于v1有哪些更新", section 1); tiled online softmax ("FlashAttention技术解析",
 * sections 2.1-2.2); deferred division by l (blogweb.cn page, section 3);
 * recompute-from-normaliser backward ("4.3 FlashAttention-2与FlashAttention-3
 * 演进", FlashAttention-3 section 3); causal block skipping and atomic dQ
 * accumulation ("Flash Attention V3技术解析", section 2.1).
 *
 * Conventions shared by every call
 *   Layout: dense row-major, no strides. Q, O, dO, dQ are [B, Hq, N, d];
 *     K, V, dK, dV are [B, Hkv, N, d]; LSE is [B, Hq, N] fp32. Query head h
 *     reads key/value head h / (Hq / Hkv) (grouped-query attention).
 *   Causal: key j is visible to query i iff j <= i (one N for queries and
 *     keys; fa_fwd_kv / fa_bwd_kv extend the rule to other key lengths).
 *   LSE_i = ln sum_j exp(scale * q_i . k_j) over the visible keys.
 *   Pointers: device pointers, 16-byte aligned, owned by the caller; the
 *     library never allocates or frees memory during a call and keeps no
 *     reference after it returns.
 *   Sizes: B, Hq, Hkv, N >= 1; Hq % Hkv == 0; d a multiple of 8 from 8 to
 *     256 (kernels are built for d = 64, 128, 192 and 256; any other d runs
 *     in the next larger one, the extra columns read as zeros and never
 *     written); scale finite and > 0. The forward calls take every such d
 *     (fa_fwd_f32 and fa_fwd_blocksparse excepted, see there); the backward
 *     calls stop at d = 128 and return FA_ERR_UNSUPPORTED for 136..256, since
 *     the dK, dV, S^T and dP^T accumulators of a 128-key tile (4 d columns)
 *     must fit the 512 TMEM columns. FlashAttention-2 raised the supported
 *     head dimension from 128 to 256 ("Flash Attention-2", section
 *     "Снижение накладных расходов").
 *   stream: a cudaStream_t (NULL = legacy default stream). Every call is
 *     asynchronous on it; argument errors are reported synchronously and
 *     launch nothing.
 *   Device: the current CUDA device must be compute capability 10.3.
 *   Errors: FA_ERR_INVALID_ARG for bad pointers or sizes, FA_ERR_UNSUPPORTED
 *     for a valid but unimplemented combination, FA_ERR_ARCH for a device that
 *     is not sm_103, FA_ERR_CUDA when a launch fails. Inside the kernels every
 *     wait is bounded (2 s, or FA_WAIT_LIMIT_MS milliseconds from the
 *     environment, read once per process); a wait that runs out makes its
 *     block unwind, store nothing and set the status word of the call's
 *     stream, which fa_device_status reports as FA_ERR_TIMEOUT; the context
 *     stays usable.
 *     FA_TEST_STALL=1 in the environment (read at every call) makes the
 *     tensor-core issuer of every fa_fwd* call (fa_fwd_fp8* included) and of
 *     fa_bwd's dK/dV pass wait on a barrier nothing arrives on, to exercise
 *     that path; unset in normal use.
 *   Threads: calls may come from several host threads; each call is
 *     independent, and device-side failures are reported per stream (see
 *     fa_device_status).
 *   CUDA graphs: every call can be captured on a stream and replayed (launch
 *     parameters, tensor maps included, are passed by value; nothing is
 *     allocated). Make one ordinary call on the device first: it does the
 *     one-time set-up (architecture check, device addresses of the status
 *     words), which is not meant to run inside a capture. A replay reads and
 *     writes the captured buffers as they are at replay time.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_ARCH = 3,
  FA_ERR_CUDA = 4,
  FA_ERR_TIMEOUT = 5,
  FA_ERR_WORKSPACE = 6,
  FA_ERR_DEVICE = 7
} fa_status;

/* Forward, bf16. q, k, v, o: bf16; lse: fp32 [B, Hq, N].
 * O_i = sum_j softmax_j(scale q_i . k_j) v_j (fp32 accumulation, bf16 result,
 * round to nearest even); lse as defined above. Tensor-core bf16 MMA with fp32
 * accumulation; the probabilities are rounded to bf16 before the P V product. */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);

/* Forward with keys of another length than the queries, bf16: q, o
 * [B, Hq, Nq, d], k, v [B, Hkv, Nk, d], lse [B, Hq, Nq]. The queries are the
 * last Nq of Nk positions (a chunk of a longer sequence whose earlier keys are
 * cached): when causal, key j is visible to query i iff j <= i + (Nk - Nq)
 * (bottom-right alignment; Nq == Nk is fa_fwd's rule). With Nq > Nk the first
 * Nq - Nk query rows see no key and get O = 0, lse = -inf. No page treats
 * unequal lengths; this is the plainest extension of the causal rule.
 * Errors as fa_fwd (FA_ERR_INVALID_ARG also for Nk < 1). */
fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale, void* stream);

/* fa_fwd_kv computed by clusters of two CTAs whose matrix products run as
 * tcgen05 cta_group::2 pairs (M = 256 over two SMs; each CTA loads half of
 * every K and V tile). Same arguments, layouts, masking and results as
 * fa_fwd_kv (bit for bit on this GPU: each row's products and softmax are
 * the same operations in the same order); bf16 only, 64 < d <= 128, no block
 * mask (FA_ERR_UNSUPPORTED otherwise). Slower than fa_fwd_kv on GB300 (one
 * issuing thread must still start an MMA every 64 cycles to keep both SMs
 * busy, and every hand-off gains a cross-CTA step), so fa_fwd and fa_fwd_kv
 * do not use it; it is kept as the measured pair form. No counterpart on the
 * pages beyond the forward itself ("FlashAttention技术解析" 2.1-2.2). */
fa_status fa_fwd_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int Nq, int Nk, int d, int causal, float scale, void* stream);


/* Forward with a block mask, bf16 ("FlashAttention技术解析", section 6.2: whole
 * blocks are skipped, as the causal mask skips the blocks above the diagonal).
 * Same arguments and outputs as fa_fwd, plus a block mask over 128 x 128 tiles:
 *   block_mask  device bytes; byte (b, h, i, j) at
 *               block_mask[b * mask_stride_b + h * mask_stride_h + i * T + j],
 *               T = ceil(N / 128), h the query head; nonzero = query tile i may
 *               see key tile j. Strides are in bytes and may be 0 (one mask
 *               broadcast over batches or heads); caller-owned, read only.
 * Key j is visible to query i iff the (i/128, j/128) byte is nonzero and, when
 * causal, j <= i. Key tiles no query tile of a CTA sees are never loaded or
 * multiplied. A query row that sees no key gets O = 0 and lse = -inf.
 * FA_ERR_INVALID_ARG for a null mask or negative strides; FA_ERR_UNSUPPORTED
 * for N > 131072 or d > 128. */
fa_status fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                             const unsigned char* block_mask, long long mask_stride_b, long long mask_stride_h,
                             int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);

/* Forward, fp32 in and out (tf32 tensor-core products, fp32 softmax and
 * accumulation). Same arguments as fa_fwd with fp32 q, k, v, o; d must be 64
 * (FA_ERR_UNSUPPORTED otherwise). */
fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                     int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);

/* FP8 forward (e4m3 inputs with block scales), d a multiple of 16 from 16 to
 * 256 (a row of one-byte codes must be a multiple of 16 bytes for TMA; d up to
 * 128 runs in the d = 128 kernel and above it in the d = 256 one, the columns
 * past d read as zeros); other head dimensions return FA_ERR_UNSUPPORTED, from
 * the quantisers and the forwards alike.
 * Source: "Flash Attention V3技术解析", section 1.3 (FP8 operands need the
 * contracted dimension contiguous, so P V reads V transposed; block-wise
 * quantisation) and section 3.2 (each block's scale from its largest
 * magnitude); "4.3 FlashAttention-2与FlashAttention-3演进", FlashAttention-3
 * section 2. Codes are e4m3 (largest finite value 448, no infinities);
 * scale = max|block| / 448 in fp32 (1 for an all-zero block); code =
 * e4m3(x / scale), division in fp32, rounded to nearest even, magnitudes
 * past 448 held at 448. A value is code * scale.
 *
 * fa_fp8_row_scales(N): scales per head of a Q or K tensor, ceil(N / 64).
 * fa_fp8_vt_keys(N): key columns of the transposed V codes, N rounded up to
 * 128. Both 0 for N < 1.
 *
 * fa_fp8_quantize_rows: x bf16 [BH, N, d] -> out uint8 codes [BH, N, d] and
 * scales fp32 [BH, fa_fp8_row_scales(N)], one per block of 64 rows over all d
 * columns (used for Q and for K). */
size_t fa_fp8_row_scales(int N);
size_t fa_fp8_vt_keys(int N);
fa_status fa_fp8_quantize_rows(const void* x, void* out, float* scales, int BH, int N, int d, void* stream);

/* fa_fp8_quantize_v: v bf16 [BH, N, d] -> vt uint8 codes [BH, d, NP]
 * (NP = fa_fp8_vt_keys(N); row c holds column c of V, keys contiguous, codes
 * 0 past N) and scales fp32 [BH, d], one per column over all N keys. The
 * scales buffer is also the call's scratch (column maxima) until it returns
 * on the stream. Three launches on `stream`. */
fa_status fa_fp8_quantize_v(const void* v, void* vt, float* scales, int BH, int N, int d, void* stream);

/* fa_fwd_fp8: attention of the dequantised inputs, the forward of fa_fwd:
 * q codes [B, Hq, N, d] with q_scale [B, Hq, ceil(N/64)], k codes
 * [B, Hkv, N, d] with k_scale [B, Hkv, ceil(N/64)], vt codes [B, Hkv, d, NP]
 * with v_scale [B, Hkv, d] (as the two calls above write them); o bf16
 * [B, Hq, N, d], lse fp32 [B, Hq, N]. The products run on e4m3 tensor cores
 * with fp32 accumulation. Contract on the probabilities: each P_ij is taken
 * relative to a reference no larger than the row's true running maximum
 * (this library lets it trail by up to a factor 2^4), scaled by a power of two
 * >= 1 (this library: 2^4) and rounded to the nearest e4m3 value below 448
 * before the P V product; the row sum and the LSE use the unrounded values.
 * With P_ij = exp(s_ij - max_j s_ij) and l_i = sum_j P_ij, the result then
 * differs from the exact attention of the dequantised inputs by at most
 * 2^-4 sum_j (P_ij / l_i)|V_jc| + 2^-10 sum_j |V_jc| / l_i per element
 * (visible keys j; e4m3's relative and subnormal rounding), plus the bf16
 * rounding of O, and the errors are unbiased to first order (round to
 * nearest). The tests also hold the mean error to its expectation under
 * independent roundings. FA_ERR_UNSUPPORTED for d not a multiple of 16. */
fa_status fa_fwd_fp8(const void* q, const float* q_scale, const void* k, const float* k_scale, const void* vt,
                     const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int N, int d, int causal,
                     float scale, void* stream);

/* fa_fwd_fp8 with keys of another length than the queries, as fa_fwd_kv:
 * q codes [B, Hq, Nq, d] and q_scale [B, Hq, ceil(Nq/64)]; k codes
 * [B, Hkv, Nk, d], k_scale [B, Hkv, ceil(Nk/64)], vt codes [B, Hkv, d, NPk]
 * (NPk = fa_fp8_vt_keys(Nk)) and v_scale [B, Hkv, d] (quantised with N = Nk);
 * o [B, Hq, Nq, d], lse [B, Hq, Nq]. The queries are the last Nq of Nk
 * positions: when causal, key j is visible to query i iff j <= i + (Nk - Nq);
 * rows that see no key get O = 0, lse = -inf. Same bound as fa_fwd_fp8. */
fa_status fa_fwd_fp8_kv(const void* q, const float* q_scale, const void* k, const float* k_scale, const void* vt,
                        const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                        int causal, float scale, void* stream);

/* Bytes of device workspace fa_bwd needs: fp32 LSE * log2(e) and fp32
 * D = rowsum(dO * O), each [B, Hq, ceil(N/128)*128], and the fp32 dQ
 * accumulator [B, Hq, N, d], each part 256-byte aligned. Returns 0 for invalid
 * sizes. */
size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d);

/* Backward, bf16. Inputs q, k, v, o, dO (bf16) and lse (fp32) from fa_fwd with
 * the same sizes, causal flag and scale. Outputs dq [B, Hq, N, d] and dk, dv
 * [B, Hkv, N, d] (bf16) are overwritten. workspace: caller-owned device
 * memory of at least fa_bwd_workspace_bytes(...) bytes, 256-byte aligned
 * (FA_ERR_WORKSPACE if too small); its contents need not be initialised and
 * are scratch after the call. dK and dV are deterministic; dQ is accumulated
 * with fp32 atomics, so its last bits may vary from run to run. */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                 int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);

/* Backward with bit-reproducible results: the same arguments as fa_bwd and
 * the same results within rounding, but dQ, dK and dV come out with the same
 * bits on every run. dQ is computed in a pass of its own over the key tiles
 * instead of accumulated across key tiles with reduce-adds, which costs about
 * 40% more tensor-core work. The workspace only needs its LSE and D parts:
 * 2 * B * Hq * ceil(N/128)*128 * 4 bytes, each half 256-byte aligned (any
 * size fa_bwd_workspace_bytes returns is enough). */
fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dO, void* dq, void* dk, void* dv, void* workspace,
                               size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, int causal,
                               float scale, void* stream);

/* Backward of fa_fwd_kv (same shapes, same visibility rule; o and lse from
 * fa_fwd_kv): dq [B, Hq, Nq, d], dk, dv [B, Hkv, Nk, d]. The workspace is
 * fa_bwd_workspace_bytes(B, Hq, Hkv, Nq, d) bytes (it scales with the
 * queries). Gradients of rows that see no key are zero. Errors as fa_bwd. */
fa_status fa_bwd_kv(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale, void* stream);

/* Backward with the same block mask as fa_fwd_blocksparse (same layout, same
 * visibility rule), bf16; the forward's O and lse must come from
 * fa_fwd_blocksparse with that mask. Outputs and numerics as fa_bwd; a (query
 * tile, key tile) pair the mask hides costs nothing, and gradients of rows that
 * see no key are zero. The workspace must hold
 * fa_bwd_blocksparse_workspace_bytes(B, Hq, Hkv, N, d) bytes (fa_bwd's parts
 * plus each dK/dV block's list of visible query steps), 256-byte aligned,
 * caller-owned, scratch after the call. FA_ERR_INVALID_ARG for a null mask or
 * negative strides, FA_ERR_WORKSPACE for a short or misaligned workspace,
 * FA_ERR_UNSUPPORTED for N > 131072. */
size_t fa_bwd_blocksparse_workspace_bytes(int B, int Hq, int Hkv, int N, int d);
fa_status fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             const unsigned char* block_mask, long long mask_stride_b, long long mask_stride_h,
                             int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);

/* The three phases fa_bwd runs, in this order on one stream, exposed for
 * callers that schedule or time them separately. Arguments mean what they
 * mean for fa_bwd; the workspace carries state from one phase to the next.
 *   fa_bwd_preprocess: D_i = sum_c dO_ic O_ic and LSE_i log2(e) into the
 *     workspace, and the dQ accumulator zeroed.
 *   fa_bwd_dkdv: dK and dV (written to dk, dv) and the unscaled fp32 dQ
 *     accumulator (in the workspace); the tensor-core phase.
 *   fa_bwd_dq: dq = scale * accumulator, rounded to bf16. */
fa_status fa_bwd_preprocess(const void* o, const float* lse, const void* dO, void* workspace,
                            size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, void* stream);
fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv,
                      void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d,
                      int causal, float scale, void* stream);
fa_status fa_bwd_dq(void* dq, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d,
                    float scale, void* stream);

/* Backward without a caller-provided workspace, for callers that cannot
 * allocate device memory when they call it (a plugin that only receives
 * fixed buffers from its host framework, a component that does not own the
 * device memory pool, a loop that cannot afford cudaMalloc's implicit device
 * synchronisation). The pages have no counterpart: this is a convenience of
 * this library. Arguments and results are those of fa_bwd minus the
 * workspace, which lives instead in a 32 MiB array of device memory owned by
 * the library (held on every device that loads it until the process exits).
 * Returns FA_ERR_WORKSPACE, launching nothing, when the problem needs more
 * than 32 MiB of scratch (fa_bwd_workspace_bytes > 33554432). The first call
 * on a device looks up the array's device address; make that first call
 * before any stream capture. Only a successful lookup is kept: if it fails
 * (FA_ERR_CUDA), the next call tries again. Allocates nothing. All calls share the one
 * array: calls whose work overlaps on the GPU (other streams, other host
 * threads on the same device) race and corrupt each other's results. */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                         int causal, float scale, void* stream);

/* Synchronises `stream`, then returns and clears the status word of that
 * stream: FA_OK, FA_ERR_TIMEOUT (a bounded wait inside a kernel ran out; that
 * call's outputs are invalid), FA_ERR_DEVICE (a kernel found the device's
 * shared-memory window unusable and did nothing) or FA_ERR_CUDA (the stream
 * reported an error). Each stream handle has its own word on each device,
 * set only by calls launched on that stream, so a failure on one stream is
 * neither reported to nor cleared by a caller that asks about another. The
 * first 255 stream handles a device sees get a word each; later ones share
 * one word (and so do threads that all pass cudaStreamPerThread, one handle
 * value). Calls on other streams are neither waited for nor reported. */
fa_status fa_device_status(void* stream);

/* Diagnostic: the mean SM clock, in MHz, of the forward (fa_fwd, fa_fwd_f32,
 * fa_fwd_kv, fa_fwd_blocksparse at d <= 128) and dK/dV (fa_bwd and its
 * variants) kernels launched on this device since the previous call, as
 * measured by the kernels themselves: each block adds the SM cycle count and
 * the nanoseconds between its start and its exit to two device-wide sums,
 * and *mhz = cycles / ns * 1000 (0 when no such kernel ran). Synchronises
 * the device, then resets the sums. Calls from several host threads or on
 * several streams share the sums. FA_ERR_INVALID_ARG for a null pointer.
 * No counterpart on the pages: it attributes a measured time to the clock it
 * ran at. */
fa_status fa_sm_clock_mhz(double* mhz, void* stream);

/* Diagnostic: throughput of the exponential instruction the softmax uses
 * (ex2.approx), measured on the current device, for the exponential ceiling
 * of the forward (one exponential per 4 d floating-point operations).
 * Source: "FlashAttention v2相比于v1有哪些更新", sections 2 and 3 ("CUDA
 * Core vs. Tensor Core": work off the matrix units runs up to 16 times
 * slower than on them).
 * Every SM runs 512 threads of eight independent ex2 chains for 4096 steps
 * (about half a millisecond); *per_sm_per_cycle receives the mean over SMs
 * of ex2 results per SM clock cycle. Synchronises `stream`. Allocates
 * nothing: the per-SM cycle counts go to a static device array, so calls that
 * overlap on the GPU race. FA_ERR_INVALID_ARG for a null pointer,
 * FA_ERR_UNSUPPORTED for more than 1024 SMs. */
fa_status fa_ex2_throughput(double* per_sm_per_cycle, void* stream);

/* Static description of a status code. */
const char* fa_status_string(fa_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

/*
 * attn.h -- C ABI of libattn.so: fused exact scaled-dot-product attention on GB300
 * (sm_103a), forward and backward.
 *
 * The operation ("Algorithm analysis" page, section 4; "FlashAttention-4 explained"
 * page, section 01: attention is two matrix products around a softmax):
 *
 *     S = scale * Q K^T          (causal: S_ij = -inf for key j > query i)
 *     P = softmax(S) row-wise
 *     O = P V,   LSE_i = ln sum_j exp(S_ij)
 *
 * computed tile by tile so that S and P never reach device memory.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are device pointers to contiguous row-major bf16 (__nv_bfloat16 bit
 *    patterns) unless stated otherwise.  Shapes: Q, O, dO, dQ are [B, Hq, N, d];
 *    K, V, dK, dV are [B, Hkv, N, d].  LSE is fp32 [B, Hq, N].
 *  - Grouped heads (GQA/MQA): Hq must be a multiple of Hkv; query head h reads
 *    key/value head h / (Hq / Hkv).
 *  - Head dim d: each entry point states the values it takes (64 and 128 everywhere;
 *    the forward entry points also 192 and 256).  N >= 0, B >= 0 (either being 0 is a
 *    no-op returning 0).  Any N >= 1 is supported (a ragged last tile is masked).
 *  - Every tensor pointer must be 16-byte aligned (TMA requirement).
 *  - scale > 0 (the usual choice is 1/sqrt(d)).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous:
 *    they enqueue kernels and return.  The caller owns every buffer and the stream; the
 *    library allocates no device memory on any call.
 *  - Return value: ATTN_OK (0) or a negative attn_status.  On error nothing was
 *    launched and attn_last_error() holds a message (thread-local).
 *  - Kernels never trap.  Every wait inside a kernel is bounded; a kernel that gives
 *    up sets a device status word and returns, leaving its outputs undefined.  Read
 *    (and clear) that word with attn_device_status().
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1, /* bad shape, null pointer, bad scale */
  ATTN_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. a head dim the call lacks) */
  ATTN_ERR_MISALIGNED = -3,  /* a pointer is not 16-byte aligned */
  ATTN_ERR_WORKSPACE = -4,   /* backward workspace missing or too small */
  ATTN_ERR_CUDA = -5,        /* a CUDA runtime call failed (message has the name) */
  ATTN_ERR_TIMEOUT = -6      /* a kernel gave up on a bounded wait */
} attn_status;

/*
 * Forward pass.  FlashAttention-4 forward pipeline: "Hotelren FA4 summary" page,
 * section 3 (two query tiles per CTA, softmax and correction warpgroups, conditional
 * rescale with tau = 8 in log2 units, exponentials split between MUFU and an FMA
 * polynomial); "Algorithm analysis" page, section 4 (tiled online softmax).
 *
 *   q   [B,Hq,N,d] bf16, in      k, v [B,Hkv,N,d] bf16, in
 *   o   [B,Hq,N,d] bf16, out     lse  [B,Hq,N] fp32, out: ln sum_j exp(S_ij)
 *   d:      64, 128, 192 or 256.  For 192 and 256 (up to the 256 of "Hotelren FA4
 *           summary" section 6.2, item 1) the two tiles' accumulators do not fit tensor
 *           memory, so a CTA takes one query tile and overlaps the softmax of one key
 *           block with the products of the next.  The backward: 64 and 128.
 *   causal: 0 or 1 (key j visible to query i only if j <= i)
 *   scale:  softmax scale applied to Q K^T
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
             int d, int causal, float scale, void* stream);

/*
 * Forward for Nq queries appended after a cache of Nk >= Nq keys (chunked prefill or
 * decoding against a key/value cache: the reverse-engineering page, KV-cache inference).
 * Query i stands at key position i + Nk - Nq; with causal it sees keys j <= i + Nk - Nq
 * (the mask aligned at the bottom-right corner; Nq = Nk is attn_fwd).
 *
 *   q, o [B,Hq,Nq,d] bf16; k, v [B,Hkv,Nk,d] bf16; lse [B,Hq,Nq] fp32; other arguments
 *       and ownership as attn_fwd.
 *   workspace: device memory of attn_fwd_kv_workspace_size(...) bytes, 16-byte aligned,
 *       owned by the caller, or NULL.  When the g = Hq/Hkv query heads of a group times Nq
 *       fit one 128-row tile (g >= 2, g * Nq <= 128) the call packs them into one tile per
 *       K/V head and splits the keys over several CTAs, which needs the workspace for the
 *       partial results; without it (NULL or too small) the ordinary tiling is used, with
 *       the same results.
 * Errors as attn_fwd, plus ATTN_ERR_INVALID_ARG when Nk = 0 < Nq or when causal and
 * Nq > Nk (the first queries would see no key).
 */
int attn_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                int Nk, int d, int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 inputs ("Hotelren FA4 summary" page, section 6.3, future directions: FP8 inputs; the
 * reverse-engineering page's FP8 path).  The pages fix neither the format nor the scaling;
 * this library reads them as e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * largest value 448, no infinities) with one fp32 scale per block of 128 consecutive rows
 * of one head: the value of an element is decode(code) * scale of its block.
 *
 * attn_quantize_fp8: x [B,H,N,d] bf16 in -> x8 [B,H,N,d] e4m3 codes (one byte each) and
 *   scales [B,H,ceil(N/128)] fp32 out.  Per block: amax = max |x|, scale = amax / 448 in
 *   fp32 (1 for an all-zero block), code = e4m3(x / scale) rounded to nearest even,
 *   saturating at +-448.  d must be 128.  x and x8 16-byte aligned, scales 4-byte aligned;
 *   all three caller-owned device memory.
 */
int attn_quantize_fp8(const void* x, void* x8, float* scales, int B, int H, int N, int d, void* stream);

/*
 * FP8 forward: O = softmax(scale * Q~ K~^T [causal]) V~ and LSE, where Q~, K~, V~ are the
 * dequantised inputs.  The score product runs on the 8-bit tensor path; P is kept at 16 bits
 * (fp16, times V's block scale) and V is widened exactly to fp16 on chip for O += P V, so the
 * result meets the bf16 forward's error bounds against the exact attention of Q~, K~, V~.
 *
 *   q8 [B,Hq,N,128], k8, v8 [B,Hkv,N,128] e4m3 codes (16-byte aligned);
 *   q_scale [B,Hq,ceil(N/128)], k_scale, v_scale [B,Hkv,ceil(N/128)] fp32, positive
 *       and finite (as attn_quantize_fp8 writes them; 256 * v_scale must stay below
 *       65504, i.e. |V| below about 1.1e5, so that P * v_scale fits fp16 with tau = 8);
 *   o [B,Hq,N,128] bf16, lse [B,Hq,N] fp32 out; d must be 128; other arguments, ownership
 *   and errors as attn_fwd.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                 const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int N, int d, int causal,
                 float scale, void* stream);

/*
 * Bytes of workspace attn_fwd_kv uses for these sizes on the current device (0 when it
 * packs nothing); (size_t)-1 for invalid sizes.
 */
size_t attn_fwd_kv_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d);

/*
 * Forward over B packed sequences of different lengths ("FlashAttention-4 explained"
 * page, section 06: sequences of different lengths, the CTAs with the most work started
 * first).  Each sequence is its own attention problem; sequence b owns query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1,
 * and within it query i stands at key position i + nk - nq as in attn_fwd_kv (causal is
 * aligned at the sequence's bottom-right corner; equal offsets give the usual causal mask).
 *
 *   q, o [Hq, total_q, d] bf16; k, v [Hkv, total_k, d] bf16; lse [Hq, total_q] fp32
 *       (natural log): the sequences one after another along the row axis of each head.
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 arrays of B + 1 offsets, 4-byte aligned:
 *       starting at 0, never decreasing, ending at total_q and total_k; a sequence with
 *       queries must have keys, and with causal at least as many keys as queries.
 *   workspace: device memory of attn_fwd_varlen_workspace_size(...) bytes, 16-byte
 *       aligned, owned by the caller, contents on entry irrelevant (it receives the
 *       order in which the tiles run, built on the device from the offsets).
 *   other arguments and ownership as attn_fwd.
 * Head dims as attn_fwd (64, 128, 192, 256).
 * Errors as attn_fwd, plus ATTN_ERR_WORKSPACE, ATTN_ERR_INVALID_ARG when total_k = 0 <
 * total_q, and ATTN_ERR_UNSUPPORTED for Hq > 65535.  The offsets are checked on the
 * device: if they break a rule above, nothing is written to o and lse and the device
 * status word reads ATTN_ERR_INVALID_ARG (attn_device_status; returned at once when
 * sync_check is set).
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k, int d, int causal,
                    float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace attn_fwd_varlen needs: a bound that depends on B, the heads and
 * total_q only (0 when there is nothing to do); (size_t)-1 for invalid sizes.
 */
size_t attn_fwd_varlen_workspace_size(int B, int Hq, int Hkv, int total_q, int d);

/*
 * Backward over packed sequences: dQ, dK, dV of attn_fwd_varlen's O for the same offsets
 * (the stages of attn_bwd, one sequence at a time; "FlashAttention-4 explained" page,
 * section 06 for the longest-first order of the key blocks).
 *
 *   q, o, dout, dq [Hq, total_q, d] bf16; k, v, dk, dv [Hkv, total_k, d] bf16; lse
 *       [Hq, total_q] fp32 as attn_fwd_varlen wrote it; dq, dk, dv out (overwritten).
 *   cu_seqlens_q, cu_seqlens_k: as attn_fwd_varlen (DEVICE int32, B + 1 entries).  Keys of
 *       a sequence without queries get dk = dv = 0.  With total_q = 0 the query-side
 *       pointers may be NULL.
 *   deterministic: 1 = dQ contributions are added in a fixed order (bit-identical runs).
 *   workspace: device memory of attn_bwd_varlen_workspace_size(...) bytes, 16-byte
 *       aligned, owned by the caller, contents on entry irrelevant.
 * Errors as attn_bwd, plus the device check of the offsets (attn_fwd_varlen).
 */
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                    int Hkv, int total_q, int total_k, int d, int causal, float scale, int deterministic,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace attn_bwd_varlen needs: fp32 dQ accumulator [Hq, total_q + 128 B, d]
 * (each sequence's rows padded to whole 128-row tiles), rowsum(dO o O) and LSE*log2(e)
 * [Hq, total_q], ordering counters when deterministic, and the table of key blocks.  A
 * bound from the sizes alone; 0 when there is nothing to do, (size_t)-1 for invalid sizes.
 */
size_t attn_bwd_varlen_workspace_size(int B, int Hq, int Hkv, int total_q, int total_k, int d, int deterministic);

/*
 * Persistent forward for d = 64 and 128 (ordinary tiling): 1 = one CTA per SM walks the
 * work list, loading the next unit's tiles and starting its products while the current
 * unit ends (fwd_persist.cu); 0 = one CTA per unit (fwd.cu).  Same results bit for bit.
 * Grouped decode, packed sequences and the exponential-split knob keep the per-unit
 * kernel.  A tuning knob, process-wide.
 */
int attn_set_fwd_persistent(int enable);

/*
 * Which forward kernel serves d = 128: 0 = two query tiles per CTA (fwd.cu), 1 = one
 * query tile per CTA with the softmax of each key block split over two warpgroups
 * (fwd_wide.cu, the kernel that always serves d = 192 and 256).  Same results up to the
 * rounding of the row sums; attn_fwd_kv's grouped decode and attn_fwd_varlen keep the
 * two-tile kernel.  A tuning knob, process-wide.
 */
int attn_set_fwd_one_tile(int enable);

/*
 * Query tile of attn_bwd (and attn_bwd_noalloc) for d = 64 and 128: 128 = one 128-key block
 * per CTA walking 128-row query tiles, dQ^T formed in the columns of dP^T (bwd.cu); 64 =
 * 64-row query tiles with dQ^T in tensor-memory columns of its own and the next tile's
 * products issued ahead of this tile's dK and dQ^T (bwd_wide.cu, the kernel that always
 * serves d = 192 and 256).  Same results within the backward's error bounds (the order of
 * the fp32 dQ additions differs).  attn_bwd_workspace_size covers both.  A tuning knob,
 * process-wide; ATTN_ERR_INVALID_ARG for other values.
 */
int attn_set_bwd_query_tile(int rows);

/*
 * Which kernel serves attn_fwd_kv's grouped decode (g * Nq <= 128) at d = 128: 1 (default) =
 * the one-tile kernel (fwd_wide.cu), in which S of the next key block overlaps the softmax of
 * the current one; 0 = the two-tile kernel with its second tile slot empty (fwd.cu).  Same
 * results up to the order of the rounding; d = 64 always uses the two-tile kernel.  A tuning
 * knob, process-wide.
 */
int attn_set_decode_one_tile(int enable);

/*
 * Order of attn_fwd_varlen's tiles and attn_bwd_varlen's key blocks: 1 (default) = the
 * CTAs with the most work first; 0 = no ordering (the order in which the scheduler meets
 * the sequences).  The results are the same either way; the knob exists to measure what
 * the ordering buys.
 */
int attn_set_varlen_order(int longest_first);

/*
 * Bytes of device workspace attn_bwd needs for these sizes (fp32 dQ accumulator
 * [B,Hq,ceil(N/128)*128,d] with each head's rows padded to whole 128-row tiles,
 * rowsum(dO o O) and LSE*log2(e) [B,Hq,N]; when deterministic, ordering counters and,
 * for d <= 128, more fp32 accumulators of the same shape: one when N <= 8064, three for
 * longer sequences).  0 when there is nothing to do.  Returns (size_t)-1 for invalid
 * sizes.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d, int deterministic);

/*
 * Backward pass: dQ, dK, dV of L given dO = dL/dO.  Recomputes P from Q, K and the
 * forward's LSE (reverse-engineering page: backward by recomputation).  Stages follow
 * "Hotelren FA4 summary" page, section 4.2: S = K Q^T, dP = dO V^T, dV = P^T dO,
 * dS = P o (dP - rowsum(dO o O)), dQ += dS K (fp32 accumulation), dK = dS^T Q.
 *
 *   q, k, v, o, lse, dout: the forward's inputs and outputs (o and lse as attn_fwd
 *       wrote them), dout [B,Hq,N,d] bf16.
 *   dq [B,Hq,N,d], dk, dv [B,Hkv,N,d] bf16, out (overwritten, not accumulated into).
 *   deterministic: 1 = dQ contributions are added in a fixed order, so repeated calls
 *       give bit-identical outputs ("FlashAttention-4 explained" page, section 06);
 *       0 = unordered fp32 atomics.
 *   workspace: device memory of at least attn_bwd_workspace_size(...) bytes, 16-byte
 *       aligned, owned by the caller; its contents on entry do not matter.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
             int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass for callers that cannot allocate device memory on the call path: code
 * running inside another runtime's plugin or callback interface (its memory belongs to
 * that runtime's pool) or in a latency-critical loop where cudaMalloc would
 * synchronise the device.  No counterpart on the pages; it exists only for such callers.
 *
 * Same arguments and results as attn_bwd, without the workspace: the library uses its
 * own fixed 64 MiB device array instead (held by every GPU that loads the library until
 * the process exits).  Sizes whose attn_bwd_workspace_size exceeds 64 MiB are rejected
 * with ATTN_ERR_WORKSPACE and a message in attn_last_error().  Nothing is allocated.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current (a failed lookup returns ATTN_ERR_CUDA and is tried again on
 * the next call); make that first call before any stream capture.  All calls
 * share the array and it keeps the last call's contents (the backward clears what must
 * start at zero itself), so calls that overlap on the GPU, e.g. on two streams, race.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                     int causal, float scale, int deterministic, void* stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* attn_last_error(void);

/* Library version string. */
const char* attn_version(void);

/*
 * Tuning and test knobs (process-wide; take effect on the next call):
 *   tau:           conditional-rescale threshold in log2 units (default 8; 0 = rescale
 *                  whenever a row maximum grows).  "Hotelren FA4 summary" section 3.3.
 *   poly_per_16:   exponentials computed by the FMA polynomial, per 16 (0, 4 or 16;
 *                  default 0).  "Hotelren FA4 summary" section 3.2.
 *   wait_limit_ns: bound on any single wait inside a kernel (default 2 s).
 *   sync_check:    1 = each call synchronises its stream and checks the device status
 *                  word (debugging only).
 */
int attn_set_debug_knobs(float tau, int poly_per_16, long long wait_limit_ns, int sync_check);
int attn_get_debug_knobs(float* tau, int* poly_per_16, long long* wait_limit_ns, int* sync_check);

/*
 * Test hook (off by default): skip_first_kv_load = 1 makes the forward's load warp never
 * issue the first K tile of each CTA, so the consumer's bounded wait runs out, the CTA
 * gives up cleanly and the device status word reads ATTN_ERR_TIMEOUT.  Used to test the
 * timeout path without faulting anything.  No counterpart on the pages.
 */
int attn_set_test_hooks(int skip_first_kv_load);

/*
 * Synchronises the current device and reads the device status word: ATTN_OK,
 * ATTN_ERR_TIMEOUT if some kernel gave up on a wait since the last clear, or
 * ATTN_ERR_INVALID_ARG if attn_fwd_varlen's offsets failed their device check.
 * clear = 1 resets the word.
 */
int attn_device_status(int clear);

/*
 * Rescale statistics: synchronises, returns in *value_out the number of (row, key tile)
 * steps after the first tile in which the forward rescaled O (counted only while
 * enabled), resets the count, and enables (1) or disables (0) counting.
 */
int attn_rescale_counter(int enable, unsigned long long* value_out);

/*
 * Software exp2 test entry: y[i] = 2^x[i] for i < n (device fp32 arrays).
 *   variant 0: the FMA-pipe polynomial exactly as the forward uses it;
 *   variant 1: the same polynomial with a correctly rounded subnormal range;
 *   variant 2: the hardware MUFU ex2.approx.ftz.
 * "FlashAttention-4 explained" page, section 04: e^x ~ 2^n (p0 + p1 f + p2 f^2 + p3 f^3).
 */
int attn_exp2_sw(const float* x, float* y, long long n, int variant, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */

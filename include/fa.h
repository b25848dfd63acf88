/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention forward library, libfa.so.
 *
 * What it computes.  Standard attention, exactly: S = scale * Q K^T, P = softmax(S)
 * row by row, O = P V ("FlashAttention面试讲解" interview canvas, element std-text).
 * The tiled method of the same canvas (elements flash-text, formula-text, qa2-a)
 * visits K/V one tile at a time with an online softmax -- a running row maximum m,
 * a running sum l and a rescaled output accumulator -- so the N x N score matrix is
 * never written to memory.  The forward pass also keeps one per-row statistic for a
 * backward pass (elements v1-card-body and qa3-a): here that is the natural-log
 * logsumexp of the scaled scores, LSE_i = ln sum_j exp(S_ij) over the valid keys.
 *
 * Conventions fixed by this library (the pages leave them open):
 *   - causal masks are bottom-right aligned: key j is visible to query i iff
 *     j <= i + (Nk - Nq); with Nq == Nk this is the usual lower triangle;
 *   - a query row that sees no key gets O = 0 and LSE = -inf;
 *   - grouped-query attention: query head h reads key/value head h / (Hq / Hkv);
 *   - P is rounded to bf16 before the P*V product; all accumulation is fp32.
 *
 * Thread safety: every entry point is reentrant.  The library's state is
 * once-initialised per-device launch settings, four device status words (one
 * each for the forward, split-KV, backward and one-launch quantizer kernels,
 * merged by fa_device_status), a per-process cache of the host-built work
 * lists (guarded by a lock), one pair of copy streams per device for
 * fa_fwd_host, and the process-wide settings of the three test hooks
 * (fa_debug_fault_injection, fa_debug_soft_exp, fa_debug_fwd_pair): a hook
 * call changes every later launch, from any thread.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,        /* a required pointer is NULL */
  FA_ERR_SHAPE = 2,       /* negative size, Hkv < 1, Hq % Hkv != 0, or Nq != Nk with cu_seqlens */
  FA_ERR_ALIGN = 3,       /* q, k, v or o not 16-byte aligned, or lse not 4-byte aligned */
  FA_ERR_UNSUPPORTED = 4, /* d not in {64, 128}, or the current device is not sm_103 */
  FA_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed while enqueueing */
  FA_ERR_TIMEOUT = 6,     /* a kernel gave up on a bounded wait (reported by fa_device_status) */
  FA_ERR_VALUE = 7        /* scale is not a finite positive number */
} fa_status;

/*
 * fa_fwd -- exact attention forward, O and LSE, on `stream`.
 *
 * Dense mode (cu_seqlens == NULL), row-major and contiguous:
 *   q   [B, Hq,  Nq, d]  bf16, device      k, v [B, Hkv, Nk, d] bf16, device
 *   o   [B, Hq,  Nq, d]  bf16, device      lse  [B, Hq, Nq]     fp32, device
 * Packed variable-length mode (cu_seqlens != NULL): B sequences are concatenated
 * along the token axis; sequence s owns tokens [cu_seqlens[s], cu_seqlens[s+1]):
 *   q, o [Hq, Nq, d], k, v [Hkv, Nq, d], lse [Hq, Nq], with Nq == Nk == total tokens.
 *   cu_seqlens is an int32 device array of B+1 non-decreasing offsets, cu_seqlens[0]
 *   == 0 and cu_seqlens[B] == Nq.  Queries attend only to keys of their own sequence
 *   (the causal mask is applied per sequence).  Offsets are clamped to [0, Nq] on the
 *   device, so malformed offsets give wrong results but never out-of-range accesses.
 *
 * scale: the factor applied to Q K^T, finite and > 0 (usually 1/sqrt(d)).
 * causal: 0 or 1.
 * d: 64 or 128.
 *
 * Ownership: the caller owns every buffer; the library allocates no device
 * memory.  The call is asynchronous: it validates arguments on the host,
 * enqueues one kernel on `stream` and returns.  Inputs must stay valid and
 * outputs untouched until the stream reaches that point.
 *
 * Empty problems (B, Hq or Nq equal to 0) return FA_OK and launch nothing.
 * With Nk == 0 every row is written as O = 0, LSE = -inf (k and v may be NULL).
 *
 * Errors: FA_ERR_NULL / SHAPE / ALIGN / UNSUPPORTED / VALUE are detected before
 * anything is enqueued and leave the outputs untouched.  FA_ERR_CUDA reports a
 * failed launch.  Device-side time-outs are recorded in the status word read by
 * fa_device_status().
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                 const int32_t* cu_seqlens, cudaStream_t stream);

/*
 * fa_decode -- the same computation as fa_fwd (dense layout only) by the
 * split-KV path for few query rows per key/value head: it requires
 * (Hq / Hkv) * Nq <= 16 and Nk >= 1, and returns FA_ERR_UNSUPPORTED otherwise.
 * fa_fwd itself takes this path for such dense problems.  Work is bound by
 * reading K and V once from HBM, since every new token reads all earlier
 * tokens' K/V (KV-cache overview canvas, element text-0023).  One thread-block
 * cluster per (batch, key/value head) splits the keys over up to 8 CTAs.
 * Their partial (max, sum, output)
 * states are merged through distributed shared memory (m* = max m_s,
 * l* = sum l_s e^(m_s - m*), O* = sum O_s e^(m_s - m*) / l*), so no scratch
 * memory is used.  Arguments, layouts, ownership and errors are as for
 * fa_fwd; the call is asynchronous on `stream`.
 */
fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                    cudaStream_t stream);

/*
 * fa_bwd -- gradients of the attention forward (dense layout), on `stream`.
 *
 * The forward pass keeps only O and the per-row LSE; this call recomputes the
 * scores and probabilities tile by tile from them instead of reading a stored
 * N x N matrix ("FlashAttention面试讲解" interview canvas, elements
 * v1-card-body and qa3-a).  With P = exp(scale Q K^T - LSE) (masked entries 0):
 *   dV = P^T dO,  dP = dO V^T,  delta_i = dO_i . O_i,  dS = P (dP - delta),
 *   dQ = scale dS K,  dK = scale dS^T Q,
 * and under grouped-query attention dK, dV of a key/value head are summed over
 * its Hq / Hkv query heads.  Masks and conventions are those of fa_fwd.
 *
 * Inputs (device, row-major, contiguous), dense mode (cu_seqlens == NULL):
 *   q, o, dout [B, Hq, Nq, d] bf16     k, v [B, Hkv, Nk, d] bf16
 *   lse        [B, Hq, Nq]    fp32     (as written by fa_fwd for the same q, k, v)
 * Outputs (device, caller-allocated):
 *   dq [B, Hq, Nq, d] bf16, dk and dv [B, Hkv, Nk, d] bf16,
 *   delta [B, Hq, Nq] fp32: the per-row statistic rowsum(dout * o).
 * Packed mode (cu_seqlens != NULL, as for fa_fwd): q, o, dout, dq [Hq, T, d],
 * k, v, dk, dv [Hkv, T, d], lse and delta [Hq, T], Nq == Nk == T; each
 * sequence's gradients involve only its own tokens.
 *
 * Three kernels are enqueued (delta, then dQ, then dK/dV); the library
 * allocates nothing and uses no atomics, so results are deterministic.
 * Empty problems (B, Hq or Nq equal to 0) return FA_OK; with Nk == 0, dq and
 * delta are written (zeros and rowsum(dout * o)) and k, v, dk, dv may be NULL.
 * Errors are reported as for fa_fwd; argument errors leave every output
 * untouched.  Device-side time-outs set bits 9-11 (dQ kernel) and 13-15
 * (dK/dV kernel) of fa_device_status().
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, float* delta,
                 int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                 const int32_t* cu_seqlens, cudaStream_t stream);

/*
 * fa_fwd_fp8 -- the attention forward with 8-bit (e4m3) inputs, on `stream`.
 * It computes O and LSE of
 *   S = scale * (q8 * q_descale) (k8 * k_descale)^T,  O = softmax(S) (v * v_descale)
 * on the tensor cores' 8-bit path ("FlashAttention v3 Hopper asynchrony"
 * canvas: FP8 is its third technique; the descale factors here are one per
 * (batch, head) slice).  P is rounded to e4m3 before the P V product
 * (relative error at most 2^-4 per term); all accumulation is fp32.
 * Dense mode (cu_seqlens == NULL), d = 64 or 128:
 *   q8   [B, Hq,  Nq, d] e4m3 codes        q_descale [B, Hq]  fp32
 *   k8   [B, Hkv, Nk, d] e4m3 codes        k_descale [B, Hkv] fp32
 *   vt8  [B, Hkv, d, Nk] e4m3 codes (V transposed: every operand of the
 *        8-bit products is K-major)        v_descale [B, Hkv] fp32
 *   o    [B, Hq, Nq, d] bf16,  lse [B, Hq, Nq] fp32 (natural log, of S).
 * Packed mode (cu_seqlens != NULL, as for fa_fwd; Nq == Nk == T tokens):
 *   q8 [Hq, T, d], k8 [Hkv, T, d], vt8 [Hkv, d, T], o [Hq, T, d], lse [Hq, T],
 *   and one descale per head: q_descale [Hq], k_descale and v_descale [Hkv]
 *   (the packed tensor is one batch).  The kernel reads each sequence's keys
 *   from the multiple of 16 at or below its start, as a TMA box on the token
 *   axis of vt8 must start on a 16-byte boundary, and masks the keys before
 *   the start; any offsets work.
 * Nk (T when packed) must be a multiple of 16 (each V^T row is Nk bytes),
 * else FA_ERR_SHAPE; other d give FA_ERR_UNSUPPORTED.  Masks, conventions,
 * ownership and the other errors are as for fa_fwd (16-byte alignment for
 * q8, k8, vt8 and o, 4 bytes for lse, cu_seqlens and the descales).
 */
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                     const float* k_descale, const float* v_descale, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                     const int32_t* cu_seqlens, cudaStream_t stream);

/*
 * fa_fp8_quantize -- e4m3 codes and per-(batch, head) descales of one bf16
 * tensor, for fa_fwd_fp8, on `stream`.  The FA3 canvas ("FlashAttention v3
 * Hopper asynchrony", element pseudo-code) names block scaling of Q, K and V
 * and incoherent processing as what keeps the 8-bit path accurate.  Here a
 * block is one (batch, head) slice, and the incoherent processing is the
 * optional rotation below.
 *   x       [B, H, N, d] bf16 (device, 16-byte aligned), d = 64 or 128
 *   x8      [B, H, N, d] e4m3 codes, or [B, H, d, N] when transpose != 0
 *           (the layout fa_fwd_fp8 takes for V); device, 16-byte aligned
 *   descale [B, H] fp32 (device, 4-byte aligned)
 *   signs   [d] int8, each +1 or -1 (device), or NULL for no rotation
 * With signs, every row is first multiplied by M = diag(signs) H_d / sqrt(d),
 * H_d the Sylvester-Hadamard matrix: M is orthogonal, so Q and K rotated with
 * the same signs give the same Q K^T, while a large channel is spread over
 * all d before rounding.  V is not rotated.  Per slice, with y the rotated
 * (unnormalised, (x * signs) H_d) or plain row values and a = max |y|:
 *   code = e4m3(y * (448 / a)) (nearest even, saturating; 0 when a = 0),
 *   descale = a / (448 sqrt(d)) with rotation, a / 448 without,
 * so that code * descale approximates x M (or x).  The values are computed in
 * float32 with the Walsh-Hadamard butterflies (strides 1, 2, ..., d/2), so the
 * codes do not depend on launch order.
 * Errors: FA_ERR_SHAPE for negative sizes or, with transpose, N not a
 * multiple of 16; FA_ERR_UNSUPPORTED for other d; FA_ERR_NULL / FA_ERR_ALIGN
 * as described; an empty tensor returns FA_OK.  Slices of at most 1024
 * rows, and unrotated, untransposed slices of at most 4096 rows (d = 128) or
 * 8192 rows (d = 64), are handled by one kernel launch: a cluster of up to
 * 16 CTAs per slice holds the slice in shared memory, reads it from global
 * memory once and combines the CTA maxima through distributed shared memory.
 * Other slices take four launches (zeroing, slice maxima, codes, descales),
 * with descale as the slice-maximum accumulator between them.  Both give
 * identical codes and descales, and no other memory is used.  Argument errors leave the outputs untouched.
 * Non-finite inputs: a NaN element is left out of its slice's maximum and
 * gets a NaN code (0x7F or 0xFF); an infinite element makes its slice's
 * maximum and descale +inf, its own code NaN and every other code of the
 * slice a zero (0x00, or 0x80 for negative values).  With the rotation a
 * non-finite element first spreads over its whole row (NaN codes for that
 * row, and for an infinity the slice's other rows become zeros).
 */
fa_status fa_fp8_quantize(const void* x, void* x8, float* descale, int B, int H, int N, int d, int transpose,
                          const int8_t* signs, cudaStream_t stream);

/*
 * fa_fwd_host -- fa_fwd for inputs and outputs in host memory.
 *
 * q_h, k_h, v_h, o_h, lse_h: host buffers in fa_fwd's layouts (dense or
 * packed); pinned (page-locked) memory makes the copies asynchronous and lets
 * them overlap the kernels.  q_d, k_d, v_d, o_d, lse_d: device buffers of the
 * same sizes that the caller provides as staging (the library allocates no
 * device memory); cu_seqlens_h / cu_seqlens_d: the packed offsets on the host
 * and B+1 int32 of device staging for them (both NULL for a dense problem).
 *
 * A dense problem is cut into `pieces` (>= 1; at most B * Hkv) slices, each a
 * range of the flattened (batch, key/value head) index with its query heads:
 * contiguous in every tensor.  Slice sizes fall linearly from the first to
 * the last (weights pieces, ..., 2, 1), which keeps the work left after the
 * last input copy short.  Each slice's host-to-device copies run on a copy-in stream,
 * its fa_fwd launch on `stream` and its device-to-host copies on a copy-out
 * stream (both copy streams belong to the library, one pair per device), so
 * the copies of one slice overlap the kernel and the copies of others.  A
 * packed batch is one slice.  Interview canvas, element flash-text: the
 * method moves data in tiles between the slow and the fast memory; here the
 * same idea overlaps the host link with the kernel.
 *
 * Asynchronous like fa_fwd: the call returns once everything is enqueued,
 * and work enqueued on `stream` afterwards sees O and LSE in host memory
 * (synchronise `stream` before reading them).  The call waits (on the device)
 * for earlier work on `stream` before it writes the staging buffers.
 * Errors: fa_fwd's argument errors, plus FA_ERR_SHAPE for pieces < 1 and
 * FA_ERR_NULL for a missing host or staging buffer, are reported before
 * anything is enqueued; FA_ERR_CUDA if a copy, stream or event call fails.
 * On an error after the first copy was issued, the copies and kernels
 * already enqueued still run, and the call still orders later work on
 * `stream` after them (as far as the CUDA calls for that succeed), so the
 * buffers may be reused once `stream` is synchronised; O and LSE are then
 * incomplete.
 */
fa_status fa_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                      void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d,
                      int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                      const int32_t* cu_seqlens_h, int32_t* cu_seqlens_d, int pieces, cudaStream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* fa_status_string(fa_status s);

/*
 * fa_device_status -- reads and clears the device status words of the current
 * device.  Every wait inside the kernels is bounded; a wait that runs out sets
 * a bit and the kernel leaves cleanly.  Bits 0-4: roles of the fa_fwd kernel
 * (K/V producer, MMA issuer, softmax of query tiles 0 and 1, Q loader);
 * bit 8: the split-KV kernel; bits 9-11 and 13-15: producer, MMA issuer and
 * softmax roles of fa_bwd's dQ and dK/dV kernels; bit 16: fa_fp8_quantize's
 * one-launch kernel.  In a library compiled with FA_DEBUG (libfa_debug.so,
 * built by the package's build(debug=True)), the fa_fwd / fa_fwd_fp8 kernel
 * and fa_bwd's dQ and dK/dV kernels check every TMA box they request (the
 * x coordinate on a 16-byte boundary, the box starting inside the tensor),
 * every output row they write and their TMEM columns before use; a failed
 * check sets bit 5 (forward) or bit 12 (backward) and the access is skipped.
 * Release builds compile the checks away and never set those bits.
 * Returns FA_OK and stores
 * 0 in *bits when nothing went wrong, FA_ERR_TIMEOUT with the bits otherwise.
 * The call first waits for all work on the current device (every stream,
 * cudaDeviceSynchronize), so no kernel can set a bit between the read and the
 * clear; FA_ERR_CUDA if that or a read fails.
 */
fa_status fa_device_status(int* bits);

/*
 * fa_debug_fault_injection -- test hook for the failure path (process-wide,
 * affects every later launch).  mode 0 is normal operation.  Modes 1-4 make
 * one kernel's ring producer withhold its first copy, so that the bounded
 * waits of the roles that need it run out:
 *   1  fa_fwd's kernel (its K/V producer; status bits 0-4),
 *   2  the split-KV kernel of fa_decode and fa_fwd (status bit 8),
 *   3  fa_bwd's dQ kernel (its K/V producer; bits 9-11),
 *   4  fa_bwd's dK/dV kernel (its Q/dO producer; bits 13-15),
 *   5  fa_fp8_quantize's one-launch kernel (its first bulk copy; bit 16).
 * The kernel then records the bits in its device status word, waits (bounded)
 * for its own copies in flight, frees its Tensor Memory and exits, leaving the
 * CUDA context usable; its outputs are undefined.  wait_limit_seconds
 * (0 < x <= 10) sets the bound on every wait inside the kernels; 0 restores
 * the default of 2 s.  Returns FA_ERR_VALUE for other arguments.
 */
fa_status fa_debug_fault_injection(int mode, double wait_limit_seconds);

/*
 * fa_debug_exp2_soft -- test entry point: y[i] = 2^x[i] computed by the
 * kernel's software exponential (FMA/ALU pipes only), for n device floats,
 * asynchronously on `stream`.  Range reduction 2^x = 2^k * 2^f with k = round(x),
 * then a degree-3 minimax polynomial for 2^f on [-1/2, 1/2]; maximum relative
 * error 7.5e-5 for -125 <= x <= 8.  Arguments below -125 give about 2^-125.
 * (The "software exp" of the interview canvas, element v4-card-body.)
 */
fa_status fa_debug_exp2_soft(const float* x, float* y, int n, cudaStream_t stream);

/*
 * fa_debug_soft_exp -- test hook (process-wide, affects every later fa_fwd and
 * fa_fwd_fp8 launch): on = 1 runs the forward kernels' instantiation that
 * computes one exponential pair in every two of each K/V tile without a mask
 * with the software 2^x of fa_debug_exp2_soft (FMA/ALU pipes) instead of the
 * exp unit; on = 0 (the default) restores the normal kernels.  The results
 * stay within the same tolerances; the path is off by default because it
 * measured slower on GB300.  FA_ERR_VALUE for other arguments.
 */
fa_status fa_debug_soft_exp(int on);

/*
 * fa_debug_fwd_pair -- test hook (process-wide, affects every later fa_fwd
 * launch of a bf16 problem with d = 128): on = 1 runs the CTA-pair forward
 * kernel instead of the single-CTA one; on = 0 (the default) restores it.
 * The pair kernel computes the same O and LSE with tensor-core products
 * shared by the two CTAs of a cluster (tcgen05 cta_group::2, M = 256: each
 * CTA holds its own 128 query rows of a product tile, and half of every K
 * tile (64 keys) and V tile (64 head dims), so a K/V tile is read from L2
 * once per pair).  The interview canvas's Blackwell notes (element
 * v4-card-body) name these 2-CTA products.  It is off by default because it
 * measured slower on GB300: the forward step there is set by the one thread
 * that issues the products and by each query tile's softmax-then-products
 * chain, and a pair has one issuing thread for two SMs.  Results stay within
 * the same tolerances.  FA_ERR_VALUE for other arguments.
 */
fa_status fa_debug_fwd_pair(int on);

/*
 * fa_debug_schedule -- the work schedule a persistent launch would use (host
 * only, enqueues nothing; for tooling and tests).  kernel: 0 the bf16
 * forward, 1 the 8-bit forward (always the built-in order), 2 the backward
 * dQ kernel, 3 the backward dK/dV kernel, each for a dense problem of the
 * given shape over `workers` persistent CTAs (the SM count on the device).
 *
 * The kernels' units are independent blocks of rows of one head (the
 * work decomposition of the FlashAttention pages: per (batch, head) blocks of
 * query rows, or of keys for dK/dV).  Under a causal mask their costs differ,
 * so the host orders them: heads are taken in groups whose K/V (or Q/dO)
 * tiles fit in L2, the longest units of a group first, each to the worker
 * predicted to be free first.  On return *table_workers is the number of
 * worker lists (0: no table, the kernel deals its units in its built-in snake
 * order), start[w] .. start[w+1] (start has table_workers + 1 entries) index
 * worker w's units in `units`, in the order it runs them.  capacity is the
 * length of `units`; FA_ERR_SHAPE if it is too small or the shape invalid,
 * FA_ERR_VALUE for an unknown kernel, FA_ERR_NULL for a null pointer.
 */
fa_status fa_debug_schedule(int kernel, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int workers,
                            int32_t* start, int32_t* units, int capacity, int* table_workers);

/* Dynamic shared memory (bytes) and threads per CTA used for head dim d;
 * 0 for an unsupported d.  For tooling and tests. */
int fa_fwd_smem_bytes(int d);
int fa_fwd_threads(void);
int fa_decode_smem_bytes(int d);
int fa_bwd_smem_bytes(int d);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

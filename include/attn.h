/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * The library computes, for every batch b, head h and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * <Q[b,h,i,:], K[b,h,j,:]> ) * V[b,h,j,:]
 *     LSE[b,h,i] = log sum_j exp( scale * <Q[b,h,i,:], K[b,h,j,:]> )
 *
 * over the allowed keys j (all j, or j <= i when causal). This is the
 * attention of "Flash Attention 4 - the algorithm and the two-MMA problem"
 * (section "The memory-bound trap") with the per-row log-sum-exp side output
 * of "Lecture 2 - Online Softmax and Numerical Correctness" (sections "The
 * classical safe softmax" and "Use it in the real stack"). It is computed
 * with the online-softmax recurrence over streamed 128-key blocks (same
 * lecture pages, "Online softmax - three running states" and "Deferred
 * normalization"), the exp2 fold of the scale ("The exp2 trick"), causal block
 * skipping with a diagonal -inf mask ("Causal masking just changes which
 * blocks contribute") and the lagging-max conditional rescale with threshold
 * tau of "FlashAttention-4's Softmax Tricks" ("Conditional rescaling").
 *
 * Conventions shared by every entry point
 *   - Layout: Q, K, V and O are contiguous row-major [B, H, N, d] (d fastest);
 *     LSE is contiguous [B, H, N]. Element (b,h,i,c) is at ((b*H + h)*N + i)*d + c.
 *   - Ownership: the caller allocates and owns every buffer; the attention
 *     entry points allocate no memory. Pointers are device pointers unless a
 *     parameter says otherwise.
 *   - Execution: calls are asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and run on the device current to the calling
 *     thread. Arguments are checked on the host before anything is launched;
 *     a rejected call launches nothing and changes no buffer.
 *   - Thread safety: the library keeps no per-call state; concurrent calls on
 *     different streams are safe if their output buffers do not overlap.
 *   - Errors: every entry point returns an attn_status_t, never aborts.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, non-finite or non-positive scale, ... */
  ATTN_ERR_UNSUPPORTED = 2, /* a well-formed request the library does not implement (e.g. d = 96) */
  ATTN_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed (launch, tensor map, ...) */
  ATTN_ERR_TIMEOUT = 5      /* a kernel gave up waiting on a pipeline barrier (see attn_get_device_status) */
} attn_status_t;

/*
 * attn_fwd -- bf16 attention forward with the per-row LSE.
 *
 *   q, k, v  const bf16 [B,H,N,d], device, 16-byte aligned.
 *   o        bf16 [B,H,N,d], device, 16-byte aligned; written, rounded to nearest even.
 *   lse      float [B,H,N], device, 4-byte aligned; natural-log units of the
 *            scaled scores: LSE_i = scale * m_i + ln(sum_j exp(scale * (s_ij - m_i))).
 *   B, H, N  >= 0. Any of them 0: nothing to do, returns ATTN_OK. N <= 2^24.
 *            N need not be a multiple of 128 (the last key block and the last
 *            query tile are masked).
 *   d        64 or 128 (others: ATTN_ERR_UNSUPPORTED).
 *   causal   0: every key is allowed; 1: key j is allowed for query i iff j <= i.
 *   scale    finite and > 0 (1/sqrt(d) in the usual use). The running max is
 *            taken on raw scores, which is the same as on scaled ones only for
 *            scale > 0.
 *   stream   cudaStream_t.
 * Uses tau = 8 (log2 units) and the MUFU exp2 for every element.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                       int N, int d, int causal, float scale, void* stream);

/*
 * attn_fwd_ex -- attn_fwd with the two softmax tunables exposed.
 *
 *   tau          rescale threshold in log2 units of the scaled score, >= 0
 *                ("FlashAttention-4's Softmax Tricks", section "Conditional
 *                rescaling": the running max moves only when it would grow by
 *                more than tau). 8 for bf16 P; 0 gives the classic rescale on
 *                every growth. Must be <= 16 so that P <= 2^tau stays far
 *                below the bf16 range.
 *   exp2_emu16   how many of every 16 columns of a score row take the software
 *                exp2 on the FMA pipe instead of the MUFU ex2 (same page,
 *                section "The emulated exp2"; the page's fractions 6.25%,
 *                12.5%, 18.75%, 25% are 1, 2, 3, 4 of 16). 0..4 are built;
 *                others give ATTN_ERR_UNSUPPORTED. Masked key blocks (the
 *                causal diagonal and a ragged tail) always use the MUFU.
 * Other arguments as attn_fwd.
 */
attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                          int N, int d, int causal, float scale, float tau, int exp2_emu16, void* stream);

/*
 * attn_fwd_2cta -- attn_fwd on CTA pairs (d = 128, non-causal): the 2-CTA tile
 * of "FlashAttention-4's Softmax Tricks", section "The emulated exp2" (the
 * 2-CTA non-causal d = 128 configuration). Two CTAs on two SMs share each
 * product (tcgen05 cta_group::2, issued by the pair's first CTA): the pair's
 * query tiles are 256 rows, each CTA holding 128 of them, and each CTA stages
 * only half of every 128-key block of K and V, so the pair reads each block
 * from L2 once. Same arguments, layouts, results (within the same tolerance)
 * and errors as attn_fwd, with tau = 8 and the MUFU exp2; d != 128 or
 * causal != 0 give ATTN_ERR_UNSUPPORTED. The grid is as many CTA pairs as the
 * device holds at once (queried on the first call on a device).
 */
attn_status_t attn_fwd_2cta(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                            int d, int causal, float scale, void* stream);

/*
 * attn_combine -- merges the results of attention over disjoint sets of keys
 * (a sequence split: the same queries against key ranges computed apart, e.g.
 * the key chunks of a context-parallel ring) into the result over all of
 * them, with the exact two-block combine of "Lecture 2 - Online Softmax and
 * Numerical Correctness", section "Combining two blocks exactly", applied to
 * every part: m = max_p LSE_p, w_p = exp(LSE_p - m), l = sum_p w_p,
 * O = sum_p w_p O_p / l (fp32 arithmetic, O rounded to bf16 once),
 * LSE = m + ln l.
 *
 *   o_parts    bf16 [parts, B, H, N, d], contiguous: part p's O (as attn_fwd
 *              writes it), 16-byte aligned
 *   lse_parts  fp32 [parts, B, H, N], contiguous: part p's LSE; -inf marks a
 *              part with no key for that row (it adds nothing, and its O row
 *              may hold anything)
 *   parts      1 .. 1024
 *   o, lse     the merged O (bf16 [B, H, N, d], 16-byte aligned) and LSE (fp32
 *              [B, H, N]); a row whose parts are all -inf gets O = 0 and
 *              LSE = -inf. They may not overlap the inputs.
 *   d          64 or 128 (other positive values: ATTN_ERR_UNSUPPORTED)
 * With parts = 1 the output equals the input bit for bit. Errors:
 * ATTN_ERR_INVALID_ARG (negative sizes, parts outside 1 .. 1024, null
 * pointers on a non-empty problem), ATTN_ERR_MISALIGNED, ATTN_ERR_CUDA.
 */
attn_status_t attn_combine(const void* o_parts, const float* lse_parts, int parts, void* o, float* lse, int B, int H,
                           int N, int d, void* stream);

/*
 * attn_fwd_rescale_log -- attn_fwd_ex (software-exp2 share 0) that also
 * records every rescale decision, for checking them against the lagging-max
 * rule of "FlashAttention-4's Softmax Tricks", section "Conditional rescaling,
 * and when it's exact": a row keeps its stale max when the block's maximum
 * raises it by at most tau (log2 units of the scaled score) and moves it
 * otherwise; a warp rescales its O rows when any of its 32 rows moved.
 *
 *   rescale_log  device bytes [B, H, N, ceil(N/128)] (128-key blocks), owned
 *                by the caller; rescale_log_bytes is its size (at least
 *                B*H*N*ceil(N/128), else ATTN_ERR_INVALID_ARG). The kernel writes byte (b, h, i, j) for every
 *                key block j that row i's query tile streams: bit 0 = row i's
 *                running max moved at block j (always set at block 0, where
 *                the max starts at -inf), bit 1 = the row's warp (rows
 *                32 floor(i/32) .. +31 of the head) rescaled O at block j
 *                (j > 0). Bytes of blocks a tile does not stream (causal:
 *                blocks past its diagonal block) are left as they were.
 * A slower debugging variant of the same kernel (the extra stores sit in the
 * softmax loop); O and LSE are the same as attn_fwd_ex's. Errors as
 * attn_fwd_ex, plus ATTN_ERR_INVALID_ARG for a null or too small rescale_log
 * on a non-empty problem.
 */
attn_status_t attn_fwd_rescale_log(const void* q, const void* k, const void* v, void* o, float* lse,
                                   unsigned char* rescale_log, size_t rescale_log_bytes, int B, int H, int N, int d,
                                   int causal, float scale, float tau, void* stream);

/*
 * attn_fwd_host -- attn_fwd with Q, K, V, O and LSE in HOST memory.
 *
 *   q, k, v, o, lse   host pointers, same layouts as attn_fwd. Page-locked
 *                     (pinned) memory lets the copies run asynchronously and
 *                     overlap; pageable memory works but copies synchronously.
 *   workspace         device memory of at least
 *                     attn_fwd_host_workspace_bytes(B, H, N, d) bytes,
 *                     256-byte aligned, owned by the caller; not read or
 *                     written after the call's work on `stream` completes.
 * The B*H heads are cut into about six chunks; each chunk is copied in,
 * computed (attn_fwd) and copied out on three library-owned streams of the
 * current device (created on first use and kept), with two chunk buffers in
 * the workspace, so copies and kernels overlap. The work is ordered after what
 * is already queued on `stream`, and `stream` waits for its completion: the
 * host buffers may be read (O, LSE) or reused once `stream` has synchronised.
 * Results are identical to attn_fwd on the same data (heads are independent).
 * Errors as attn_fwd; ATTN_ERR_INVALID_ARG for a null or too small workspace.
 */
size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d);
attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * attn_fwd_host_noalloc -- attn_fwd_host without a caller workspace, for
 * callers that cannot allocate device memory: a process whose device memory
 * budget is fixed at start-up, or a plug-in inside a host framework whose own
 * allocator owns the device, so that a cudaMalloc of its own would fail or
 * break that framework's accounting. The pages have no counterpart: this is a
 * convenience of the library, not part of the method.
 *
 * The chunk buffers live in one fixed device array of the library,
 * attn_fwd_host_noalloc_max_workspace() bytes (128 MiB); nothing is allocated
 * or freed, by the library or by a routine it calls. Problems whose
 * attn_fwd_host_workspace_bytes(B, H, N, d) exceeds that size are rejected
 * with ATTN_ERR_UNSUPPORTED before any work. The array is a device variable of
 * the library's module: with lazy module loading (CUDA_MODULE_LOADING=LAZY, the
 * runtime's default) a device reserves it when this entry point first runs
 * there; with eager loading every context that loads the library reserves it,
 * and keeps it until the process exits.
 *
 * The first call on a device does a one-time set-up with that device current:
 * it looks up the array's device address and creates one event. Make that
 * first call before any stream capture. Calls on one device share the array and
 * are serialised by the library: each call's work starts after the previous
 * call's copies back have finished, whatever streams the calls use, so calls
 * issued on different streams do not race on it. Nothing in the array needs to
 * start at zero (each call overwrites the parts it reads). Other arguments,
 * ordering and errors as attn_fwd_host; results identical to it.
 */
size_t attn_fwd_host_noalloc_max_workspace(void);
attn_status_t attn_fwd_host_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                    int N, int d, int causal, float scale, void* stream);

/*
 * MXFP8 variant ("PyTorch FlashAttention-4 adds MXFP8 block-scaled forward and
 * backward for Blackwell"): Q, K, V in E4M3 with one E8M0 (power-of-two) scale
 * per 32 x 32 block -- Q and K blocked along d for S = Q K^T, V along the
 * sequence for O = P V (section "Quantization along both axes and jagged
 * tensors") -- and P converted to MXFP8 online per 32 keys inside the kernel
 * (section "Softmax conversion and unroll-KV"). Only d = 128.
 *
 * Scale arrays ("atoms"): for each (b, h) and each 128-row tile t of the
 * sequence, 512 bytes at offset ((b*H + h) * ceil(N/128) + t) * 512 holding the
 * E8M0 scales of 128 rows x 4 blocks of 32 along the GEMM's K dimension; row r,
 * block kb at byte (r % 32) * 16 + (r / 32) * 4 + kb. For Q and K (role 0) the
 * row is the sequence position in the tile and kb = d / 32; for V (role 1) the
 * row is the d column and kb the 32-key block of the tile. This is the layout
 * the block-scaled tensor-core MMA reads after tcgen05.cp.
 */

/* Bytes of one tensor's scale array: B*H*ceil(N/128)*512; 0 if any size is
 * <= 0 or d != 128. The caller allocates it (device, 16-byte aligned). */
size_t attn_mxfp8_scale_bytes(int B, int H, int N, int d);

/*
 * attn_mxfp8_quantize -- fp32 [B,H,N,d] (device, 16-byte aligned) to E4M3
 * codes [B,H,N,d] (x_e4m3, one byte each) and the scale array (x_scales).
 * Each 32 x 32 block (rows past N count as zero) takes the smallest power of
 * two 2^e with amax / 2^e <= 448; elements are multiplied by 2^-e and rounded
 * to E4M3, nearest even, saturating at +-448. role 0: the atom layout of a
 * product along d (Q, K of the forward); role 1: along the sequence (V of the
 * forward); role 2: both (the blocks are square, so the codes are the same),
 * x_scales then holding 2 * attn_mxfp8_scale_bytes bytes, role 0's array
 * first and role 1's right after it (Q, K, dO of attn_bwd_mxfp8).
 * d must be 128 (else ATTN_ERR_UNSUPPORTED); B*H <= 65535. Asynchronous on
 * stream; allocates nothing.
 */
attn_status_t attn_mxfp8_quantize(const float* x, void* x_e4m3, void* x_scales, int B, int H, int N, int d,
                                  int role, void* stream);

/*
 * attn_fwd_mxfp8 -- attention forward from MXFP8 inputs (the outputs of
 * attn_mxfp8_quantize: q8/q_sf and k8/k_sf with role 0, v8/v_sf with role 1),
 * block-scaled tensor-core MMAs with fp32 accumulation, P converted to
 * E4M3 with one E8M0 scale per 32 keys (the block's amax from its score max),
 * the row sum taken from fp32 P. o, lse, B, H, N, causal, scale as attn_fwd;
 * d must be 128. All pointers device, 16-byte aligned (lse: 4).
 * tau = 0: the threshold is dtype-aware ("FlashAttention-4's Softmax Tricks",
 * section "Where exact breaks: P in FP8": 8 for 16-bit P, 0 for FP8). With a
 * stale max a row's largest P is 2^delta, not exactly 1, and E4M3's 3-bit
 * mantissa rounds it by up to 2^-4, which on peaked rows moves O by several
 * 1e-2; with tau = 0 it is exactly 1 and exact in E4M3 after its scale.
 */
attn_status_t attn_fwd_mxfp8(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v8,
                             const void* v_sf, void* o, float* lse, int B, int H, int N, int d, int causal,
                             float scale, void* stream);

/* How attn_fwd_mxfp8_ex scales P before converting it to FP8 for the P V
 * product (V stays E4M3). */
enum {
  /* one E8M0 scale per 32 keys of a row, from the group's largest P (the
   * exp of its largest score): the conversion attn_fwd_mxfp8 uses */
  ATTN_P_SCALE_BLOCK_AMAX = 0,
  /* the constant 2^-8 ("PyTorch FlashAttention-4 adds MXFP8 block-scaled
   * forward and backward for Blackwell", section "Softmax conversion and
   * unroll-KV": softmax keeps P in [0, 1], so a fixed scale is robust): P = 1
   * maps to 256; needs tau <= log2(448 / 256) ~ 0.807 so that 2^tau * 256
   * stays within E4M3 (else ATTN_ERR_INVALID_ARG) */
  ATTN_P_SCALE_CONSTANT = 1,
  /* the same constant 2^-8 with P held in E5M2 ("FlashAttention-4's Softmax
   * Tricks", section "Where 'exact' breaks: P in FP8": E5M2's largest value
   * 57344 leaves room for a stale maximum that E4M3 lacks, at 2 mantissa
   * bits instead of 3): needs tau <= log2(57344 / 256) ~ 7.807 (else
   * ATTN_ERR_INVALID_ARG) */
  ATTN_P_SCALE_CONSTANT_E5M2 = 2
};

/* attn_fwd_mxfp8 with tau in [0, 16], a software-exp2 share of 0, 2 or 4 of
 * every 16 score columns (others: ATTN_ERR_UNSUPPORTED) and p_scaling one of
 * ATTN_P_SCALE_* (else ATTN_ERR_INVALID_ARG). */
attn_status_t attn_fwd_mxfp8_ex(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v8,
                                const void* v_sf, void* o, float* lse, int B, int H, int N, int d, int causal,
                                float scale, float tau, int exp2_emu16, int p_scaling, void* stream);

/*
 * attn_fwd_mxfp8_unroll_kv -- attn_fwd_mxfp8 (tau = 0, P scaled per 32 keys
 * from the block amax, MUFU exp2) on the unroll-KV schedule of "PyTorch
 * FlashAttention-4 adds MXFP8 block-scaled forward and backward for
 * Blackwell", section "Softmax conversion and unroll-KV": in the last key
 * block of a work item the next item's first QK^T product is issued between
 * this item's last two P V products, and the softmax takes P's fp32 row sum
 * after handing P over. Same arguments, layouts, results (within the same
 * tolerance) and errors as attn_fwd_mxfp8. Slower than attn_fwd_mxfp8 on
 * GB300 (its softmax warps run the epilogue, which already hides the
 * item-boundary wait); kept for comparison.
 */
attn_status_t attn_fwd_mxfp8_unroll_kv(const void* q8, const void* q_sf, const void* k8, const void* k_sf,
                                       const void* v8, const void* v_sf, void* o, float* lse, int B, int H, int N,
                                       int d, int causal, float scale, void* stream);

/*
 * attn_fwd_mxfp8_rescale_log -- attn_fwd_mxfp8_ex (P scaled per 32 keys from
 * the block amax, MUFU exp2, any tau in [0, 16]) that also records every
 * rescale decision in rescale_log, exactly as attn_fwd_rescale_log does for
 * the bf16 kernel: device bytes [B, H, N, ceil(N/128)] (rescale_log_bytes at
 * least that), bit 0 = the row's max moved at that key block, bit 1 = its warp
 * rescaled O; bytes of blocks a tile does not stream are left as they were. A
 * debugging variant of the same kernel. Errors as attn_fwd_mxfp8_ex, plus
 * ATTN_ERR_INVALID_ARG for a null or too small rescale_log on a non-empty
 * problem.
 */
attn_status_t attn_fwd_mxfp8_rescale_log(const void* q8, const void* q_sf, const void* k8, const void* k_sf,
                                         const void* v8, const void* v_sf, void* o, float* lse,
                                         unsigned char* rescale_log, size_t rescale_log_bytes, int B, int H, int N,
                                         int d, int causal, float scale, float tau, void* stream);

/*
 * attn_selftest_wait_timeout -- exercises the kernels' failure detection
 * without a fault: launches one small kernel on stream whose warps wait, with
 * the same bounded wait the attention kernels use, on barriers that nothing
 * completes. One wait gives up after limit_cycles SM clock cycles, records
 * ATTN_ERR_TIMEOUT in the device status word and raises the block's abort
 * flag; the other (64 times the limit) returns early on that flag, so the
 * kernel ends after about limit_cycles. attn_get_device_status then reports
 * ATTN_ERR_TIMEOUT (and clears it); the context stays usable.
 * limit_cycles in [1000, 1e10], else ATTN_ERR_INVALID_ARG. Asynchronous.
 */
attn_status_t attn_selftest_wait_timeout(long long limit_cycles, void* stream);

/*
 * attn_exp2_emulated -- y[i] = software exp2 of x[i] for i < n, computed by
 * the very device function the attention kernels use on the FMA pipe (see
 * attn_fwd_ex). For checking that function bit for bit against a scalar model.
 *   x, y   float, device, n elements each (may not overlap unless x == y).
 *   n      >= 0.
 */
attn_status_t attn_exp2_emulated(const float* x, float* y, long long n, void* stream);

/*
 * attn_get_device_status -- synchronise `stream`, then report and clear the
 * device-side error word of the current device. Every pipeline wait inside the
 * kernels has an iteration/time limit (about two seconds); a wait that runs out
 * records ATTN_ERR_TIMEOUT there and its kernel drains and exits instead of
 * hanging. Returns ATTN_OK if no kernel recorded an error since the last call.
 */
attn_status_t attn_get_device_status(void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* attn_status_string(attn_status_t status);

/*
 * attn_bwd -- the backward pass: dQ, dK, dV of O = softmax(s Q K^T [causal
 * mask]) V for an upstream gradient dO, with P rebuilt from the forward's LSE
 * ("Lecture 2 - Online Softmax and Numerical Correctness", section "Use it in
 * the real stack": the LSE side output makes the backward cheap) and the five
 * products S, dP, dV, dK, dQ of "PyTorch FlashAttention-4 adds MXFP8
 * block-scaled forward and backward for Blackwell", section "TMEM allocation
 * and scale factor placement" (dK and dV accumulated per key tile):
 *   P = exp(s Q K^T - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
 *   dS = P * (dP - D), dQ = s dS K, dK = s dS^T Q.
 *
 *   q, k, v, o, dout  bf16 [B, H, N, d] contiguous, device memory, 16-byte
 *                     aligned: the forward's inputs, its output O and dL/dO.
 *   lse               fp32 [B, H, N], the forward's LSE (4-byte aligned).
 *   dq, dk, dv        bf16 [B, H, N, d] outputs, 16-byte aligned.
 *   B, H, N, d, causal, scale   as attn_fwd (d 64 or 128).
 *   workspace         device memory of at least attn_bwd_workspace_bytes(B,
 *                     H, N, d) bytes, 256-byte aligned, owned by the caller:
 *                     an fp32 dQ accumulator, D and LSE log2(e).
 * Asynchronous on `stream` (three kernels: preparation, the main kernel, dQ
 * conversion); nothing is allocated. Errors as attn_fwd, plus
 * ATTN_ERR_INVALID_ARG for a null or too small workspace and
 * ATTN_ERR_UNSUPPORTED for B*H > 65535.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                       float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_mxfp8 -- the backward pass with all five products on the
 * block-scaled tensor cores ("PyTorch FlashAttention-4 adds MXFP8
 * block-scaled forward and backward for Blackwell", section "Quantization
 * along both axes and jagged tensors": square 32 x 32 blocks for Q, K and dO,
 * whose one E4M3 payload serves the products along d and along the sequence,
 * and for dS, which the dK and dQ products both read). The same gradient as
 * attn_bwd, computed from the quantised inputs, with
 *   P entering dV as E4M3 with the constant scale 2^-8 (P = 1 held as 256);
 *   dS = P (dP - D) from the unrounded P, rounded to E4M3 in 32 x 32 blocks
 *   of (queries, keys) with the quantiser's scale rule;
 *   D = rowsum(dO * O) from the dequantised dO and O.
 *
 *   q8, k8, do8       E4M3 [B, H, N, 128] from attn_mxfp8_quantize with
 *   q_sf, k_sf, do_sf role 2 (their scale arrays hold both layouts);
 *   v8, v_sf          V from attn_mxfp8_quantize with role 0;
 *   o                 bf16 [B, H, N, 128], the forward's output;
 *   lse               fp32 [B, H, N], the forward's LSE (4-byte aligned);
 *   dq, dk, dv        bf16 [B, H, N, 128] outputs;
 *   workspace         as attn_bwd: attn_bwd_workspace_bytes(B, H, N, 128)
 *                     bytes, 256-byte aligned, owned by the caller.
 * d must be 128 (else ATTN_ERR_UNSUPPORTED), B*H <= 65535. All other
 * pointers device memory, 16-byte aligned. Asynchronous on `stream` (three
 * kernels); nothing is allocated. Errors as attn_bwd.
 */
attn_status_t attn_bwd_mxfp8(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v8,
                             const void* v_sf, const void* o, const void* do8, const void* do_sf, const float* lse,
                             void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */

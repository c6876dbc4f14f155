/*
 * zyfa.h -- C ABI of the GB300 (sm_103a) causal attention forward library.
 *
 * The operation is the causal FlashAttention forward (prefill) pass of
 * "ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4"
 * (arXiv 2611.07496):
 *
 *     O = softmax(c Q K^T + M) V,   c = 1/sqrt(d_qk),  M the causal mask
 *                                   (Sec. II-B),
 *
 * computed FlashAttention-style over blocks of 128 keys with a running row
 * maximum in base-2 units and lazy rescaling (Sec. II-B; Sec. IV-A "Lazy
 * rescaling": tau = 0.125 in FP8, 0.5 in BF16 at d_qk = 128, 8 in BF16 at
 * d_qk = 192).  In FP8 the inputs are e4m3 codes with one FP32 scale per
 * tensor (Sec. II-C); each probability is rounded to e4m3 before the PV
 * product either by Lean P, the code y = 8(x + 6 + 7) - 0.35 rounded to an
 * integer (Sec. IV-B1, Eq. 2), or by exact P, e4m3(2^(x+6)); each block of 64
 * keys of a row is scaled by 2^o, o the whole binades between the block
 * maximum and the row maximum, and the PV product by 2^-o (Sec. IV-B2); the
 * output divides by the sum of the rounded probabilities (Sec. IV-B3).
 *
 * Common conventions
 *   - Layout: contiguous BSHD.  q [B, N, Hq, d_qk], k [B, N, Hkv, d_qk],
 *     v [B, N, Hkv, d_v], out [B, N, Hq, d_v].  Query head h reads key/value
 *     head h / (Hq / Hkv) (grouped-query attention, Table VI).  The
 *     *_strided entry points take any strides (BHSD among them).
 *   - Supported: causal = 1 (the paper's setting) or 0 (every query sees
 *     every key); N a multiple of 128; (d_qk, d_v) = (128, 128) or
 *     (192, 128); Hq a multiple of Hkv.
 *   - Ownership: every buffer is device memory owned by the caller (but
 *     zyfa_fwd_host, which takes host buffers and a device workspace).  The
 *     attention entry points allocate no device memory, keep no pointer
 *     after the call returns and write nothing but `out` (and `lse`, and
 *     zyfa_fwd_host's workspace).
 *     zyfa_quantize takes stream-ordered scratch (cudaMallocAsync /
 *     cudaFreeAsync on `stream`) when it needs a per-call maximum or a mean.
 *   - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and the call returns without synchronising.
 *   - Errors: a bad argument returns a negative status before anything is
 *     launched; a failed launch returns ZYFA_ERR_CUDA.  Every wait inside the
 *     kernel is bounded (about 1.5 s); a wait that runs out ends the kernel
 *     early and is reported by zyfa_last_device_status().
 *   - B = 0 or N = 0 is an empty problem: ZYFA_OK, nothing launched, the
 *     pointers are not inspected.
 */
#ifndef ZYFA_H
#define ZYFA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZYFA_OK = 0,
    ZYFA_ERR_NULL = -1,         /* a required pointer is NULL                     */
    ZYFA_ERR_SHAPE = -2,        /* negative/zero sizes, Hq % Hkv, N % 128, limits */
    ZYFA_ERR_UNSUPPORTED = -3,  /* causal not 0/1, head dims, p_mode / block_scale */
    ZYFA_ERR_ALIGN = -4,        /* a tensor not 16-byte aligned, a scale not 4    */
    ZYFA_ERR_CUDA = -5,         /* launch or driver call failed                   */
    ZYFA_ERR_TIMEOUT = -6,      /* a device-side wait ran out (see below)         */
    ZYFA_ERR_SCRATCH = -7       /* needs more scratch or workspace than given      */
} zyfa_status;

enum { ZYFA_P_EXACT = 0, ZYFA_P_LEAN = 1 };

/*
 * FP8 e4m3 causal attention forward.
 *   q, k, v      e4m3 ("fn" variant) codes, one byte per element, BSHD.
 *   descale_q/k/v  pointers to one FP32 value each in device memory: the
 *                scale that maps a code back to its real value; NULL means
 *                1.0.  They enter the score scale c*dq*dk and the output.
 *   out          BF16 output, BSHD, d_v = 128 (round to nearest even).
 *   p_mode       ZYFA_P_LEAN (Eq. 2) or ZYFA_P_EXACT.
 *   block_scale  1: per-64-key power-of-two scaling (Sec. IV-B2); 0: o = 0.
 *   stream       cudaStream_t the kernel is launched on.
 * Returns a zyfa_status.
 */
int zyfa_fwd(const void* q, const void* k, const void* v,
             const float* descale_q, const float* descale_k, const float* descale_v,
             void* out, int B, int Hq, int Hkv, int N, int d_qk, int d_v,
             int causal, int p_mode, int block_scale, void* stream);

/*
 * BF16 causal attention forward (the comparison path of Sec. IV-D): q, k, v
 * and out are BF16, BSHD.  Probabilities p = 2^(t - m) are computed in FP32,
 * rounded to BF16 for the PV product, and the row sum adds the unrounded p.
 * Same conventions and status codes as zyfa_fwd.
 */
int zyfa_fwd_bf16(const void* q, const void* k, const void* v, void* out,
                  int B, int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                  void* stream);

/*
 * zyfa_fwd with the log-sum-exp of each query row (NEXT to the forward pass:
 * the paper's kernels return it so that results over different key ranges
 * can be merged, Sec. IV-B3).
 *   lse   NULL, or FP32 device memory [B, Hq, N] (4-byte aligned) that
 *         receives ln(sum_j exp(c * dq * dk * q_i . k_j)) computed from the
 *         same rounded, block-scaled probabilities the output is normalised
 *         by: ln(l) + (m - 6) ln 2, l the rounded row sum relative to the
 *         final running maximum m (base-2 units) and 6 the probability shift.
 * Everything else as zyfa_fwd.
 */
int zyfa_fwd_ex(const void* q, const void* k, const void* v,
                const float* descale_q, const float* descale_k, const float* descale_v,
                void* out, float* lse, int B, int Hq, int Hkv, int N, int d_qk, int d_v,
                int causal, int p_mode, int block_scale, void* stream);

/*
 * zyfa_fwd_bf16 with the log-sum-exp of each row, ln(l) + m ln 2 with l the
 * FP32 row sum of the unrounded probabilities; lse as in zyfa_fwd_ex.
 */
int zyfa_fwd_bf16_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                     int B, int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                     void* stream);

/*
 * Quantisation pass before FP8 attention (Sec. V-A, "FP8 inputs and
 * policies" and "Rotation and K smoothing"; Table XIII): BF16 -> e4m3 with
 * one power-of-two scale per tensor, computed after the optional transforms.
 * For each row x of D channels (row (b, n, h) of a BSHD tensor):
 *     u = x - mean_n(x[b, :, h, :])      if smooth (K smoothing), else x
 *     y = u R,  R = diag(s) (C_m kron H_{D/m})   if signs != NULL, else u
 *     code = e4m3(y / d), round to nearest even, saturating at +-448,
 *            NaN -> 0x7F
 * with H the normalised Sylvester-Hadamard matrix, C_m the orthonormal
 * DCT-II of size m (m = 1 for D = 128, 3 for D = 192), the element index
 * j = a*(D/m) + b of R's rows and columns split as (DCT index a, Hadamard
 * index b), and all arithmetic in FP32.  Rotate Q and K with the same
 * signs: (QR)(KR)^T = QK^T, so the attention output is unchanged up to
 * rounding; V is not rotated.
 *   x             BF16 [B, N, H, D], contiguous, 16-byte aligned.
 *   signs         NULL (no rotation) or D FP32 values in device memory whose
 *                 sign bits are the s of R (the paper draws them at random
 *                 with seed 0; any fixed +-1 vector is a valid R).
 *   smooth        1: subtract the mean over the N positions of each (b, h)
 *                 pair, channel by channel, before the rotation; 0: no.
 *   static_descale  > 0: the descale d, a power of two in [2^-126, 2^127]
 *                 (a static, calibrated scale; larger values saturate);
 *                 0: per call, d = the smallest power of two >= 2^-126 with
 *                 max |y| <= 448 d over the finite y (d = 1 if none is
 *                 nonzero).
 *   out           e4m3 codes [B, N, H, D], 16-byte aligned.
 *   descale_out   one FP32 in device memory (required): receives d, so it
 *                 can be passed straight to zyfa_fwd as descale_q/k/v.
 *   mean_out      NULL, or FP32 [B, H, D] device memory (16-byte aligned)
 *                 that receives the subtracted means (smooth = 1 only).
 *   D             128 or 192.
 * Reductions are deterministic (fixed summation order; the maximum is
 * order-free), so repeated calls give identical bytes.  An empty tensor
 * (B, N or H = 0) only writes descale_out.  Errors: ZYFA_ERR_SHAPE
 * (negative sizes, grid limits), ZYFA_ERR_UNSUPPORTED (D, smooth,
 * static_descale), ZYFA_ERR_NULL, ZYFA_ERR_ALIGN, ZYFA_ERR_CUDA (scratch
 * allocation or launch).  Asynchronous on `stream`.
 */
int zyfa_quantize(const void* x, const float* signs, int smooth, float static_descale,
                  void* out, float* descale_out, float* mean_out,
                  int B, int N, int H, int D, void* stream);

/*
 * zyfa_quantize without any device allocation (no counterpart in the
 * paper).  For callers that must not allocate device memory once running
 * -- a serving process with a fixed memory budget, or one whose device
 * memory pool is managed by another allocator -- the scratch that
 * zyfa_quantize takes with cudaMallocAsync (the per-call maximum word, the
 * partial sums of the mean key and, when mean_out is NULL, the mean) comes
 * from a fixed 16 MiB array in device memory, one per device.  Same
 * arguments, same kernels, same results bit for bit.
 *   - Limit: a call that needs more than 16 MiB of scratch returns
 *     ZYFA_ERR_SCRATCH before launching anything.  Static scales without
 *     smoothing need none, a per-call scale 256 bytes.  Smoothing needs
 *     4 x B x nchunk x H x D bytes of partial sums, the library choosing
 *     nchunk = min(ceil(608 / (B x ceil(H x D / 4096))), ceil(N / 16)),
 *     plus 4 x B x H x D for the mean when mean_out is NULL: about 10 MB
 *     for B = 1, H = 32, D = 128, N = 32768.
 *   - The first call on each device looks the array up with
 *     cudaGetSymbolAddress, which may load the module: make it outside any
 *     stream capture.  The address is kept per device together with the
 *     context it was found in; a call that finds another context current
 *     (after a device reset) looks it up again, which is then such a first
 *     call.
 *   - The array used is the current device's: `stream` must belong to the
 *     current device (ZYFA_ERR_UNSUPPORTED otherwise, checked before
 *     anything is launched, when the call needs scratch).
 *   - The maximum word is zeroed on `stream` by every call that uses it;
 *     the rest of the scratch is written before it is read.
 *   - All calls on one device share the array: calls whose work overlaps in
 *     time (other streams, other host threads) race and must be serialised
 *     by the caller.
 */
int zyfa_quantize_noalloc(const void* x, const float* signs, int smooth, float static_descale,
                          void* out, float* descale_out, float* mean_out,
                          int B, int N, int H, int D, void* stream);

/*
 * zyfa_fwd_ex on tensors with any strides (Table VI runs both the BSHD and
 * the BHSD layout).  Each tensor is addressed as [B, N, H, d] with a
 * contiguous last dimension:
 *   strides   NULL (contiguous BSHD, as zyfa_fwd_ex), or 12 element strides
 *             {q_b, q_n, q_h, k_b, k_n, k_h, v_b, v_n, v_h, o_b, o_n, o_h}:
 *             the distance between consecutive batches, positions and heads
 *             of q, k, v and out.  BHSD is {H N d, d, N d} for each.
 * Each stride must be positive; q, k and v strides times the element size
 * must be multiples of 16 bytes (TMA) and below 2^40 bytes, out strides
 * multiples of 8 elements and below 2^39 elements (the FP8 kernels write out
 * through a tensor map too).  ZYFA_ERR_SHAPE / ZYFA_ERR_ALIGN otherwise.
 * Everything else as zyfa_fwd_ex (lse stays [B, Hq, N] contiguous).
 */
int zyfa_fwd_strided(const void* q, const void* k, const void* v,
                     const float* descale_q, const float* descale_k, const float* descale_v,
                     void* out, float* lse, int B, int Hq, int Hkv, int N, int d_qk, int d_v,
                     int causal, int p_mode, int block_scale, const long long* strides,
                     void* stream);

/* zyfa_fwd_bf16_ex on strided tensors; strides as in zyfa_fwd_strided. */
int zyfa_fwd_bf16_strided(const void* q, const void* k, const void* v, void* out, float* lse,
                          int B, int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                          const long long* strides, void* stream);

/*
 * BF16 QK^T with FP8 PV: the variant the paper's conclusion recommends
 * (V adds the least input error, so keeping QK^T in BF16 and running only PV
 * in FP8 removes most of the input error).  Q and K are BF16 (no descale),
 * the scores come from a BF16 MMA, and everything after them is the FP8 path
 * of zyfa_fwd: running maximum (tau = 0.125), Lean P or exact P codes with
 * sigma = 6, per-64-key block scaling, the block-scaled e4m3 PV product with
 * V's descale, division by the rounded row sum.
 *   q, k        BF16 [B, N, H, d_qk];  v  e4m3 codes [B, N, Hkv, d_v].
 *   descale_v   one FP32 in device memory, or NULL for 1.0.
 *   strides     as zyfa_fwd_strided (q and k strides x 2 bytes, v strides
 *               x 1 byte must be multiples of 16), or NULL for BSHD.
 * Everything else as zyfa_fwd_ex.
 */
int zyfa_fwd_bf16qk_fp8pv(const void* q, const void* k, const void* v, const float* descale_v,
                          void* out, float* lse, int B, int Hq, int Hkv, int N, int d_qk,
                          int d_v, int causal, int p_mode, int block_scale,
                          const long long* strides, void* stream);

/*
 * Attention over the keys [key_begin, key_end) only: the split-key form of
 * the forward.  The paper returns the LSE so that results over different key
 * ranges can be merged (Sec. IV-B3); this call gives one such result and
 * zyfa_merge combines them (to spread one long sequence over more SMs, or to
 * combine results computed over separate parts of K and V).
 * The method runs on the range's keys alone: query i sees key j iff
 * key_begin <= j < key_end and (causal) j <= i; the running maximum, the
 * lazy rescale and the block scales start at key_begin.  Rows that see no
 * key of the range get out = 0 and lse = -inf (the merge's identity).
 *   key_begin, key_end   multiples of 128, 0 <= key_begin <= key_end <= N
 *                        (ZYFA_ERR_SHAPE otherwise);
 *   lse                  required (ZYFA_ERR_NULL when NULL), FP32 [B, Hq, N].
 * Everything else as zyfa_fwd_strided (strides NULL for BSHD), with the same
 * kernels.  Merging disjoint ranges that cover [0, N) gives attention over
 * all keys up to the BF16 rounding of each part and the per-range choices of
 * maximum and block scale.
 */
int zyfa_fwd_partial(const void* q, const void* k, const void* v,
                     const float* descale_q, const float* descale_k, const float* descale_v,
                     void* out, float* lse, int B, int Hq, int Hkv, int N, int d_qk, int d_v,
                     int causal, int p_mode, int block_scale, int key_begin, int key_end,
                     const long long* strides, void* stream);

/* zyfa_fwd_partial for BF16 inputs (the zyfa_fwd_bf16 method over a range). */
int zyfa_fwd_bf16_partial(const void* q, const void* k, const void* v, void* out, float* lse,
                          int B, int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                          int key_begin, int key_end, const long long* strides, void* stream);

/*
 * Merge of partial results over disjoint key ranges by their LSE
 * (Sec. IV-B3).  Per row, in FP32: M = max_i LSE_i, L = M + ln sum_i
 * exp(LSE_i - M), out = BF16_RNE(sum_i exp(LSE_i - L) O_i); rows whose LSEs
 * are all -inf get out = 0 and L = -inf.
 *   outs      host array of n_parts device pointers, BF16 [B, N, Hq, d_v]
 *             contiguous, 16-byte aligned;
 *   lses      host array of n_parts device pointers, FP32 [B, Hq, N];
 *   n_parts   1 .. 16 (ZYFA_ERR_SHAPE below, ZYFA_ERR_UNSUPPORTED above);
 *   out       BF16 [B, N, Hq, d_v], caller-owned; may be one of outs;
 *   lse       FP32 [B, Hq, N] for L, or NULL; may be one of lses;
 *   d_v       a power of two from 8 to 4096; B x Hq x N below 2^31
 *             (ZYFA_ERR_SHAPE otherwise).
 * The arrays outs and lses are read during the call only.  Asynchronous on
 * `stream`; allocates nothing.
 */
int zyfa_merge(const void* const* outs, const float* const* lses, int n_parts, void* out,
               float* lse, int B, int Hq, int N, int d_v, void* stream);

/*
 * The FP8 forward end to end on HOST buffers: the inputs are copied to
 * device memory, zyfa_fwd_strided's kernels run, and the output (and the
 * LSE) are copied back.  Attention is independent per batch element and per
 * query head (Sec. II-B; a key/value head serves Hq / Hkv query heads,
 * Table VI), so the work is cut into chunks whose copies overlap the other
 * chunks' kernels (zyfa_fwd_host_plan): ranges of batch elements with all
 * heads when B >= n_chunks; else, with w = ceil(n_chunks / B) chunks per
 * batch element, its key/value heads in the largest number of equal groups
 * not above w when Hkv >= w, or else one key/value head per chunk group
 * with its query heads split into the largest number of equal sub-ranges
 * not above ceil(w / Hkv) (K and V copied once, by the first sub-range).
 * The result is bit-identical to zyfa_fwd_ex on the same data.
 *   q, k, v      HOST e4m3 codes, contiguous BSHD as zyfa_fwd.  Page-locked
 *                memory (cudaHostAlloc / cudaHostRegister) lets the copies
 *                overlap the kernels; pageable memory also works, but the
 *                copies then block the host and do not overlap.
 *   descale      HOST array {descale_q, descale_k, descale_v}, read during
 *                the call (the values are passed to the device by value),
 *                or NULL for 1.0 each.
 *   out          HOST BF16 [B, N, Hq, d_v];  lse  HOST FP32 [B, Hq, N] or
 *                NULL.  Both are written when the work enqueued on `stream`
 *                completes (synchronise `stream` before reading them).
 *   n_chunks     0 (the library's choice, 16) or 1 .. 32 (ZYFA_ERR_SHAPE
 *                otherwise); the plan holds at most 2 x n_chunks - 1 chunks.
 *   workspace    device memory owned by the caller, 256-byte aligned
 *                (ZYFA_ERR_ALIGN), of at least
 *                zyfa_fwd_host_workspace_bytes(B, Hq, Hkv, N, d_qk, d_v,
 *                lse != NULL) bytes (ZYFA_ERR_SCRATCH when smaller): the
 *                device copies of q, k, v, out and lse and the three scales.
 *                It must not be used by other work until `stream` has passed
 *                the call.
 * Everything else (shapes, modes, errors) as zyfa_fwd_ex; every argument
 * error is returned before anything is enqueued.  The work runs on four
 * streams the library keeps per device (created on the first call and kept
 * for the life of the process), forked from `stream` and joined back to it
 * with events, so the call is ordered on `stream` like the other entry
 * points and can be captured into a CUDA graph (page-locked buffers only).
 * Calls from several host threads take a lock while they enqueue.  A copy
 * or launch that fails returns ZYFA_ERR_CUDA after the streams are joined.
 */
int zyfa_fwd_host(const void* q, const void* k, const void* v, const float* descale, void* out,
                  float* lse, int B, int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                  int p_mode, int block_scale, int n_chunks, void* workspace,
                  size_t workspace_bytes, void* stream);

/* The chunk plan zyfa_fwd_host follows, as pure host arithmetic (no CUDA
 * call): writes the first `cap` chunks as 7 ints each, {b0, nb, g0, hk, h0,
 * hq, kv}: batch elements [b0, b0 + nb), key/value heads [g0, g0 + hk),
 * query heads [h0, h0 + hq), kv = 1 when the chunk copies K and V in (0:
 * an earlier chunk copied them).  Returns the number of chunks (at most
 * 2 x n_chunks - 1; n_chunks = 0 means 16), or ZYFA_ERR_SHAPE (B, Hq or
 * Hkv below 1, Hq % Hkv, n_chunks outside 0 .. 32, cap < 0) or
 * ZYFA_ERR_NULL (chunks NULL with cap > 0). */
int zyfa_fwd_host_plan(int B, int Hq, int Hkv, int n_chunks, int* chunks, int cap);

/* Device bytes zyfa_fwd_host needs as workspace (the device copies rounded
 * up to 256 bytes each, plus 256 for the scales); 0 for negative sizes, Hq
 * or Hkv below 1, or a total beyond 2^63.  Pure host arithmetic. */
size_t zyfa_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d_qk, int d_v,
                                     int with_lse);

/* Static, NUL-terminated description of a status code. */
const char* zyfa_status_string(int status);

/*
 * Synchronises `stream`, then reports and clears the device status word of
 * the current device: ZYFA_ERR_TIMEOUT if any kernel of this library has had
 * a bounded wait run out since the last call, else ZYFA_OK (or
 * ZYFA_ERR_CUDA if the synchronisation itself failed).
 */
int zyfa_last_device_status(void* stream);

/*
 * Test hook for the failure path (no counterpart in the paper): launches one
 * thread that waits on an mbarrier nothing arrives at.  Its bounded wait
 * runs out after about 1.5 s, records a timeout in the device status word
 * and the kernel returns normally, so the next zyfa_last_device_status()
 * on this device reports ZYFA_ERR_TIMEOUT and the context stays usable.
 * Asynchronous on `stream`; returns ZYFA_OK or ZYFA_ERR_CUDA.
 */
int zyfa_selftest_timeout(void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int zyfa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZYFA_H */

/*
 * qmm.h -- C ABI of libqmm: block-quantized weight x Q8 activation matmul on
 * GB300 (sm_103a).
 *
 * y = W . x where W stays in its block-quantized form (Q4_0, Q8_0, Q4_K, Q6_K,
 * Q2_K; also Q4_1, Q5_0, Q5_1, Q5_K) and is never dequantized as a whole, x is
 * quantized on the fly to Q8_0 or Q8_K, and every block is an exact integer dot
 * product whose per-block scales (and mins) are folded into an fp32
 * accumulator once per block.
 *
 * A decode token and a prefill, with device buffers (error checks elided):
 *
 *   size_t wb = qmm_row_bytes(QMM_Q8_0, K) * N;          // W: N rows of Q8_0
 *   size_t sb = qmm_row_bytes(qmm_act_type(QMM_Q8_0), K); // one quantized row
 *   // x: f32 [1][K], y: f32 [1][N], scratch: sb bytes, all 16-byte aligned
 *   qmm_linear_q8_0(W, x, scratch, sb, y, 1, N, K, stream);
 *   // M tokens: scratch of M * sb bytes; M >= 8 runs on the tensor cores
 *   qmm_linear_q8_0(W, X, scratch, M * sb, Y, M, N, K, stream);
 *   // or quantize once and reuse the rows: qmm_quantize_q8_0(X, xq, M, K,
 *   // stream); qmm_matmul_q8_0(W, xq, Y, M, N, K, stream);
 *   // results are ready when the stream reaches them; a device-side timeout
 *   // is read back with qmm_device_status(1).
 *
 * Pages the operations follow (cited by title and section):
 *   [minfer] "10 . CPU matmul: quantized weights x Q8_0 activations"
 *   [ggml]   "ggml Q4_0 vec_dot Walkthrough"
 *   [krafla] "Architecture"
 *   [kvad]   "kvad -- the same ideas, at scale"
 *
 * Conventions shared by every call
 *   Layout.   All buffers are little-endian, packed, with no padding.  W is
 *             row-major: N rows of qmm_row_bytes(type, K) bytes.  Activation
 *             blocks are [M][K / block_values] blocks, and outputs are fp32
 *             [M][N], token-major ([minfer] s2.3 and s3.4: out is [nt][od]).
 *   Pointers. Device pointers, owned by the caller, valid for the whole
 *             asynchronous call.  The library keeps no device memory between
 *             calls; the one allocation is the prefill's stream-ordered
 *             workspace (see "prefill matmul" below).
 *   Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *             default stream).  Calls are asynchronous on it; none synchronizes.
 *   Chaining. The matvec, linear and matmul kernels are launched as
 *             programmatic dependent launches: each lets the next kernel on
 *             the stream launch early, and may itself start streaming W before
 *             the kernel ahead of it has finished (W is read-only to every
 *             call).  Everything else it reads, and everything it writes, waits
 *             for that kernel to complete.  A kernel that writes W therefore
 *             must not both directly precede a multiply and release its
 *             dependents early (griddepcontrol.launch_dependents); ordinary
 *             kernels, and this library's weight and activation quantizers,
 *             never release early, so a multiply right after them sees all of
 *             W.
 *   Errors.   Every call returns a qmm_status.  Arguments are checked on the
 *             host before anything is launched; a failed check launches
 *             nothing.  A launch failure returns QMM_E_CUDA.  No call aborts,
 *             and no kernel traps: a device-side wait that runs out of time
 *             records QMM_E_TIMEOUT, read back with qmm_device_status().
 *   Alignment. Every base pointer must be 16-byte aligned (W, xq, x, y).
 *   Limits.   M, N, K >= 1; K a multiple of 32 (Q4_0, Q8_0) or 256 (K-quants,
 *             [minfer] s3.4: "id % 256 == 0 for K-quants"); K <= 65536;
 *             N <= 2^31 - 1; M <= 2^31 - 1.
 *   Results.  Each output element is computed by exactly one thread in a fixed
 *             order, so results are identical from run to run ([minfer] s3.3).
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMM_OK = 0,
    QMM_E_NULL = 1,     /* a required pointer is NULL */
    QMM_E_SHAPE = 2,    /* M, N or K out of range, or K not a multiple of the block */
    QMM_E_TYPE = 3,     /* unknown type code */
    QMM_E_ALIGN = 4,    /* a base pointer is not 16-byte aligned */
    QMM_E_SCRATCH = 5,  /* a caller scratch buffer is too small */
    QMM_E_CUDA = 6,     /* a CUDA runtime call or kernel launch failed */
    QMM_E_TIMEOUT = 7,  /* a bounded device wait ran out (see qmm_device_status) */
    QMM_E_BOUNDS = 8    /* a kernel index fell outside its buffer and the access was
                           skipped: only a library built with -DQMM_CHECK_BOUNDS checks */
} qmm_status;

/* Block types.  Byte sizes per block: Q4_0 18 B / 32 values, Q8_0 34 B / 32,
 * Q4_K 144 B / 256, Q6_K 210 B / 256, Q2_K 84 B / 256, Q8_K 292 B / 256
 * ([minfer] s2.3 block.rs; [ggml] s1.1 and s1.2).
 *   Q4_0: f16 d @0, qs[16] @2; byte j holds element j (low nibble) and j+16
 *         (high nibble); value d*(q-8)                              [ggml] s2
 *   Q8_0: f16 d @0, int8 qs[32] @2; value d*q                       [ggml] s1.1
 *   Q4_K: f16 d @0, f16 dmin @2, 12 B of 6-bit scales/mins @4, qs[128] @16;
 *         value d*sc_s*q - dmin*m_s per 32-value sub-block s      [minfer] s3.2
 *   Q6_K: ql[128] @0, qh[64] @128, int8 scales[16] @192, f16 d @208;
 *         value d*sc_g*(q-32) per 16-value group       (GGUF layout, a reading)
 *   Q2_K: scales[16] @0 (sc low, m high nibble), qs[64] @16, f16 d @80,
 *         f16 dmin @82; value d*sc_g*q - dmin*m_g                   [ggml] s1.2
 *   Q8_K: f32 d @0, int8 qs[256] @4, int16 bsums[16] @260 (activations only)
 * Q4_1 20 B / 32, Q5_0 22 B / 32, Q5_1 24 B / 32, Q5_K 176 B / 256 ([minfer] s1
 * and s3.2 give the 22/24/176-B sizes and that the five-bit types add a plane of
 * high bits; the byte layouts are GGUF's, a reading):
 *   Q4_1: f16 d @0, f16 m @2, qs[16] @4; value d*q + m (q the nibble)
 *   Q5_0: f16 d @0, qh[4] @2, qs[16] @6; value d*(q-16)
 *   Q5_1: f16 d @0, f16 m @2, qh[4] @4, qs[16] @8; value d*q + m
 *         (q = nibble as in Q4_0, plus bit i of the 32-bit qh as bit 4 of element i)
 *   Q5_K: f16 d @0, f16 dmin @2, scales @4 (the Q4_K packing), qh[32] @16,
 *         qs[128] @48; element 64j+l (64j+32+l) is the low (high) nibble of
 *         qs[32j+l] plus bit 2j (2j+1) of qh[l] as bit 4; value d*sc_s*q - dmin*m_s
 * Q4_1, Q5_0 and Q5_1 pair with Q8_0 activations, Q5_K with Q8_K. */
typedef enum {
    QMM_Q4_0 = 0, QMM_Q8_0 = 1, QMM_Q4_K = 2, QMM_Q6_K = 3, QMM_Q2_K = 4, QMM_Q8_K = 5,
    QMM_Q4_1 = 6, QMM_Q5_0 = 7, QMM_Q5_1 = 8, QMM_Q5_K = 9
} qmm_type;

typedef void* qmm_stream_t; /* a cudaStream_t */

/* ---- formats ------------------------------------------------------------ */
QMM_API size_t qmm_block_bytes(int type);                 /* 0 for an unknown type */
QMM_API int qmm_block_values(int type);                   /* 32 or 256; 0 for an unknown type */
QMM_API size_t qmm_row_bytes(int type, int64_t K);        /* 0 if K is not a positive multiple */
QMM_API int qmm_act_type(int wtype);                      /* QMM_Q8_0 or QMM_Q8_K: the pairing rule
                                                     of [minfer] s2.4; -1 for a bad type */
QMM_API const char* qmm_status_str(qmm_status s);         /* static string, never NULL */

/* ---- activation quantizers (hot path) ----------------------------------- */
/* [minfer] s3.2 "The activation quantizers" (quantize_row_q8_0): per 32 values
 * amax = max|x|, d = amax/127 stored as f16 (round to nearest even), inverse
 * 127/amax (0 for an all-zero block), codes = x * inverse rounded to nearest even
 * and saturated to int8.  x: f32 [M][K]; xq: [M][K/32] Q8_0 blocks (34 B each).
 * Every float operation is IEEE-rounded as written, so the codes and d are
 * bit-identical to a scalar implementation of the same steps.  Also quantizes
 * Q8_0 weights (same block, same rule). */
QMM_API qmm_status qmm_quantize_q8_0(const float* x, void* xq, int64_t M, int64_t K, qmm_stream_t stream);

/* [minfer] s3.2 (quantize_row_q8_k_buf): per 256 values amax, d = amax/127 kept
 * as f32, the same rounding with inverse 127/amax (a reading: the page's sketch
 * writes 1/d), codes saturated to [-128, 127], and bsums[g] the exact sum of the
 * 16 saturated codes of group g.  x: f32 [M][K]; xq: [M][K/256] Q8_K blocks. */
QMM_API qmm_status qmm_quantize_q8_K(const float* x, void* xq, int64_t M, int64_t K, qmm_stream_t stream);

/* ---- weight quantizers (input preparation, not on the timed path) ------- */
/* Each turns f32 weights [N][K] into N rows of blocks, with every float step
 * IEEE-rounded as written.
 *   Q4_0 ([ggml] s1.1; [kvad] "The scale that wasted a code"): m = the value of
 *     largest magnitude (first on a tie), d = m / -8 stored as f16, codes
 *     min(15, trunc(x / d + 8.5)) (x times the f32 inverse 1/d) -- m decodes as
 *     code -8, the opposite extreme clips to 7/8.
 *   Q4_K (reading): per sub-block min_s = max(0, -min x), scale_s =
 *     (max x + min_s)/15; d = max scale_s / 63, dmin = max min_s / 63 (f16);
 *     6-bit sc_s = rne(scale_s/d), m_s = rne(min_s/dmin); codes
 *     rne((x + f16(dmin)*m_s) / (f16(d)*sc_s)) in 0..15.
 *   Q2_K (reading): the same over 16 groups of 16 with /3, /15, 4-bit sc/m,
 *     codes 0..3.
 *   Q6_K (reading): per group the signed extreme m_g, s_g = m_g / -32;
 *     d = max|s_g| / 127 (f16), int8 sc_g = rne(s_g/d), codes
 *     rne(x / (f16(d)*sc_g)) in -32..31, stored +32.
 *   Q4_1, Q5_1 (reading): m = min x, d = (max x - m) / 15 (31), codes
 *     min(15 (31), trunc((x - m) * (1/d) + 0.5)); d and m stored as f16.
 *   Q5_0 (reading): the Q4_0 scheme on five bits: d = m / -16, codes
 *     min(31, trunc(x / d + 16.5)).
 *   Q5_K (reading): the Q4_K scheme with (max x + min_s)/31 and codes 0..31.
 * Q8_0 weights use qmm_quantize_q8_0. */
QMM_API qmm_status qmm_quantize_q4_0(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_quantize_q4_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_quantize_q6_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_quantize_q2_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_quantize_q4_1(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_quantize_q5_0(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_quantize_q5_1(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_quantize_q5_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream);

/* ---- decode matvec, one token (hot path) -------------------------------- */
/* y[o] = sum over blocks b of the row's block dot, folded in fp32:
 *   Q4_0, Q8_0 (x in Q8_0): y += (float)isum_b * d_w * d_x, isum_b the exact
 *     int32 code dot of block b ([minfer] s3.2 scalar kernel; [ggml] s2).
 *   Q4_K, Q2_K (x in Q8_K): per super-block, with d = d_w*d_x and
 *     dmin = dmin_w*d_x: y -= dmin*min_term; y += d*value_term, where
 *     value_term = sum of sc * (code dot) over the sub-blocks/groups and
 *     min_term = sum of m * (activation group sums from bsums)
 *     ([minfer] s3.2, the K-quant dot walked; [ggml] s1.2).
 *   Q6_K (x in Q8_K): y += (d_w*d_x) * sum_g sc_g * sum (q-32)*a (reading).
 *   Q5_0 (x in Q8_0): as Q4_0 with isum_b = sum (q-16)*a.
 *   Q4_1, Q5_1 (x in Q8_0): y += (float)isum_b * d_w * d_x + (float)asum_b *
 *     m_w * d_x, isum_b = sum q*a and asum_b the exact sum of the activation
 *     block's codes (the min meets it: sum (d q + m) a = d sum q a + m sum a).
 *   Q5_K (x in Q8_K): as Q4_K with five-bit codes.
 * W: N rows; xq: one activation row; y: f32 [N].  The fp32 fold per thread and
 * the reduction across threads follow a fixed order, which differs from a
 * left-to-right scalar sum; results agree with one within 1e-5 of the row's
 * L2 norm ([krafla] Numerics: block sums exact, float order per machine). */
QMM_API qmm_status qmm_matvec_q4_0(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q8_0(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q4_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q6_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q2_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q4_1(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q5_0(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q5_1(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_matvec_q5_K(const void* W, const void* xq, float* y, int64_t N, int64_t K, qmm_stream_t stream);

/* ---- quantize + matvec with the pairing fixed (hot path) ---------------- */
/* [minfer] s3.2 (cpu_quant_matmul_f32): the activation format is chosen by the
 * weight type in one place, so no caller can pair the wrong formats.  Quantizes
 * x (f32 [M][K]) into the caller's scratch (at least M * qmm_row_bytes(
 * qmm_act_type(wtype), K) bytes, 16-byte aligned), then computes y (f32 [M][N]).
 * A token row is quantized inside the multiply kernel (every CTA quantizes the
 * row it needs, with the same arithmetic as qmm_quantize_q8_0/q8_K, and one CTA
 * stores it to the scratch), so a token is one launch; a row too large for that
 * kernel's shared memory is quantized by the separate quantizer first.  The
 * 32-value formats (Q4_0, Q8_0, Q4_1, Q5_0, Q5_1) with M >= 8 and K % 256 == 0,
 * and Q4_K / Q6_K / Q2_K / Q5_K with M >= 8 and K % 2048 == 0, quantize all rows,
 * then run the prefill matmul (Q4_0 with 1 < M < 8 also quantizes all rows
 * first, then multiplies token by token).  Other shapes multiply token by
 * token. */
QMM_API qmm_status qmm_linear_q4_0(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q8_0(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q4_K(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q6_K(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q2_K(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q4_1(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q5_0(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q5_1(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_q5_K(const void* W, const float* x, void* xq_scratch, size_t scratch_bytes, float* y,
                           int64_t M, int64_t N, int64_t K, qmm_stream_t stream);

/* ---- quantize + multiply with host buffers -------------------------------- */
/* qmm_linear_<wtype> for a caller whose input and output live in host memory:
 * x_host (f32 [M][K]) in, y_host (f32 [M][N]) out, everything queued on the
 * stream; the caller synchronizes the stream before it reads y_host.  Results
 * equal qmm_linear_<wtype>'s bit for bit.
 *   - Both host buffers pinned (page-locked and mapped, e.g. cudaHostAlloc),
 *     16-byte aligned, and M * N <= 65536: the activation quantizer reads x_host
 *     over the host link into the scratch and the multiply writes y_host
 *     directly; x_dev and y_dev are not touched (they may be NULL).
 *   - Otherwise: x_host is copied to x_dev, qmm_linear_<wtype> runs (x_dev, the
 *     scratch and y_dev as there), and y_dev is copied back to y_host
 *     (cudaMemcpyAsync; asynchronous only when the host buffers are pinned).
 * Errors as for qmm_linear_<wtype>; QMM_E_NULL for a null host buffer (or a null
 * x_dev / y_dev on the copying path); QMM_E_CUDA when a copy cannot be queued. */
QMM_API qmm_status qmm_linear_host(int wtype, const void* W, const float* x_host, float* x_dev, void* xq_scratch,
                                   size_t scratch_bytes, float* y_dev, float* y_host, int64_t M, int64_t N, int64_t K,
                                   qmm_stream_t stream);

/* ---- quantize + multiply without a caller workspace ---------------------- */
/* No counterpart on the pages: an addition for callers that cannot give the
 * library a device buffer (a plugin inside an application that owns all device
 * memory and passes in only inputs and outputs; a loop that must never call
 * cudaMalloc, which can block on the device or fail; a fixed memory budget).
 * Same result as qmm_linear_<wtype> (wtype a QMM_Q* weight type), but the
 * quantized activation rows go to one 1 MiB array in device memory owned by the
 * library, which every GPU that loads the library keeps until the process exits.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Limit: M * qmm_row_bytes(qmm_act_type(wtype), K) <= 1 MiB (240 tokens of
 *     Q8_0 or 224 of Q8_K at K = 4096); larger calls return QMM_E_SCRATCH and
 *     launch nothing.
 *   - The first call on a device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.
 *   - Every call, on every stream, uses the same array: calls that may overlap
 *     on the GPU race with each other.  Issue them on one stream (or order them).
 *   - The array keeps the last call's contents; nothing in it needs to start at
 *     zero, because each call writes every byte it reads.
 * Errors as for qmm_linear_<wtype>, plus QMM_E_TYPE for a non-weight type. */
QMM_API qmm_status qmm_linear_noalloc(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t N,
                                      int64_t K, qmm_stream_t stream);

/* ---- several weight matrices on one input row, one launch per token ------ */
/* No counterpart on the pages: an addition for the projections of a decoder
 * layer that read the same input row (Q, K and V; gate and up).  For each of
 * the G (1..8) matrices W[g] (N[g] rows of qmm_row_bytes(wtype, K) bytes; all of
 * one weight type and K), y[g] (f32 [M][N[g]]) holds the result
 * qmm_linear_<wtype> gives for W[g] alone, bit for bit.  W, N and y are HOST
 * arrays of G entries (device pointers for W[g] and y[g]).  Where
 * qmm_linear_<wtype> runs a launch per token, the SMs are shared among the
 * matrices in proportion to their rows and each token row is quantized once per
 * CTA, so the G products cost one launch per token instead of G; where it takes
 * a tensor-core prefill (see qmm_linear_norm), the rows are quantized once and
 * each matrix gets its own prefill launch.  Scratch as for qmm_linear_<wtype>:
 * it receives the quantized rows.
 * Errors as for qmm_linear_<wtype>; QMM_E_SHAPE also for G outside 1..8;
 * QMM_E_TYPE for a non-weight type. */
QMM_API qmm_status qmm_linear_group(int wtype, int G, const void* const* W, const int64_t* N, const float* x,
                                    void* xq_scratch, size_t scratch_bytes, float* const* y, int64_t M, int64_t K,
                                    qmm_stream_t stream);

/* ---- RMSNorm fused ahead of the quantizer --------------------------------- */
/* [krafla] "Architecture", "Data flow for one token": h = rmsnorm(x) ; qa =
 * quantize_q8(h), then the matvecs that read qa.  The page gives no formula;
 * reading: h_i = (x_i * s) * w_i, s = 1 / sqrt(ss / K + eps), ss = sum of x_i^2,
 * every step an f32 operation rounded once.  The kernels sum ss in f32 in one
 * fixed order (8-value sequential partials, then a pairwise tree), so results
 * are identical run to run; that sum is within (8 + log2 K) units in the last
 * place of the exact one.  Since h and its block maximum scale together, the
 * codes agree with those of an exactly summed ss except where h_i * 127/amax
 * lies within a few roundings of a tie (there by at most 1), and each block's
 * d agrees to within that relative bound.  A model whose norm scales by 1 + w
 * passes that vector as w.
 *
 * qmm_rmsnorm_quantize: act QMM_Q8_0 or QMM_Q8_K; x f32 [M][K], w f32 [K]
 * (16-byte aligned), xq as for qmm_quantize_q8_0/q8_K; K <= 65536.
 * qmm_linear_norm: qmm_linear_group on the normed rows (G = 1 for one matrix),
 * the quantized normed rows left in the scratch.  A decode token is one launch
 * (every CTA norms and quantizes the row itself); a prefill that takes the
 * tensor-core matmul (Q4_0 with M > 1; Q8_0/Q4_1/Q5_0/Q5_1 with M >= 8 and
 * K % 256 == 0; Q4_K/Q6_K/Q2_K/Q5_K with M >= 8 and K % 2048 == 0)
 * norms and quantizes all rows first.  Errors as for qmm_linear_group, plus
 * QMM_E_NULL for w. */
QMM_API qmm_status qmm_rmsnorm_quantize(int act, const float* x, const float* w, float eps, void* xq, int64_t M,
                                        int64_t K, qmm_stream_t stream);
QMM_API qmm_status qmm_linear_norm(int wtype, int G, const void* const* W, const int64_t* N, const float* x,
                                   const float* w, float eps, void* xq_scratch, size_t scratch_bytes, float* const* y,
                                   int64_t M, int64_t K, qmm_stream_t stream);

/* ---- prefill matmul, M tokens (hot path) -------------------------------- */
/* Y[t][o] = sum_b d_w[o,b] * d_x[t,b] * isum[t,o,b] for M tokens at once: the
 * weights are read once per tile of tokens and reused across them ([krafla]
 * "Batched prompt prefill"; [kvad] "Batched prefill, and i8mm").  The integer
 * block sums run on the tensor cores with integer-valued operands (exact), and
 * each 32-wide block's sum is rescaled into fp32 by d_w*d_x.
 * W: N rows of Q4_0 (or Q8_0, Q4_1, Q5_0, Q5_1); xq: [M][K/32] Q8_0 blocks;
 * Y: f32 [M][N].  K a multiple of 256 and M >= 8 take this path; other shapes
 * run one matvec per token (same results as qmm_matvec).  Q8_0 x Q8_0 block sums
 * reach 32 * 127 * 127 < 2^24 and five-bit ones 32 * 31 * 127, exact in the fp32
 * accumulator.  Q4_1 and Q5_1 add each block's min term after its value term:
 * y += (d_w*d_x) * isum; y += m_w * (d_x * sum(a)), with sum(a) the exact
 * integer sum of the token's block codes.  Results agree with the scalar order
 * within 1e-5 of the row's L2 norm.
 * Workspace: on the tensor-core path, Q4_1 and Q5_1 here and every K-quant
 * below convert the activation once, into a workspace taken with
 * cudaMallocAsync and returned with cudaFreeAsync on `stream` (captured into a
 * CUDA graph as memory nodes): ceil(M/128) * K/256 * 73,728 bytes for Q4_1 and
 * Q5_1, * 70,144 for the K-quants (~4.7 / 4.5 MB at M = 512, K = 4096).  The
 * qmm_linear_* calls that route M >= 8 here do the same.  If the allocation
 * fails, every CTA converts the activation itself: the results are the same,
 * bit for bit.  qmm_linear_noalloc never allocates. */
QMM_API qmm_status qmm_matmul_q4_0(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
QMM_API qmm_status qmm_matmul_q8_0(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
QMM_API qmm_status qmm_matmul_q4_1(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
QMM_API qmm_status qmm_matmul_q5_0(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
QMM_API qmm_status qmm_matmul_q5_1(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
/* The same for the K-quants against Q8_K rows ([minfer] s3.2, the K-quant dot
 * walked; [ggml] s1.2).  Per 256-value super-block the integer value term
 * (sum of sc * code dots, Q6_K in two exact parts) and the integer min term
 * (f_g * bsum_g: Q4_K and Q5_K m_{g/2}, Q2_K m_g, Q6_K 32 sc_g) run on the
 * tensor cores with integer-valued operands (Q5_K: sc * q <= 63 * 31, exact in
 * fp16); each super-block then folds into fp32:
 * y -= (dmin_w*d_x) * min; y += (d_w*d_x) * value (Q4_K, Q5_K, Q2_K), or
 * y += (d_w*d_x) * (value - min) (Q6_K).  Results agree with the scalar order
 * within 1e-5 of the row's L2 norm.  K a multiple of 2048 and M >= 8 take this
 * path; other shapes run one matvec per token (same results as qmm_matvec).
 * W: N rows of the format; xq: [M][K/256] Q8_K blocks; Y: f32 [M][N]. */
QMM_API qmm_status qmm_matmul_q4_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
QMM_API qmm_status qmm_matmul_q6_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
QMM_API qmm_status qmm_matmul_q2_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);
QMM_API qmm_status qmm_matmul_q5_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream);

/* ---- embedding lookup ----------------------------------------------------- */
/* out[r][k] = value k of row ids[r] of W, dequantized ([minfer] s3.2, "The
 * embedding 'matmul'": each token id's row walked block by block, scale x code).
 * Each value is computed in f32 with at most one rounding (Q4_0 d*(n-8), Q8_0
 * d*q, Q6_K (d*sc)*(q-32), Q5_0 d*(q-16): exact; Q4_K, Q5_K and Q2_K
 * fma(d*sc, q, -(dmin*m)), Q4_1 and Q5_1 fma(d, q, m): one rounding), so it
 * equals the exact dequantized value rounded once to f32.
 * W: N rows of wtype (a weight type); ids: int32 [R] device array; out: f32
 * [R][K].  An id outside [0, N) gives a zero row and makes qmm_device_status()
 * return QMM_E_SHAPE. */
QMM_API qmm_status qmm_get_rows(int wtype, const void* W, const int32_t* ids, float* out, int64_t R, int64_t N,
                                int64_t K, qmm_stream_t stream);

/* ---- the Q8 KV cache of decode attention --------------------------------- */
/* [krafla] "Architecture", Attention ("Q8 cache"): each position's K and V are
 * kept per KV head as int8 codes with one float scale, quantized by the
 * activations' rule, and each query head is quantized the same way; a score is
 * an integer dot product, and the V sum widens the int8 values to float as it
 * goes.  Readings where the page is silent:
 *   row     one head vector of hd values: f32 d @0, int8 codes @4 (4 + hd bytes,
 *           68 at hd = 64); d = amax/127, codes rne(x * 127/amax) saturated to
 *           int8 (0 for an all-zero vector) -- over 256 values exactly a Q8_K
 *           block's d and codes
 *   cache   row (p, kvh) at byte (p*Hkv + kvh) * (4 + hd): appending position p
 *           writes Hkv consecutive rows
 *   heads   query head h reads KV head h / (Hq/Hkv) (the page's "Data flow for
 *           one token": GQA head h -> kv head h / (n_heads / n_kv_heads))
 * hd: a multiple of 16 in 16..256; Hq a multiple of Hkv with Hq/Hkv <= 8; P >= 1.
 * Pointers: 4-byte aligned (the V-sum scratch 16-byte aligned).  Errors:
 * QMM_E_NULL, QMM_E_SHAPE, QMM_E_ALIGN, QMM_E_SCRATCH, QMM_E_CUDA, as above. */
QMM_API size_t qmm_kv_row_bytes(int64_t hd);  /* 4 + hd; 0 for an unsupported hd */

/* rows head vectors x (f32 [rows][hd]) into rows quantized rows at out; the
 * codes and d are bit-identical to a scalar implementation of the rule. */
QMM_API qmm_status qmm_kv_quantize(const float* x, void* out, int64_t rows, int64_t hd, qmm_stream_t stream);

/* scores[h][p] = ((dq_h * dk_p) * isum) * scale for the Hq quantized query rows q
 * against positions 0..P-1 of the K cache kc, with isum the exact int32 dot of
 * the codes and every float step rounded once (so the result is bit-identical
 * to a scalar implementation); scale is the caller's factor (1/sqrt(hd) for
 * attention).  scores: f32 [Hq][P]. */
QMM_API qmm_status qmm_kv_scores(const void* q, const void* kc, float* scores, int64_t Hq, int64_t Hkv, int64_t P,
                                 int64_t hd, float scale, qmm_stream_t stream);

/* out[h][i] = sum_p w[h][p] * dv_p * v_p[i] over positions 0..P-1 of the V cache
 * vc, w f32 [Hq][P] (the attention weights), out f32 [Hq][hd].  Summed in f32
 * in an order fixed by P alone (an FMA chain over each 32-position chunk in
 * order, the chunk sums in the scratch, then a fixed tree), so the result is the
 * same on every GPU and within (P + 2) * 2^-24 * sum_p |w dv v| of the exact sum.
 * scratch: at least qmm_kv_wsum_scratch_bytes(Hq, P, hd) bytes. */
QMM_API size_t qmm_kv_wsum_scratch_bytes(int64_t Hq, int64_t P, int64_t hd);
QMM_API qmm_status qmm_kv_wsum(const float* w, const void* vc, float* out, void* scratch, size_t scratch_bytes,
                               int64_t Hq, int64_t Hkv, int64_t P, int64_t hd, qmm_stream_t stream);

/* ---- verification hooks (not on the hot path) --------------------------- */
/* The exact int32 block sums the kernels fold, for bit-exact checking:
 * s[t][o][b] for every token t, row o and block b; Q4_0/Q8_0 give one int32 per
 * 32-value block (sum of code products), the K-quants two per super-block:
 * (value term, min term) -- Q4_K: (sum_s sc_s*dot_s, sum_s m_s*(bsum_2s +
 * bsum_2s+1)); Q2_K: (sum_g sc_g*dot_g, sum_g m_g*bsum_g); Q6_K: (sum_g sc_g *
 * dot_g with the stored codes 0..63, sum_g sc_g*bsum_g), whose integer is
 * value - 32*min; Q5_K as Q4_K.  Q5_0 gives sum (q-16)*a per block, Q4_1 and
 * Q5_1 sum q*a (their min meets the activation's own code sum).  s: int32
 * [M][N][per-row count], computed by the matvec's per-block decode routines
 * (the super-unit decoders it takes when K % 256 == 0 are checked through
 * outputs that are exact integers instead).  One generic call for every weight
 * type, where the per-type calls of the multiply would add nine names for a
 * test hook. */
QMM_API qmm_status qmm_blocksums(int wtype, const void* W, const void* xq, int32_t* s, int64_t M, int64_t N, int64_t K,
                         qmm_stream_t stream);

/* A test of the failure path ([krafla] "Architecture", Error handling: status
 * codes, no library code aborts): launches one thread that waits, through the
 * same bounded wait every kernel here uses for its copies, on an mbarrier that
 * nothing arrives at, for limit_ns nanoseconds (clamped to 1 us .. 100 ms).  The
 * wait runs out, records QMM_E_TIMEOUT in the device error word and returns;
 * qmm_device_status() then reports QMM_E_TIMEOUT and the context stays usable.
 * Returns QMM_E_CUDA if the launch fails. */
QMM_API qmm_status qmm_test_wait_timeout(uint64_t limit_ns, qmm_stream_t stream);

/* Reads (and with clear != 0 resets) the device error words that bounded waits
 * (QMM_E_TIMEOUT), qmm_get_rows (QMM_E_SHAPE for an id outside [0, N)) and, in a
 * bounds-checked build, the kernels' index checks (QMM_E_BOUNDS) set; a timeout
 * is reported first, then a bounds record.  Synchronizes the device.  QMM_OK
 * when nothing was recorded. */
QMM_API qmm_status qmm_device_status(int clear);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */

// matmul_kq.cu -- the prefill matmul Y[M][N] for K-quant weights (Q4_K, Q2_K,
// Q6_K) x Q8_K activations, M tokens at once, on the 5th-generation tensor cores.
//
// Per 256-value super-block the pages' K-quant dot is ([minfer] "10 . CPU
// matmul: quantized weights x Q8_0 activations" s3.2, the K-quant dot walked;
// [ggml] "ggml Q4_0 vec_dot Walkthrough" s1.2):
//   value = sum_s sc_s * sum_{i in s} q_i a_i       (integer)
//   min   = sum_g f_g * bsum_g                       (integer)
//   y    += (d_w d_x) * value - (c_w d_x) * min
// with, per format, f_g and c_w:
//   Q4_K  (8 sub-blocks of 32, 6-bit sc/m)  f_g = m_{g/2},  c_w = dmin
//   Q2_K  (16 groups of 16, 4-bit sc/m)     f_g = m_g,      c_w = dmin
//   Q6_K  (16 groups of 16, int8 sc)        f_g = 32 sc_g,  c_w = d   (codes q in 0..63 stand for q - 32)
// Both integers come out of tcgen05.mma .kind::f16 exactly: the weight operand
// holds sc * q per element (Q4_K <= 63*15, Q2_K <= 15*3: exact fp16 integers;
// Q6_K's sc*q reaches 127*63, so it goes in two exact parts, sc*(q & 7) and
// 8*sc*(q >> 3)), the activation operand the int8 codes; the min term is one
// more K = 16 MMA of f_g against the 16 group sums bsum_g (|bsum_g| <= 2048,
// exact in fp16).  Each super-block's two sums land in TMEM and are folded into
// fp32 registers once per super-block by d_w*d_x and c_w*d_x, in super-block
// order, as the scalar kernel folds them.
//
// One CTA per tile of 128 weight rows x 128 tokens:
//   warp 0    TMEM allocation; one thread issues, per 32-value block, the MMAs
//             into the super-block's accumulator, and per super-block the min
//             MMA into a second accumulator (2 super-blocks in flight, 512 columns)
//   warps 1-4 weight converters, warps 5-8 activation converters: each thread
//             owns one weight row / token.  A role's super-block bytes arrive by
//             TMA, one 2-D box per super-block (128 rows x the super-block's
//             16-byte aligned superset, as 8-byte elements) in a ring of two
//             stages; after reading a stage the role's four warps meet at a
//             named barrier and one thread loads the box two super-blocks ahead
//             into it.  Each thread decodes its row and writes fp16 operands in
//             the UMMA K-major core-matrix layout, plus the min operands and scales
//   warps 9-24 epilogue: per super-block tcgen05.ld of both sums, the fp32 fold,
//             and at the end the token-major store
// With the activation pre-pass (every format, given a workspace; see
// kq_xprep_kernel) the activation converters give way to one warp that
// bulk-copies the prepared operands, and each weight row gets two threads:
// warps 1-4 convert the even groups of blocks of every super-block, warps 5-8
// the odd ones; warp 9 copies; warps 10-25 are the epilogue.
// Shapes: K a multiple of 2048 (so that every row of W and of the activation is
// a whole number of 16-byte chunks, as a TMA row pitch must be) and M >= 8;
// others run one matvec per token.
// All waits are bounded; a timeout records QMM_E_TIMEOUT, every warp still
// reaches the end, and TMEM is freed.
#include "qmm_device.cuh"
#include "qmm_host.h"
#include "tc_device.cuh"

namespace qmm {

static __device__ unsigned int g_matmul_kq_error = 0;

qmm_status matvec_dispatch(int wt, const void* W, const void* xq, float* y, int64_t N, int64_t K, cudaStream_t stream,
                           bool pdl);

namespace kq {

constexpr int BM = 128, BN = 128;
constexpr int RAWX = 304;                 // a Q8_K super-block (292 B) as whole 16-byte chunks
constexpr int SC_SLOTS = 4;               // super-blocks of scales in flight
constexpr int OP_BYTES = BM * 32 * 2;     // 8192: one 32-value block of one fp16 operand
constexpr int MIN_BYTES = BM * 16 * 2;    // 4096: one 16-value min operand
constexpr int NUM_W_WARPS = 4, NUM_EPI_WARPS = 16;
constexpr int CONV0 = 1;  // first weight-converter warp
// The activation side: four converter warps (XP false), or one warp that copies
// the operands a pre-pass kernel prepared (XP true, see kq_xprep_kernel).
template <bool XP>
struct Roles {
    // XP: two threads per weight row (8 warps); half h of them converts the groups of
    // blocks of parity h (see the converters)
    static constexpr int W_WARPS = XP ? 2 * NUM_W_WARPS : NUM_W_WARPS;
    static constexpr int X_WARPS = XP ? 1 : 4;
    static constexpr int X0 = CONV0 + W_WARPS;            // first activation warp
    static constexpr int EPI0 = X0 + X_WARPS;             // first epilogue warp
    static constexpr int THREADS = (EPI0 + NUM_EPI_WARPS) * 32;  // 800, or 832 with the pre-pass
    static constexpr int OP_FULL_WARPS = XP ? NUM_W_WARPS : NUM_W_WARPS + 4;  // arrivals per operand slot
};
// A super-block of prepared activation operands, as the pre-pass writes it (the
// kernel brings it in as two bulk copies of half of it, see XSPAN): 8 blocks of
// fp16 codes (128 tokens x 32 values in the UMMA K-major core-matrix layout),
// then the 16 group sums as fp16 in the min operand's layout.
constexpr int XP_BLOCK = BN * 32 * 2;                // 8192
constexpr int TMEM_COLS = 512;            // 2 super-blocks x (value, min) x 128 columns

template <int WT> struct Fmt;
// BB bytes per super-block, RAWW its 16-byte aligned superset, SPLIT: two
// weight operands, OP_SLOTS blocks in flight without the pre-pass (with it, see
// Slots), GROUP blocks converted together
template <> struct Fmt<QMM_Q4_K> { static constexpr int BB = 144, RAWW = 144, SPLIT = 0, OP_SLOTS = 4, GROUP = 2; };
template <> struct Fmt<QMM_Q2_K> { static constexpr int BB = 84, RAWW = 96, SPLIT = 0, OP_SLOTS = 4, GROUP = 2; };
template <> struct Fmt<QMM_Q6_K> { static constexpr int BB = 210, RAWW = 224, SPLIT = 1, OP_SLOTS = 3, GROUP = 1; };
template <> struct Fmt<QMM_Q5_K> { static constexpr int BB = 176, RAWW = 176, SPLIT = 0, OP_SLOTS = 4, GROUP = 2; };
// The weight box's row pitch in shared memory: an odd number of 16-byte chunks, so
// that the 16-byte reads of eight consecutive rows fall in eight distinct bank
// groups (Q2_K's 96 and Q6_K's 224 bytes are 6 and 14 chunks: rows r and r + 4
// collided).  The box is that wide (the bytes past the super-block's superset are
// the next one's, or the zero fill past the row).  Q6_K without the pre-pass keeps
// 224: its shared memory is full.
template <int WT, bool XP>
struct WPitch {
    static constexpr int P = WT == QMM_Q2_K ? 112 : (WT == QMM_Q6_K && XP) ? 240 : Fmt<WT>::RAWW;
    static_assert(P >= Fmt<WT>::RAWW && P % 16 == 0, "the box covers the super-block's superset");
};

constexpr int XP_BYTES = 8 * XP_BLOCK + MIN_BYTES;  // 69632
// The kernel takes a super-block's prepared operands in two bulk copies of half
// a super-block, XSPAN blocks each (the second also carries the min operand),
// through a ring of two stages of XSTAGE_BYTES.  Half stages leave the shared
// memory for more weight-operand slots (Slots).
constexpr int XSPAN = 4, XCOPIES = 8 / XSPAN;
constexpr int XSTAGE_BYTES = XSPAN * XP_BLOCK + MIN_BYTES;  // 36864
// Operand slots in flight.  With the pre-pass 12 for Q4_K and Q5_K, 8 for Q2_K
// (12 spilled more and ran slower) and 4 for Q6_K (two operands per slot): the
// converters run further ahead of the MMA issuer than with the 4 that fit beside
// whole-super-block stages (Q4_K at M = 512: 110.6 us with 4, 103.7 with 8, 102.5
// with 12).  An even number of handover barriers in every case (see the converters).
template <int WT, bool XP>
struct Slots {
    static constexpr int S = XP ? (WT == QMM_Q6_K ? 4 : WT == QMM_Q2_K ? 8 : 12) : Fmt<WT>::OP_SLOTS;
};

template <int WT, bool XP = false>
struct Layout {
    using F = Fmt<WT>;
    static constexpr int RAW_STAGE = BM * WPitch<WT, XP>::P + (XP ? 0 : BN * RAWX);
    static constexpr int OFF_RAW = 0;                                          // 2 stages
    static constexpr int S = Slots<WT, XP>::S;
    static constexpr int OFF_XP = OFF_RAW + 2 * RAW_STAGE;                     // XP: 2 stages of XSTAGE_BYTES
    static constexpr int OFF_OPA = OFF_XP + (XP ? 2 * XSTAGE_BYTES : 0);       // A (Q6_K: sc*(q&7))
    static constexpr int OFF_OPH = OFF_OPA + S * OP_BYTES;                     // Q6_K: 8*sc*(q>>3)
    static constexpr int OFF_OPB = OFF_OPH + F::SPLIT * S * OP_BYTES;          // activation codes
    static constexpr int OFF_MINA = OFF_OPB + (XP ? 0 : S * OP_BYTES);         // 2 slots of f_g
    static constexpr int OFF_MINB = OFF_MINA + 2 * MIN_BYTES;                  // 2 slots of bsum_g
    static constexpr int OFF_SCD = OFF_MINB + (XP ? 0 : 2 * MIN_BYTES);        // d_w per row
    static constexpr int OFF_SCC = OFF_SCD + SC_SLOTS * BM * 4;                // c_w per row
    static constexpr int OFF_SCX = OFF_SCC + SC_SLOTS * BM * 4;                // d_x per token
    static constexpr int OFF_BAR = OFF_SCX + (XP ? 0 : SC_SLOTS * BN * 4);
    // op_full[S] mma_done[S] acc_full[2] acc_empty[2] sc_empty[SC_SLOTS] raw_full[2 roles][2 stages]
    // x_empty[2] (XP: the MMAs of a prepared stage are done)
    static constexpr int NBARS = 2 * S + 4 + SC_SLOTS + 4 + 2;
    static constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
    static constexpr int SMEM = OFF_TMEM + 16;
};
static_assert(Layout<QMM_Q6_K>::SMEM <= 232448, "Q6_K layout exceeds shared memory");
static_assert(Layout<QMM_Q4_K>::SMEM <= 232448, "Q4_K layout exceeds shared memory");
static_assert(Layout<QMM_Q5_K>::SMEM <= 232448, "Q5_K layout exceeds shared memory");
static_assert(Layout<QMM_Q4_K, true>::SMEM <= 232448 && Layout<QMM_Q2_K, true>::SMEM <= 232448 &&
                  Layout<QMM_Q5_K, true>::SMEM <= 232448 && Layout<QMM_Q6_K, true>::SMEM <= 232448,
              "pre-pass layout exceeds shared memory");
static_assert(Layout<QMM_Q4_K, true>::OFF_OPA % 128 == 0 && Layout<QMM_Q2_K, true>::OFF_OPA % 128 == 0 &&
                  Layout<QMM_Q5_K, true>::OFF_OPA % 128 == 0 && Layout<QMM_Q6_K, true>::OFF_OPA % 128 == 0 &&
                  XSTAGE_BYTES % 128 == 0 && XP_BYTES % 128 == 0,
              "operand tiles need 128-byte alignment");

template <int WT, bool XP>
struct Bars {
    static constexpr int S = Slots<WT, XP>::S;
    uint32_t base;
    // Operand slots are handed over in groups of Fmt::GROUP blocks (the blocks a
    // converter writes together): group g of the S / GROUP groups uses barrier g.
    __device__ uint32_t op_full(int i) const { return base + 8u * i; }
    __device__ uint32_t op_empty(int i) const { return base + 8u * (S + i); }  // MMAs of the group's blocks done
    __device__ uint32_t acc_full(int i) const { return base + 8u * (2 * S + i); }
    __device__ uint32_t acc_empty(int i) const { return base + 8u * (2 * S + 2 + i); }
    __device__ uint32_t sc_empty(int i) const { return base + 8u * (2 * S + 4 + i); }
    // role `role`'s bytes (0 weights, 1 activation: a TMA box, or with the pre-pass
    // its prepared operands) landed in stage s
    __device__ uint32_t raw_full(int role, int s) const { return base + 8u * (2 * S + 4 + SC_SLOTS + 2 * role + s); }
    __device__ uint32_t x_empty(int s) const { return base + 8u * (2 * S + 4 + SC_SLOTS + 4 + s); }
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, kWaitLimitNs)) return true;
    atomicOr(&g_matmul_kq_error, kErrTimeout);
    *abort_flag = 1;
    return false;
}

// A barrier among the NTHREADS threads (whole warps) that use barrier ID
// (1..15; 0 is __syncthreads): true on every one of them if `cond` held on any.
template <int ID, int NTHREADS>
__device__ __forceinline__ bool named_bar_any(bool cond) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)cond), "n"(ID), "n"(NTHREADS)
        : "memory");
    return r != 0;
}

// Byte offset of element k (0..15) of row r in a 16-value K-major operand:
// core matrix (r/8, k/8) at ((r/8)*2 + k/8)*128.
__device__ __forceinline__ uint32_t min_off(int r, int kq) { return (uint32_t)(((r >> 3) * 2 + kq) * 128 + (r & 7) * 16); }

// fp16 bits of small integers
__device__ __forceinline__ uint32_t h2_of(int lo, int hi) {
    const __half2 h = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t hpair(int v) { return h2_of(v, v); }
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// A thread's raw super-block in shared memory: its row of the role's TMA box,
// the 16-byte chunks of the super-block's aligned superset in order.  OFF is
// the (uniform) byte offset of the super-block's first byte within chunk 0.
// The row pitches (Q4_K 144, Q5_K 176, Q8_K 304 bytes) put the 16-byte loads of
// eight consecutive rows in distinct banks; Q2_K (96) and Q6_K (224) pair them.
struct Raw {
    const uint8_t* p;  // this thread's chunk 0
    __device__ __forceinline__ uint4 chunk(int c) const { return *reinterpret_cast<const uint4*>(p + c * 16); }
};
__device__ __forceinline__ uint32_t comp(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// NW little-endian words starting at super-block byte P (P + OFF even), from
// chunks loaded here; all indices are compile-time after unrolling.
template <int OFF, int P, int NW>
__device__ __forceinline__ void words(const Raw& raw, uint32_t* out) {
    constexpr int B0 = OFF + P;                 // raw byte of the first word
    constexpr int A0 = B0 & ~3;                 // aligned word below it
    constexpr int SH = (B0 & 3) * 8;            // 0 or 16
    constexpr int NA = NW + (SH ? 1 : 0);       // aligned words needed
    constexpr int C0 = A0 / 16, C1 = (A0 + 4 * NA - 1) / 16;
    uint4 ch[C1 - C0 + 1];
#pragma unroll
    for (int c = C0; c <= C1; c++) ch[c - C0] = raw.chunk(c);
    uint32_t a[NA];
#pragma unroll
    for (int i = 0; i < NA; i++) {
        const int wb = A0 + 4 * i;
        a[i] = comp(ch[wb / 16 - C0], (wb % 16) / 4);
    }
#pragma unroll
    for (int i = 0; i < NW; i++) out[i] = SH ? __funnelshift_r(a[i], a[i + 1], SH) : a[i];
}

// 4 unsigned bytes of w (each < 1024) -> 2 fp16 pairs, times the fp16 pair s
__device__ __forceinline__ void bytes4_to_h(uint32_t w, uint32_t s, uint32_t* h01, uint32_t* h23) {
    const uint32_t m1024 = 0x64006400u;
    *h01 = h2_mul(h2_sub(bytes_to_h2(w, 0x5140), m1024), s);
    *h23 = h2_mul(h2_sub(bytes_to_h2(w, 0x7362), m1024), s);
}
// 8 words of unsigned byte codes (32 values of one block) times per-element fp16
// scale pairs (s_lo for values 0..15, s_hi for 16..31) into the operand row r
__device__ __forceinline__ void put_block(uint8_t* op, int r, const uint32_t* q, uint32_t s_lo, uint32_t s_hi) {
#pragma unroll
    for (int kq = 0; kq < 4; kq++) {  // values 8kq..8kq+7: words 2kq, 2kq+1
        const uint32_t s = kq < 2 ? s_lo : s_hi;
        uint4 v;
        bytes4_to_h(q[2 * kq], s, &v.x, &v.y);
        bytes4_to_h(q[2 * kq + 1], s, &v.z, &v.w);
        *reinterpret_cast<uint4*>(op + op_off(r, kq)) = v;
    }
}
// The same for scales sc <= 63 (Q4_K, Q5_K, Q2_K): sc * q as one fma per pair,
// (1024 + q) * sc - 1024 * sc, whose exact value q * sc < 2048 is an fp16
// integer, so the fma's one rounding leaves it exact.  c_* = -1024 * s_*.
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                              *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ void put_block_fma(uint8_t* op, int r, const uint32_t* q, int sc_lo, int sc_hi) {
    const uint32_t slo = hpair(sc_lo), shi = hpair(sc_hi);
    const uint32_t clo = hpair(-1024 * sc_lo), chi = hpair(-1024 * sc_hi);
#pragma unroll
    for (int kq = 0; kq < 4; kq++) {  // values 8kq..8kq+7: words 2kq, 2kq+1
        const uint32_t s = kq < 2 ? slo : shi, c = kq < 2 ? clo : chi;
        uint4 v;
        v.x = h2_fma(bytes_to_h2(q[2 * kq], 0x5140), s, c);
        v.y = h2_fma(bytes_to_h2(q[2 * kq], 0x7362), s, c);
        v.z = h2_fma(bytes_to_h2(q[2 * kq + 1], 0x5140), s, c);
        v.w = h2_fma(bytes_to_h2(q[2 * kq + 1], 0x7362), s, c);
        *reinterpret_cast<uint4*>(op + op_off(r, kq)) = v;
    }
}
// 16 fp16 values (as 8 pairs) into the min operand row r
__device__ __forceinline__ void put_min(uint8_t* op, int r, const uint32_t* h) {
    *reinterpret_cast<uint4*>(op + min_off(r, 0)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(op + min_off(r, 1)) = make_uint4(h[4], h[5], h[6], h[7]);
}

// ------------------------------------------------------------------ weight decoders
// Per super-block header, kept packed in registers (no arrays indexed at run
// time): the f16 d and c_w, and four words of per-group scale bytes.
struct Hdr {
    uint32_t d_bits, c_bits;  // f16 d and c_w (dmin, or d for Q6_K)
    uint32_t w0, w1, w2, w3;  // per format, see below
};
__device__ __forceinline__ uint32_t pick4(const Hdr& h, int i) { return i == 0 ? h.w0 : i == 1 ? h.w1 : i == 2 ? h.w2 : h.w3; }

// Q4_K: d@0, dmin@2, 12 bytes of 6-bit scales/mins @4 (GGUF packing, a reading), qs@16.
// w0 = sc of sub-blocks 0..3, w1 = sc 4..7, w2 = m 0..3, w3 = m 4..7 (one byte each)
template <int OFF>
__device__ __forceinline__ void hdr_q4_K(const Raw& raw, Hdr& h) {
    uint32_t w[4];
    words<OFF, 0, 4>(raw, w);
    h.d_bits = w[0] & 0xFFFFu;
    h.c_bits = w[0] >> 16;
    h.w0 = w[1] & 0x3F3F3F3Fu;
    h.w2 = w[2] & 0x3F3F3F3Fu;
    h.w1 = (w[3] & 0x0F0F0F0Fu) | ((w[1] >> 2) & 0x30303030u);
    h.w3 = ((w[3] >> 4) & 0x0F0F0F0Fu) | ((w[2] >> 2) & 0x30303030u);
}
__device__ __forceinline__ int sc_q4_K(const Hdr& h, int s) { return (int)byte_of(s < 4 ? h.w0 : h.w1, s & 3); }
__device__ __forceinline__ int f_q4_K(const Hdr& h, int g) { return (int)byte_of((g >> 1) < 4 ? h.w2 : h.w3, (g >> 1) & 3); }
// block j = sub-block j: low (j even) or high (j odd) nibbles of qs[32(j/2) .. +32]
template <int OFF>
__device__ __forceinline__ void ld_q4_K(const Raw& raw, int j, uint32_t* q) {
    switch (j >> 1) {
    case 0: words<OFF, 16, 8>(raw, q); break;
    case 1: words<OFF, 48, 8>(raw, q); break;
    case 2: words<OFF, 80, 8>(raw, q); break;
    default: words<OFF, 112, 8>(raw, q); break;
    }
}
__device__ __forceinline__ void st_q4_K(const Hdr& h, int j, uint32_t* q, uint8_t* opA, int r) {
    const int sh = (j & 1) * 4;
#pragma unroll
    for (int i = 0; i < 8; i++) q[i] = (q[i] >> sh) & 0x0F0F0F0Fu;
    put_block_fma(opA, r, q, sc_q4_K(h, j), sc_q4_K(h, j));
}

// Q5_K: the Q4_K header (d, dmin, packed scales and mins) @0, qh[32]@16,
// qs[128]@48 (GGUF layout, a reading).  Sub-block j takes the low (j even) or
// high (j odd) nibbles of qs[32(j/2) .. +32] and bit j of each qh[l] as bit 4:
// codes 0..31, so sc*q <= 63*31 is still an exact fp16 integer.
template <int OFF>
__device__ __forceinline__ void ld_q5_K(const Raw& raw, int j, uint32_t* q) {
    switch (j >> 1) {
    case 0: words<OFF, 48, 8>(raw, q); break;
    case 1: words<OFF, 80, 8>(raw, q); break;
    case 2: words<OFF, 112, 8>(raw, q); break;
    default: words<OFF, 144, 8>(raw, q); break;
    }
}
__device__ __forceinline__ void st_q5_K(const Hdr& h, int j, uint32_t* q, const uint32_t* qh, uint8_t* opA, int r) {
    const int sh = (j & 1) * 4;
#pragma unroll
    for (int i = 0; i < 8; i++) q[i] = ((q[i] >> sh) & 0x0F0F0F0Fu) | (((qh[i] >> j) & 0x01010101u) << 4);
    put_block_fma(opA, r, q, sc_q4_K(h, j), sc_q4_K(h, j));
}

// Q2_K: scales[16]@0 (sc low nibble, m high), qs[64]@16, d@80, dmin@82;
// value 128h + 32s + l is (qs[32h + l] >> 2s) & 3 (GGUF order, a reading).
// w0..w3 = the 16 scale bytes.
template <int OFF>
__device__ __forceinline__ void hdr_q2_K(const Raw& raw, Hdr& h) {
    uint32_t w[4], dd[1];
    words<OFF, 0, 4>(raw, w);
    words<OFF, 80, 1>(raw, dd);
    h.d_bits = dd[0] & 0xFFFFu;
    h.c_bits = dd[0] >> 16;
    h.w0 = w[0], h.w1 = w[1], h.w2 = w[2], h.w3 = w[3];
}
__device__ __forceinline__ int sc_q2_K(const Hdr& h, int g) { return (int)(byte_of(pick4(h, g >> 2), g & 3) & 15u); }
__device__ __forceinline__ int f_q2_K(const Hdr& h, int g) { return (int)(byte_of(pick4(h, g >> 2), g & 3) >> 4); }
template <int OFF>
__device__ __forceinline__ void ld_q2_K(const Raw& raw, int j, uint32_t* q) {
    if (j < 4) words<OFF, 16, 8>(raw, q);
    else words<OFF, 48, 8>(raw, q);
}
__device__ __forceinline__ void st_q2_K(const Hdr& h, int j, uint32_t* q, uint8_t* opA, int r) {
    const int sh = 2 * (j & 3);
#pragma unroll
    for (int i = 0; i < 8; i++) q[i] = (q[i] >> sh) & 0x03030303u;
    put_block_fma(opA, r, q, sc_q2_K(h, 2 * j), sc_q2_K(h, 2 * j + 1));
}

// Q6_K (GGUF layout, a reading): ql[128]@0, qh[64]@128, int8 scales[16]@192,
// d@208; values 128n + l, +32, +64, +96 take their low 4 bits from ql[64n+l]&15,
// ql[64n+l+32]&15, ql[64n+l]>>4, ql[64n+l+32]>>4 and their high 2 bits from
// qh[32n+l] bits 0-1, 2-3, 4-5, 6-7.  Block j = 4n + part.  w0..w3 = the 16
// int8 scales.
template <int OFF>
__device__ __forceinline__ void hdr_q6_K(const Raw& raw, Hdr& h) {
    uint32_t w[4], dd[1];
    words<OFF, 192, 4>(raw, w);
    words<OFF, 206, 1>(raw, dd);  // bytes 206..209: d in the high half (no read past byte 209)
    h.d_bits = dd[0] >> 16;
    h.c_bits = h.d_bits;
    h.w0 = w[0], h.w1 = w[1], h.w2 = w[2], h.w3 = w[3];
}
__device__ __forceinline__ int sc_q6_K(const Hdr& h, int g) { return (int)(int8_t)byte_of(pick4(h, g >> 2), g & 3); }
template <int OFF>
__device__ __forceinline__ void ld_q6_K(const Raw& raw, int j, uint32_t* ql, uint32_t* qh) {
    switch (j) {  // ql run: 64n + 32*(part & 1); qh run: 128 + 32n
    case 0: case 2: words<OFF, 0, 8>(raw, ql); words<OFF, 128, 8>(raw, qh); break;
    case 1: case 3: words<OFF, 32, 8>(raw, ql); words<OFF, 128, 8>(raw, qh); break;
    case 4: case 6: words<OFF, 64, 8>(raw, ql); words<OFF, 160, 8>(raw, qh); break;
    default: words<OFF, 96, 8>(raw, ql); words<OFF, 160, 8>(raw, qh); break;
    }
}
__device__ __forceinline__ void st_q6_K(const Hdr& h, int j, const uint32_t* ql, const uint32_t* qh, uint8_t* opA,
                                        uint8_t* opH, int r) {
    const int part = j & 3;
    const int lsh = (part >> 1) * 4, hsh = 2 * part;
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const uint32_t q = ((ql[i] >> lsh) & 0x0F0F0F0Fu) | (((qh[i] >> hsh) & 0x03030303u) << 4);  // 0..63
        lo[i] = q & 0x07070707u;
        hi[i] = (q >> 3) & 0x07070707u;
    }
    const int s0 = sc_q6_K(h, 2 * j), s1 = sc_q6_K(h, 2 * j + 1);
    put_block(opA, r, lo, hpair(s0), hpair(s1));
    put_block(opH, r, hi, hpair(8 * s0), hpair(8 * s1));
}

// the min operand f_g of a weight row, as 8 fp16 pairs
template <int WT>
__device__ __forceinline__ void min_row(const Hdr& h, uint32_t* hv) {
#pragma unroll
    for (int i = 0; i < 8; i++) {
        if constexpr (WT == QMM_Q4_K || WT == QMM_Q5_K) hv[i] = h2_of(f_q4_K(h, 2 * i), f_q4_K(h, 2 * i + 1));
        else if constexpr (WT == QMM_Q2_K) hv[i] = h2_of(f_q2_K(h, 2 * i), f_q2_K(h, 2 * i + 1));
        else hv[i] = h2_of(32 * sc_q6_K(h, 2 * i), 32 * sc_q6_K(h, 2 * i + 1));
    }
}

// ------------------------------------------------------------------ activation decoder
// Q8_K: f32 d@0, int8 qs[256]@4, int16 bsums[16]@260
template <int OFF>
__device__ __forceinline__ void ld_x(const Raw& raw, int j, uint32_t* q) {
    switch (j) {
    case 0: words<OFF, 4, 8>(raw, q); break;
    case 1: words<OFF, 36, 8>(raw, q); break;
    case 2: words<OFF, 68, 8>(raw, q); break;
    case 3: words<OFF, 100, 8>(raw, q); break;
    case 4: words<OFF, 132, 8>(raw, q); break;
    case 5: words<OFF, 164, 8>(raw, q); break;
    case 6: words<OFF, 196, 8>(raw, q); break;
    default: words<OFF, 228, 8>(raw, q); break;
    }
}
__device__ __forceinline__ void st_x(const uint32_t* q, uint8_t* opB, int r) {
    const uint32_t m1152 = 0x64806480u;  // 1024 + (a + 128) - 1152 = a
#pragma unroll
    for (int kq = 0; kq < 4; kq++) {
        const uint32_t w0 = q[2 * kq] ^ 0x80808080u, w1 = q[2 * kq + 1] ^ 0x80808080u;
        uint4 v;
        v.x = h2_sub(bytes_to_h2(w0, 0x5140), m1152);
        v.y = h2_sub(bytes_to_h2(w0, 0x7362), m1152);
        v.z = h2_sub(bytes_to_h2(w1, 0x5140), m1152);
        v.w = h2_sub(bytes_to_h2(w1, 0x7362), m1152);
        *reinterpret_cast<uint4*>(opB + op_off(r, kq)) = v;
    }
}
template <int OFF>
__device__ __forceinline__ void hdr_x(const Raw& raw, uint32_t* d_bits, uint32_t* bs /* 8 words */) {
    uint32_t w[1];
    words<OFF, 0, 1>(raw, w);
    *d_bits = w[0];
    words<OFF, 260, 8>(raw, bs);
}

// ------------------------------------------------------------------ the activation pre-pass
// Every CTA of a token tile converts the same Q8_K rows, so with a workspace
// they are converted once: CTA (sb, ty) writes super-block sb of token tile ty
// as XP_BYTES of prepared operands -- for each of its 8 blocks the fp16 codes of
// the tile's 128 tokens in the core-matrix layout the MMA reads, then the 16
// group sums as fp16 -- and the tile's 128 scales d_x to dxg.  One thread per
// token; tokens past M get zeros.  The same conversion as the in-kernel path
// (st_x, the bsum pairs), so the operands are the same bits.
__global__ void __launch_bounds__(BN) kq_xprep_kernel(const uint8_t* __restrict__ xq, uint8_t* __restrict__ xp,
                                                      float* __restrict__ dxg, int M, int nsb, int pdl) {
    if (pdl) pdl_launch_dependents();
    if (pdl) pdl_wait();  // the rows come from the previous kernel
    const int r = threadIdx.x, sb = blockIdx.x, ty = blockIdx.y;
    const int t = ty * BN + r;
    const size_t unit = (size_t)ty * nsb + sb;
    uint8_t* out = xp + unit * XP_BYTES;
    const bool real = t < M && QMM_IN_BOUNDS(g_matmul_kq_error, t, M);
    const uint32_t* row = reinterpret_cast<const uint32_t*>(xq + ((size_t)(real ? t : 0) * nsb + sb) * 292);
#pragma unroll 2
    for (int j = 0; j < 8; j++) {  // block j: code words 1 + 8j .. 8 + 8j
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; i++) q[i] = real ? row[1 + 8 * j + i] : 0x00000000u;
        st_x(q, out + j * XP_BLOCK, r);
    }
    uint32_t hv[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const uint32_t bp = real ? row[65 + i] : 0u;  // the bsum pair of groups 2i, 2i + 1
        hv[i] = h2_of((int)(int16_t)(bp & 0xFFFFu), (int)(int16_t)(bp >> 16));
    }
    put_min(out + 8 * XP_BLOCK, r, hv);
    dxg[unit * BN + r] = real ? __uint_as_float(row[0]) : 0.0f;
}

// ------------------------------------------------------------------ the kernel
// XP: the activation operands come prepared by kq_xprep_kernel (xp, and the
// scales d_x in dxg); otherwise xmap's raw Q8_K rows are converted here.
template <int WT, bool XP>
__global__ void __launch_bounds__(Roles<XP>::THREADS, 1)
    matmul_kq_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                     const uint8_t* __restrict__ xp, const float* __restrict__ dxg, float* __restrict__ Y, int M,
                     int N, int K, int pdl) {
    using F = Fmt<WT>;
    using L = Layout<WT, XP>;
    using R = Roles<XP>;
    constexpr int S = Slots<WT, XP>::S;
    if (pdl) pdl_launch_dependents();
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 127u) {  // operand tiles need 128-byte alignment
        if (threadIdx.x == 0) atomicOr(&g_matmul_kq_error, kErrTimeout);
        return;
    }
    const Bars<WT, XP> bars{sbase + L::OFF_BAR};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_TMEM + 8);
    float* scd = reinterpret_cast<float*>(smem + L::OFF_SCD);
    float* scc = reinterpret_cast<float*>(smem + L::OFF_SCC);
    float* scx = reinterpret_cast<float*>(smem + L::OFF_SCX);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BM, t0 = blockIdx.y * BN;
    const int nsb = K / 256;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(bars.op_full(i), R::OP_FULL_WARPS);
            mbar_init(bars.op_empty(i), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bars.acc_full(i), 1);
            mbar_init(bars.acc_empty(i), NUM_EPI_WARPS);
        }
        for (int i = 0; i < SC_SLOTS; i++) mbar_init(bars.sc_empty(i), NUM_EPI_WARPS);
        for (int i = 0; i < 4; i++) mbar_init(bars.raw_full(i >> 1, i & 1), 1);
        for (int i = 0; i < 2; i++) mbar_init(bars.x_empty(i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc_f16(BM, BN);
            const uint64_t a0 = smem_desc(sbase + L::OFF_OPA, 128, 512);
            const uint64_t h0 = smem_desc(sbase + L::OFF_OPH, 128, 512);
            const uint64_t b0 = smem_desc(sbase + L::OFF_OPB, 128, 512);
            const uint64_t ma0 = smem_desc(sbase + L::OFF_MINA, 128, 256);
            const uint64_t mb0 = smem_desc(sbase + L::OFF_MINB, 128, 256);
            for (int sb = 0; sb < nsb; sb++) {
                const int as = sb & 1;
                if (sb >= 2 && !wait_or_abort(bars.acc_empty(as), ((sb >> 1) - 1) & 1, abort_flag)) break;
                const uint32_t dv = tmem + (uint32_t)(as * 128), dm = tmem + (uint32_t)(256 + as * 128);
                bool ok = true;
                constexpr int G = F::GROUP, NG = S / G;  // blocks handed over together, groups of slots
                // unrolled: the issuing thread is on the critical path (a rolled loop made the
                // Q4_K prefill 1.4x slower)
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int b = sb * 8 + j, os = b % S;
                    const int gi = b / G, gs = gi % NG;  // the block's group and its barrier
                    // XP: copy xc of the prepared activation operands holds block j, in stage xc & 1
                    const int xc = sb * XCOPIES + j / XSPAN;
                    if (XP && j % XSPAN == 0 && !wait_or_abort(bars.raw_full(1, xc & 1), (xc >> 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (b % G == 0 && !wait_or_abort(bars.op_full(gs), (gi / NG) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xs = sbase + L::OFF_XP + (uint32_t)((xc & 1) * XSTAGE_BYTES);
                    const uint64_t so = (uint64_t)(os * (OP_BYTES >> 4));
                    const uint64_t bj = XP ? smem_desc(xs + (uint32_t)((j % XSPAN) * XP_BLOCK), 128, 512) : b0 + so;
                    mma_f16(dv, a0 + so, bj, idesc, j > 0 ? 1u : 0u);
                    mma_f16(dv, a0 + so + (256 >> 4), bj + (256 >> 4), idesc, 1u);
                    if (F::SPLIT) {
                        mma_f16(dv, h0 + so, bj, idesc, 1u);
                        mma_f16(dv, h0 + so + (256 >> 4), bj + (256 >> 4), idesc, 1u);
                    }
                    if (j == 7) {
                        const uint64_t mo = (uint64_t)(as * (MIN_BYTES >> 4));
                        const uint64_t mb = XP ? smem_desc(xs + (uint32_t)(XSPAN * XP_BLOCK), 128, 256) : mb0 + mo;
                        mma_f16(dm, ma0 + mo, mb, idesc, 0u);
                    }
                    if (b % G == G - 1) mma_commit(bars.op_empty(gs));  // the group's slots may be refilled
                    if (j == 7) mma_commit(bars.acc_full(as));
                    if (XP && j % XSPAN == XSPAN - 1) mma_commit(bars.x_empty(xc & 1));  // the stage may be refilled
                }
                if (!ok) break;
            }
        }
    } else if (XP && warp == R::X0) {
        // ------------------------------------------------------------ prepared activation operands
        if (lane == 0) {
            if (pdl) pdl_wait();  // the pre-pass kernel wrote them
            const uint8_t* src = xp + (size_t)blockIdx.y * nsb * XP_BYTES;
            for (int xc = 0; xc < nsb * XCOPIES; xc++) {
                // copy xc: part xc % XCOPIES of super-block xc / XCOPIES, into stage xc & 1
                const int sb = xc / XCOPIES, part = xc % XCOPIES, s = xc & 1;
                // the prepared units are gridDim.y token tiles x nsb super-blocks
                if (!QMM_IN_BOUNDS(g_matmul_kq_error, (int64_t)blockIdx.y * nsb + sb, (int64_t)gridDim.y * nsb)) break;
                if (xc >= 2 && !wait_or_abort(bars.x_empty(s), ((xc >> 1) - 1) & 1, abort_flag)) break;
                // XSPAN blocks of codes, and after the last of them the min operand
                const uint32_t bytes = (uint32_t)(XSPAN * XP_BLOCK + (part == XCOPIES - 1 ? MIN_BYTES : 0));
                mbar_arrive_expect_tx(bars.raw_full(1, s), bytes);
                // every CTA of this token tile reads the same bytes: no eviction hint
                bulk_g2s_nohint(sbase + L::OFF_XP + (uint32_t)(s * XSTAGE_BYTES),
                                src + (size_t)sb * XP_BYTES + (size_t)part * XSPAN * XP_BLOCK, bytes, bars.raw_full(1, s));
            }
        }
    } else if (warp < R::EPI0) {
        // ------------------------------------------------------------ converters
        const bool is_w = XP || warp < R::X0;
        const int role = is_w ? 0 : 1;
        // XP: half h converts every other group of blocks, those with gi % 2 == h.  Group
        // gi fills slots and hands over on barrier gi % NG (NG = S / G, even), so each
        // barrier is used by one half only and every one of its phases is waited on by
        // that half, in order.  A parity wait is only right while the barrier is at most
        // one phase away from it; a barrier shared by the halves, each waiting only on its
        // own phases, could be two phases on and alias.
        static_assert(!XP || ((S / F::GROUP) % 2 == 0 && 8 % (2 * F::GROUP) == 0),
                      "with the pre-pass each operand barrier belongs to one converter half");
        const int half = XP ? (warp - CONV0) / NUM_W_WARPS : 0;
        const int r = (is_w ? (warp - CONV0) % NUM_W_WARPS : warp - R::X0) * 32 + lane;  // row or token
        const int j_begin = XP ? F::GROUP * half : 0, j_step = XP ? 2 * F::GROUP : F::GROUP;
        if (!is_w && pdl) pdl_wait();  // the activation comes from the previous kernel
        const int BBs = is_w ? F::BB : 292;
        const int pitch = is_w ? WPitch<WT, XP>::P : RAWX;  // the box's row pitch in shared memory
        const uint32_t raw_role = is_w ? 0u : (uint32_t)(BM * WPitch<WT, XP>::P);
        // super-block sb of the role's 128 rows into stage sb & 1 (one thread of the role):
        // the box starts at the 16-byte boundary at or below the super-block's first byte
        auto load = [&](int sb) {
            const uint32_t bar = bars.raw_full(role, sb & 1);
            const uint32_t dst = sbase + L::OFF_RAW + (uint32_t)((sb & 1) * L::RAW_STAGE) + raw_role;
            const int x = (int)((((uint64_t)sb * BBs) & ~15ull) / 8);  // in 8-byte elements: a 16-byte multiple
            fence_proxy_async_smem();  // the stage's previous bytes were read through the generic proxy
            mbar_arrive_expect_tx(bar, (uint32_t)(128 * pitch));
            if (is_w) tma_load_2d(dst, &wmap, x, o0, bar);
            else tma_load_2d(dst, &xmap, x, t0, bar);
        };
        if (r == 0 && half == 0) {
            load(0);
            if (nsb > 1) load(1);
        }
        for (int sb = 0; sb < nsb; sb++) {
            bool ok = wait_or_abort(bars.raw_full(role, sb & 1), (sb >> 1) & 1, abort_flag);
            const Raw raw{smem + L::OFF_RAW + (sb & 1) * L::RAW_STAGE + raw_role + r * pitch};
            const int off = (int)(((uint64_t)sb * BBs) & 15u);
            const int ss = sb % SC_SLOTS, as = sb & 1;
            if (ok && half == 0 && sb >= SC_SLOTS &&
                !wait_or_abort(bars.sc_empty(ss), ((sb / SC_SLOTS) - 1) & 1, abort_flag))
                ok = false;
            if (ok) {
                Hdr h;
                uint32_t xd = 0, bs[8];
                if (is_w) {
                    if constexpr (WT == QMM_Q4_K || WT == QMM_Q5_K) {
                        hdr_q4_K<0>(raw, h);
                    } else if constexpr (WT == QMM_Q2_K) {
                        switch (off) {
                        case 0: hdr_q2_K<0>(raw, h); break;
                        case 4: hdr_q2_K<4>(raw, h); break;
                        case 8: hdr_q2_K<8>(raw, h); break;
                        default: hdr_q2_K<12>(raw, h); break;
                        }
                    } else {
                        switch (off) {
                        case 0: hdr_q6_K<0>(raw, h); break;
                        case 2: hdr_q6_K<2>(raw, h); break;
                        case 4: hdr_q6_K<4>(raw, h); break;
                        case 6: hdr_q6_K<6>(raw, h); break;
                        case 8: hdr_q6_K<8>(raw, h); break;
                        case 10: hdr_q6_K<10>(raw, h); break;
                        case 12: hdr_q6_K<12>(raw, h); break;
                        default: hdr_q6_K<14>(raw, h); break;
                        }
                    }
                    if (half == 0) {
                        scd[ss * BM + r] = h2f(h.d_bits);
                        scc[ss * BM + r] = h2f(h.c_bits);
                    }
                } else {
                    switch (off) {
                    case 0: hdr_x<0>(raw, &xd, bs); break;
                    case 4: hdr_x<4>(raw, &xd, bs); break;
                    case 8: hdr_x<8>(raw, &xd, bs); break;
                    default: hdr_x<12>(raw, &xd, bs); break;
                    }
                    scx[ss * BN + r] = __uint_as_float(xd);
                }
                // blocks in groups of G: all of a group's loads are issued before its
                // stores, so the group's decode chains overlap
                constexpr int G = F::GROUP;
                for (int jg = j_begin; jg < 8; jg += j_step) {
                    int osl[G];
#pragma unroll
                    for (int u = 0; u < G; u++) osl[u] = (sb * 8 + jg + u) % S;
                    // the group's slots, one barrier for all of them (last used NG groups ago)
                    const int gi = (sb * 8 + jg) / G, gs = gi % (S / G);
                    if (gi >= S / G && !wait_or_abort(bars.op_empty(gs), ((gi / (S / G)) - 1) & 1, abort_flag))
                        ok = false;
                    if (!ok) break;
                    if (is_w) {
                        if constexpr (WT == QMM_Q6_K) {
                            uint32_t ql[G][8], qh[G][8];
#pragma unroll
                            for (int u = 0; u < G; u++) {
                                switch (off) {
                                case 0: ld_q6_K<0>(raw, jg + u, ql[u], qh[u]); break;
                                case 2: ld_q6_K<2>(raw, jg + u, ql[u], qh[u]); break;
                                case 4: ld_q6_K<4>(raw, jg + u, ql[u], qh[u]); break;
                                case 6: ld_q6_K<6>(raw, jg + u, ql[u], qh[u]); break;
                                case 8: ld_q6_K<8>(raw, jg + u, ql[u], qh[u]); break;
                                case 10: ld_q6_K<10>(raw, jg + u, ql[u], qh[u]); break;
                                case 12: ld_q6_K<12>(raw, jg + u, ql[u], qh[u]); break;
                                default: ld_q6_K<14>(raw, jg + u, ql[u], qh[u]); break;
                                }
                            }
#pragma unroll
                            for (int u = 0; u < G; u++)
                                st_q6_K(h, jg + u, ql[u], qh[u], smem + L::OFF_OPA + osl[u] * OP_BYTES,
                                        smem + L::OFF_OPH + osl[u] * OP_BYTES, r);
                        } else if constexpr (WT == QMM_Q5_K) {
                            uint32_t q[G][8], qh[8];
                            words<0, 16, 8>(raw, qh);  // the fifth bits of every sub-block
#pragma unroll
                            for (int u = 0; u < G; u++) ld_q5_K<0>(raw, jg + u, q[u]);
#pragma unroll
                            for (int u = 0; u < G; u++)
                                st_q5_K(h, jg + u, q[u], qh, smem + L::OFF_OPA + osl[u] * OP_BYTES, r);
                        } else {
                            uint32_t q[G][8];
#pragma unroll
                            for (int u = 0; u < G; u++) {
                                if constexpr (WT == QMM_Q4_K) {
                                    ld_q4_K<0>(raw, jg + u, q[u]);
                                } else {
                                    switch (off) {
                                    case 0: ld_q2_K<0>(raw, jg + u, q[u]); break;
                                    case 4: ld_q2_K<4>(raw, jg + u, q[u]); break;
                                    case 8: ld_q2_K<8>(raw, jg + u, q[u]); break;
                                    default: ld_q2_K<12>(raw, jg + u, q[u]); break;
                                    }
                                }
                            }
#pragma unroll
                            for (int u = 0; u < G; u++) {
                                if constexpr (WT == QMM_Q4_K)
                                    st_q4_K(h, jg + u, q[u], smem + L::OFF_OPA + osl[u] * OP_BYTES, r);
                                else st_q2_K(h, jg + u, q[u], smem + L::OFF_OPA + osl[u] * OP_BYTES, r);
                            }
                        }
                    } else {
                        uint32_t q[G][8];
#pragma unroll
                        for (int u = 0; u < G; u++) {
                            switch (off) {
                            case 0: ld_x<0>(raw, jg + u, q[u]); break;
                            case 4: ld_x<4>(raw, jg + u, q[u]); break;
                            case 8: ld_x<8>(raw, jg + u, q[u]); break;
                            default: ld_x<12>(raw, jg + u, q[u]); break;
                            }
                        }
#pragma unroll
                        for (int u = 0; u < G; u++) st_x(q[u], smem + L::OFF_OPB + osl[u] * OP_BYTES, r);
                    }
                    if (jg + G == 8) {
                        // the min operands of this super-block; their slot was last read by
                        // the min MMA of super-block sb - 2, complete once its acc_full fired
                        if (sb >= 2 && !wait_or_abort(bars.acc_full(as), ((sb - 2) >> 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint32_t hv[8];
                        if (is_w) {
                            min_row<WT>(h, hv);
                            put_min(smem + L::OFF_MINA + as * MIN_BYTES, r, hv);
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; i++)
                                hv[i] = h2_of((int)(int16_t)(bs[i] & 0xFFFFu), (int)(int16_t)(bs[i] >> 16));
                            put_min(smem + L::OFF_MINB + as * MIN_BYTES, r, hv);
                        }
                    }
                    fence_proxy_async_smem();  // the operands are read by the tensor core (async proxy)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.op_full(gi % (S / G)));
                }
            }
            // Every thread of the role has read this stage: one of them refills it.  The
            // barrier also makes the decision to stop the same on all of the role's threads
            // (128, or 256 weight threads with the pre-pass), so none is left waiting at a
            // later barrier.
            const bool stop = !ok || *abort_flag;
            if (is_w ? (XP ? named_bar_any<1, 256>(stop) : named_bar_any<1, 128>(stop)) : named_bar_any<2, 128>(stop))
                break;
            if (r == 0 && half == 0 && sb + 2 < nsb) load(sb + 2);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = warp - R::EPI0;
        if (XP && pdl) pdl_wait();  // d_x comes from the pre-pass kernel
        const int quad = warp & 3, cg = e >> 2;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(cg * 32);
        uint64_t acc[16];
#pragma unroll
        for (int j = 0; j < 16; j++) acc[j] = 0;
        for (int sb = 0; sb < nsb; sb++) {
            const int as = sb & 1, ss = sb % SC_SLOTS;
            if (!wait_or_abort(bars.acc_full(as), (sb >> 1) & 1, abort_flag)) break;
            tc_fence_after();
            const float dw = scd[ss * BM + row], cw = scc[ss * BM + row];
            const uint64_t dw2 = f2_pack(__float_as_uint(dw), __float_as_uint(dw));
            const uint64_t cw2 = f2_pack(__float_as_uint(-cw), __float_as_uint(-cw));
            const uint64_t* dxs =
                XP ? reinterpret_cast<const uint64_t*>(dxg + ((size_t)blockIdx.y * nsb + sb) * BN + cg * 32)
                   : reinterpret_cast<const uint64_t*>(scx + ss * BN + cg * 32);
#pragma unroll
            for (int qq = 0; qq < 4; qq++) {  // 8 columns at a time
                uint32_t v[8], m[8];
                tmem_ld8(lane_base + (uint32_t)(as * 128 + 8 * qq), v);
                tmem_ld8(lane_base + (uint32_t)(256 + as * 128 + 8 * qq), m);
                tmem_ld_wait();
                if (qq == 3) {  // both sums are in registers: the accumulators may be reused
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.acc_empty(as));
                }
#pragma unroll
                for (int jj = 0; jj < 4; jj++) {
                    const uint64_t dx = dxs[4 * qq + jj];
                    uint64_t& a = acc[4 * qq + jj];
                    if constexpr (WT == QMM_Q6_K) {
                        // one scale for both sums: the exact integer value - 32*min first
                        const float a0 = __uint_as_float(v[2 * jj]) - __uint_as_float(m[2 * jj]);
                        const float a1 = __uint_as_float(v[2 * jj + 1]) - __uint_as_float(m[2 * jj + 1]);
                        a = f2_fma(f2_pack(__float_as_uint(a0), __float_as_uint(a1)), f2_mul(dw2, dx), a);
                    } else {
                        // the pages' order: subtract the min term, then add the value term
                        a = f2_fma(f2_pack(m[2 * jj], m[2 * jj + 1]), f2_mul(cw2, dx), a);
                        a = f2_fma(f2_pack(v[2 * jj], v[2 * jj + 1]), f2_mul(dw2, dx), a);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.sc_empty(ss));
        }
        if (pdl) pdl_wait();  // Y may be read or written by the previous kernel
        const int o = o0 + row;
        if (!*abort_flag && o < N) {
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const int t = t0 + cg * 32 + j;
                const uint32_t bits = (j & 1) ? (uint32_t)(acc[j >> 1] >> 32) : (uint32_t)acc[j >> 1];
                if (t < M && QMM_IN_BOUNDS(g_matmul_kq_error, (size_t)t * N + o, (size_t)M * N))
                    Y[(size_t)t * N + o] = __uint_as_float(bits);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace kq
}  // namespace qmm

// ------------------------------------------------------------------ host side
namespace qmm {

// The tensor-core path needs every row of W and of the activation to be whole
// 16-byte chunks (K a multiple of 2048) and enough tokens to fill a tile
// reasonably; other shapes run one matvec per token.
static bool kq_tensor_core_shape(int64_t M, int64_t K) { return K % 2048 == 0 && M >= 8; }

// One launch of the tensor-core kernel; XP: the activation operands were prepared
// into xp / dxg by kq_xprep_kernel (xq is then not read).
template <int WT, bool XP>
static qmm_status launch_kq_kernel(const void* W, const void* xq, const uint8_t* xp, const float* dxg, float* Y,
                                   int64_t M, int64_t N, int64_t K, cudaStream_t stream, bool pdl) {
    using L = kq::Layout<WT, XP>;
    using F = kq::Fmt<WT>;
    // the rows of W and of the activation as TMA maps of 8-byte elements; a box is
    // one super-block's 16-byte aligned superset of 128 rows (tokens)
    const uint64_t nsb = (uint64_t)(K / 256);
    CUtensorMap wmap, xmap;
    if (!make_row_map(&wmap, W, nsb * F::BB, (uint64_t)N, kq::WPitch<WT, XP>::P, 8)) return QMM_E_CUDA;
    if (XP) {
        xmap = CUtensorMap{};  // not read
    } else if (!make_row_map(&xmap, xq, nsb * 292, (uint64_t)M, kq::RAWX, 8)) {
        return QMM_E_CUDA;
    }
    static PerDeviceOnce attr_once;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_E_CUDA;
    const qmm_status ast = attr_once.run(dev, [] {
        return cudaFuncSetAttribute(kq::matmul_kq_kernel<WT, XP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    L::SMEM) == cudaSuccess
                   ? QMM_OK
                   : QMM_E_CUDA;
    });
    if (ast != QMM_OK) return ast;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + kq::BM - 1) / kq::BM), (unsigned)((M + kq::BN - 1) / kq::BN));
    cfg.blockDim = dim3(kq::Roles<XP>::THREADS);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kq::matmul_kq_kernel<WT, XP>, wmap, xmap, xp, dxg, Y, (int)M, (int)N,
                                             (int)K, pdl ? 1 : 0);
    return e == cudaSuccess ? QMM_OK : QMM_E_CUDA;
}

// Set while qmm_linear_noalloc runs on this thread: its callers must not see an
// allocation, so the prefill converts the activation in the kernel itself.
thread_local bool tl_no_workspace_alloc = false;

// The activation is converted once, in a pre-pass, into a stream-ordered
// workspace (cudaMallocAsync / cudaFreeAsync on the caller's stream: ~4.4 MB for
// 512 tokens at K = 4096); without one (no pool memory, or inside
// qmm_linear_noalloc) every CTA converts it.
template <int WT>
static qmm_status launch_kq(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                            cudaStream_t stream, bool pdl) {
    if (!tl_no_workspace_alloc) {
        const int64_t ntt = (M + kq::BN - 1) / kq::BN, nsb = K / 256;
        const size_t xp_bytes = (size_t)(ntt * nsb) * kq::XP_BYTES;
        const size_t dx_bytes = (size_t)(ntt * nsb) * kq::BN * sizeof(float);
        void* buf = nullptr;
        if (ntt * nsb <= 0x7FFFFFFF && cudaMallocAsync(&buf, xp_bytes + dx_bytes, stream) == cudaSuccess) {
            uint8_t* xp = static_cast<uint8_t*>(buf);
            float* dxg = reinterpret_cast<float*>(xp + xp_bytes);
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)nsb, (unsigned)ntt);
            cfg.blockDim = dim3(kq::BN);
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = pdl ? 1 : 0;
            qmm_status st = cudaLaunchKernelEx(&cfg, kq::kq_xprep_kernel, (const uint8_t*)xq, xp, dxg, (int)M,
                                               (int)nsb, pdl ? 1 : 0) == cudaSuccess
                                ? QMM_OK
                                : QMM_E_CUDA;
            if (st == QMM_OK) st = launch_kq_kernel<WT, true>(W, xq, xp, dxg, Y, M, N, K, stream, true);
            if (cudaFreeAsync(buf, stream) != cudaSuccess && st == QMM_OK) st = QMM_E_CUDA;
            return st;
        }
        (void)cudaGetLastError();  // no workspace: convert in the kernel
    }
    return launch_kq_kernel<WT, false>(W, xq, nullptr, nullptr, Y, M, N, K, stream, pdl);
}

bool kq_uses_tensor_cores(int wt, int64_t M, int64_t K);

// Y[M][N] for a K-quant W against M Q8_K rows (internal: arguments checked).
qmm_status matmul_kq_launch(int wt, const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                            cudaStream_t stream, bool pdl) {
    if (!kq_uses_tensor_cores(wt, M, K)) {  // per token: small M, ragged K, or no tensor-core kernel
        const size_t xrb = row_bytes_of(QMM_Q8_K, K);
        for (int64_t t = 0; t < M; t++) {
            qmm_status st = matvec_dispatch(wt, W, (const uint8_t*)xq + t * xrb, Y + t * N, N, K, stream, pdl);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    if ((N + kq::BM - 1) / kq::BM > 0x7FFFFFFF || (M + kq::BN - 1) / kq::BN > 65535) return QMM_E_SHAPE;
    switch (wt) {
    case QMM_Q4_K: return launch_kq<QMM_Q4_K>(W, xq, Y, M, N, K, stream, pdl);
    case QMM_Q2_K: return launch_kq<QMM_Q2_K>(W, xq, Y, M, N, K, stream, pdl);
    case QMM_Q6_K: return launch_kq<QMM_Q6_K>(W, xq, Y, M, N, K, stream, pdl);
    case QMM_Q5_K: return launch_kq<QMM_Q5_K>(W, xq, Y, M, N, K, stream, pdl);
    default: return QMM_E_TYPE;
    }
}

bool kq_uses_tensor_cores(int wt, int64_t M, int64_t K) {
    return (wt == QMM_Q4_K || wt == QMM_Q2_K || wt == QMM_Q6_K || wt == QMM_Q5_K) && kq_tensor_core_shape(M, K);
}

static qmm_status matmul_kq_checked(int wt, const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                                    qmm_stream_t stream) {
    if (!W || !xq || !Y) return QMM_E_NULL;
    qmm_status st = check_shape(wt, M, N, K);
    if (st != QMM_OK) return st;
    if (!aligned16(W) || !aligned16(xq) || !aligned16(Y)) return QMM_E_ALIGN;
    return matmul_kq_launch(wt, W, xq, Y, M, N, K, (cudaStream_t)stream, true);
}

}  // namespace qmm

using namespace qmm;

extern "C" {

qmm_status qmm_matmul_q4_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_kq_checked(QMM_Q4_K, W, xq, Y, M, N, K, stream);
}
qmm_status qmm_matmul_q2_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_kq_checked(QMM_Q2_K, W, xq, Y, M, N, K, stream);
}
qmm_status qmm_matmul_q6_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_kq_checked(QMM_Q6_K, W, xq, Y, M, N, K, stream);
}
qmm_status qmm_matmul_q5_K(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return matmul_kq_checked(QMM_Q5_K, W, xq, Y, M, N, K, stream);
}

unsigned qmm_internal_matmul_kq_error(int clear) {
    unsigned v = 0;
    cudaMemcpyFromSymbol(&v, g_matmul_kq_error, sizeof(v));
    if (clear) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_matmul_kq_error, &z, sizeof(z));
    }
    return v;
}

}  // extern "C"

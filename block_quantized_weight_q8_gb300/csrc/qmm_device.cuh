// qmm_device.cuh -- device-side building blocks shared by the libqmm kernels:
// block-format constants, shared-memory and PTX helpers (mbarrier, bulk copy),
// and the per-format block decoders that turn weight bytes plus an unpacked
// activation row into exact integer block sums.
//
// The decoders follow the pages' block layouts and dot formulas:
//   [minfer] "10 . CPU matmul: quantized weights x Q8_0 activations", s2.3, s3.2
//   [ggml]   "ggml Q4_0 vec_dot Walkthrough", s1.1, s1.2, s2
// and the GGUF reading for the Q6_K layout, Q2_K code order and Q4_K 6-bit packing.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

// ---------------------------------------------------------------- formats
template <int T> struct Fmt;
template <> struct Fmt<QMM_Q4_0> { static constexpr int BB = 18, BV = 32, ACT = QMM_Q8_0; };
template <> struct Fmt<QMM_Q8_0> { static constexpr int BB = 34, BV = 32, ACT = QMM_Q8_0; };
template <> struct Fmt<QMM_Q4_K> { static constexpr int BB = 144, BV = 256, ACT = QMM_Q8_K; };
template <> struct Fmt<QMM_Q6_K> { static constexpr int BB = 210, BV = 256, ACT = QMM_Q8_K; };
template <> struct Fmt<QMM_Q2_K> { static constexpr int BB = 84, BV = 256, ACT = QMM_Q8_K; };
template <> struct Fmt<QMM_Q4_1> { static constexpr int BB = 20, BV = 32, ACT = QMM_Q8_0; };
template <> struct Fmt<QMM_Q5_0> { static constexpr int BB = 22, BV = 32, ACT = QMM_Q8_0; };
template <> struct Fmt<QMM_Q5_1> { static constexpr int BB = 24, BV = 32, ACT = QMM_Q8_0; };
template <> struct Fmt<QMM_Q5_K> { static constexpr int BB = 176, BV = 256, ACT = QMM_Q8_K; };

constexpr int Q8_0_BB = 34;
constexpr int Q8_K_BB = 292;

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float h2f(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)(bits & 0xFFFFu)));
}
__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a((int)a, (int)b, c);
}
// unsigned bytes of a times signed bytes of b, summed into c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t byte_of(uint32_t w, int k) { return (w >> (8 * k)) & 0xFFu; }
// two-way dot products: a holds two signed 16-bit values, b four signed bytes;
// lo pairs a with bytes 0, 1 of b, hi with bytes 2, 3
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// try_wait that lets the hardware suspend the thread (up to `hint_ns`) until the
// phase completes, instead of returning at once: waiting warps stop competing
// for issue slots with the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after `limit_ns` of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}
// The same copy without an L2 cache hint (bytes that other CTAs read too).
__device__ __forceinline__ void bulk_g2s_nohint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar` (both
// addresses 16-byte aligned, size a multiple of 16), with an L2 eviction policy.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Programmatic dependent launch: let the next grid in the stream start early /
// wait until the previous grid's memory is visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate copy
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrBounds = 4u;  // an index outside its buffer (bounds-checked builds only)

// Bounds-checked builds (compiled with -DQMM_CHECK_BOUNDS): QMM_IN_BOUNDS(err, i, n)
// is true when 0 <= i < n; otherwise it records kErrBounds in the translation
// unit's device error word `err` and is false, so that the access it guards is
// skipped instead of faulting.  qmm_device_status() reports the record as
// QMM_E_BOUNDS.  In normal builds it is the constant true and its arguments are
// not evaluated.
#ifdef QMM_CHECK_BOUNDS
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}
__device__ __forceinline__ bool in_bounds_or_record(unsigned int* err, int64_t i, int64_t n) {
    if (i >= 0 && i < n) return true;
    atomicOr(err, kErrBounds);
    return false;
}
#define QMM_IN_BOUNDS(err, i, n) ::qmm::in_bounds_or_record(&(err), (int64_t)(i), (int64_t)(n))
#else
#define QMM_IN_BOUNDS(err, i, n) true
#endif

// ---------------------------------------------------------------- unaligned byte reader
// A view of bytes in shared memory at a 2-byte-aligned offset.  word(i) returns
// the 4 bytes at off + 4i (little-endian), assembled from aligned 32-bit loads.
// Plain C++ loads, so the compiler orders them after the barriers that publish
// the data and is free to batch them.
struct SmemBytes {
    const uint8_t* base;  // shared-memory pointer to byte 0 of the view (16-byte aligned)
    __device__ __forceinline__ uint32_t w32(uint32_t off) const {  // off % 4 == 0
        return *reinterpret_cast<const uint32_t*>(base + off);
    }
    __device__ __forceinline__ uint32_t u16(uint32_t off) const {  // off % 2 == 0
        return *reinterpret_cast<const unsigned short*>(base + off);
    }
    // NW consecutive little-endian words starting at byte `off` (off even)
    template <int NW>
    __device__ __forceinline__ void words(uint32_t off, uint32_t* out) const {
        const uint32_t a0 = off & ~3u;
        const uint32_t sh = (off & 3u) * 8u;
        uint32_t raw[NW + 1];
#pragma unroll
        for (int i = 0; i <= NW; i++) raw[i] = w32(a0 + 4u * i);
#pragma unroll
        for (int i = 0; i < NW; i++) out[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
    }
    // the same when `off` is known to be 4-byte aligned
    template <int NW>
    __device__ __forceinline__ void words_aligned(uint32_t off, uint32_t* out) const {
#pragma unroll
        for (int i = 0; i < NW; i++) out[i] = w32(off + 4u * i);
    }
};

// The activation row, unpacked once per CTA into shared memory, chunk-major:
//   q         int8 codes as 16-byte chunks, chunk c of block u at (c*n + u)*16,
//             so lanes working on consecutive blocks read consecutive 16-byte
//             words -- no bank conflicts
//   d[]       f32 block scales (Q8_0: from f16; Q8_K: as stored), d[u]
//   s         Q8_0: int32 sum of each block's 32 codes, s[u] (for the Q4_0 -8);
//             Q8_K: the bsums as packed int16 pairs (groups 2k, 2k+1 in one
//             word, as the block stores them), pair k of block u at s[k*n + u].
// n is the pitch: the blocks per row for Q8_0; for Q8_K the super-blocks per
// row made odd (q8k_pitch), because the writers of a Q8_K row put the chunks of
// one super-block into consecutive lanes, n*16 bytes apart, and with n a
// multiple of 8 every lane of a store would hit the same four banks.
__host__ __device__ constexpr int q8k_pitch(int ns) { return ns | 1; }

struct ActView {
    const uint8_t* q;
    const float* d;
    const int* s;
    int n;
    __device__ __forceinline__ uint4 chunk(int u, int c) const {
        return *reinterpret_cast<const uint4*>(q + ((uint32_t)c * n + u) * 16);
    }
    __device__ __forceinline__ uint32_t bpair(int u, int k) const {
        return reinterpret_cast<const uint32_t*>(s)[k * n + u];
    }
};

// ---------------------------------------------------------------- block decoders
// Each decoder computes the exact integer sums of one weight block (or
// super-block) `u` at shared byte offset `o` against the activation, and
// returns the weight's scale fields.  Integers never round; the float fold is
// done by the caller.

// Q4_0 x Q8_0: isum = sum_j (n_j - 8) * a_j.  The nibbles of byte j are
// elements j (low) and j+16 (high) ([ggml] s2).  The -8 is applied once per
// block as -8 * sum(a), the same integers as subtracting it per element
// ([kvad] "The nibble kernel the compiler would not write").
__device__ __forceinline__ int q4_0_isum(const SmemBytes& w, uint32_t o, const ActView& a, int b,
                                         uint32_t* d_bits) {
    *d_bits = w.u16(o);
    uint32_t qs[4];
    w.words<4>(o + 2, qs);
    const uint4 lo = a.chunk(b, 0), hi = a.chunk(b, 1);
    const uint32_t al[4] = {lo.x, lo.y, lo.z, lo.w}, ah[4] = {hi.x, hi.y, hi.z, hi.w};
    int s0 = 0, s1 = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        s0 = dp4a(qs[i] & 0x0F0F0F0Fu, al[i], s0);
        s1 = dp4a((qs[i] >> 4) & 0x0F0F0F0Fu, ah[i], s1);
    }
    return s0 + s1 - 8 * a.s[b];
}

// Q8_0 x Q8_0: isum = sum_j w_j * a_j ([minfer] s3.2, the Q8_0 kernel).
__device__ __forceinline__ int q8_0_isum(const SmemBytes& w, uint32_t o, const ActView& a, int b,
                                         uint32_t* d_bits) {
    *d_bits = w.u16(o);
    uint32_t qs[8];
    w.words<8>(o + 2, qs);
    const uint4 lo = a.chunk(b, 0), hi = a.chunk(b, 1);
    int s0 = 0, s1 = 0;
    s0 = dp4a(qs[0], lo.x, s0); s1 = dp4a(qs[1], lo.y, s1); s0 = dp4a(qs[2], lo.z, s0); s1 = dp4a(qs[3], lo.w, s1);
    s0 = dp4a(qs[4], hi.x, s0); s1 = dp4a(qs[5], hi.y, s1); s0 = dp4a(qs[6], hi.z, s0); s1 = dp4a(qs[7], hi.w, s1);
    return s0 + s1;
}

// Q4_K x Q8_K ([minfer] s3.2, the K-quant dot walked): for chunk j of 32 nibble
// bytes, low nibbles pair with activations 64j + l, high with 64j + 32 + l;
// value = sum_j s_lo*sc[2j] + s_hi*sc[2j+1]; min = sum_s m_s*(bsum_2s + bsum_2s+1).
// 144-byte super-blocks in 16-byte aligned rows: read with 16-byte loads.
__device__ __forceinline__ void q4_K_isums(const SmemBytes& w, uint32_t o, const ActView& a, int u, int* value,
                                           int* minterm, uint32_t* d_bits, uint32_t* dmin_bits) {
    const uint4 h = *reinterpret_cast<const uint4*>(w.base + o);
    *d_bits = h.x & 0xFFFFu;
    *dmin_bits = h.x >> 16;
    // 6-bit scales and mins (GGUF packing, a reading): bytes b0..b11 = h.y, h.z, h.w
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;                                   // sc 0..3
    const uint32_t mn_lo = h.z & 0x3F3F3F3Fu;                                   // m 0..3
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);   // sc 4..7
    const uint32_t mn_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);  // m 4..7
    // m_s * (bsum_2s + bsum_2s+1): pair s against the bytes (m_s, m_s)
    int m = 0;
    m = dp2a_lo(a.bpair(u, 0), __byte_perm(mn_lo, 0, 0x1100), m);
    m = dp2a_hi(a.bpair(u, 1), __byte_perm(mn_lo, 0, 0x1100), m);
    m = dp2a_lo(a.bpair(u, 2), __byte_perm(mn_lo, 0, 0x3322), m);
    m = dp2a_hi(a.bpair(u, 3), __byte_perm(mn_lo, 0, 0x3322), m);
    m = dp2a_lo(a.bpair(u, 4), __byte_perm(mn_hi, 0, 0x1100), m);
    m = dp2a_hi(a.bpair(u, 5), __byte_perm(mn_hi, 0, 0x1100), m);
    m = dp2a_lo(a.bpair(u, 6), __byte_perm(mn_hi, 0, 0x3322), m);
    m = dp2a_hi(a.bpair(u, 7), __byte_perm(mn_hi, 0, 0x3322), m);
    int v = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(w.base + o + 16 + 32 * j);
        const uint4 q1 = *reinterpret_cast<const uint4*>(w.base + o + 32 + 32 * j);
        const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint4 l0 = a.chunk(u, 4 * j), l1 = a.chunk(u, 4 * j + 1);
        const uint4 h0 = a.chunk(u, 4 * j + 2), h1 = a.chunk(u, 4 * j + 3);
        const uint32_t al[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
        const uint32_t ah[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        int s_lo = 0, s_hi = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            s_lo = dp4a(q[i] & 0x0F0F0F0Fu, al[i], s_lo);
            s_hi = dp4a((q[i] >> 4) & 0x0F0F0F0Fu, ah[i], s_hi);
        }
        const uint32_t scw = j < 2 ? sc_lo : sc_hi;
        v += s_lo * (int)byte_of(scw, (2 * j) & 3) + s_hi * (int)byte_of(scw, (2 * j + 1) & 3);
    }
    *value = v;
    *minterm = m;
}

// Q2_K x Q8_K ([ggml] s1.2): value = sum_g sc_g * sum_{i in g} q_i a_i,
// min = sum_g m_g * bsum_g; element 128h + 32s + l is (qs[32h + l] >> 2s) & 3
// (GGUF order, a reading).  The codes of shift s are taken in place, masked to
// 4^s * q (bytes up to 192: an unsigned x signed dp4a), and the power of four is
// divided out once per shift: every such sum is an exact multiple of it.  The
// min term is four pairs of two-way dots of the bsum pairs against the m
// nibbles.  84-byte blocks in 4-byte aligned rows: aligned words.
__device__ __forceinline__ void q2_K_isums(const SmemBytes& w, uint32_t o, const ActView& a, int u, int* value,
                                           int* minterm, uint32_t* d_bits, uint32_t* dmin_bits) {
    uint32_t scw[4];
    w.words_aligned<4>(o, scw);
    const uint32_t dd = w.w32(o + 80);
    *d_bits = dd & 0xFFFFu;
    *dmin_bits = dd >> 16;
    int m = 0;
    uint32_t scl[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint32_t mw = (scw[k] >> 4) & 0x0F0F0F0Fu;
        m = dp2a_lo(a.bpair(u, 2 * k), mw, m);
        m = dp2a_hi(a.bpair(u, 2 * k + 1), mw, m);
        scl[k] = scw[k] & 0x0F0F0F0Fu;
    }
    int vs[4] = {0, 0, 0, 0};
#pragma unroll
    for (int h = 0; h < 2; h++) {
        uint32_t q[8];
        w.words_aligned<8>(o + 16 + 32 * h, q);
#pragma unroll
        for (int s = 0; s < 4; s++) {
            const uint4 a0 = a.chunk(u, 8 * h + 2 * s), a1 = a.chunk(u, 8 * h + 2 * s + 1);
            const uint32_t mask = 0x03030303u << (2 * s);
            int g0 = 0, g1 = 0;
            g0 = dp4a_us(q[0] & mask, a0.x, g0);
            g0 = dp4a_us(q[1] & mask, a0.y, g0);
            g0 = dp4a_us(q[2] & mask, a0.z, g0);
            g0 = dp4a_us(q[3] & mask, a0.w, g0);
            g1 = dp4a_us(q[4] & mask, a1.x, g1);
            g1 = dp4a_us(q[5] & mask, a1.y, g1);
            g1 = dp4a_us(q[6] & mask, a1.z, g1);
            g1 = dp4a_us(q[7] & mask, a1.w, g1);
            const int g = 8 * h + 2 * s;
            // byte g & 3 of the scale word, zero-extended (selector 4 takes a zero byte)
            vs[s] += (int)__byte_perm(scl[g >> 2], 0, 0x4440u | (g & 3)) * g0;
            vs[s] += (int)__byte_perm(scl[(g + 1) >> 2], 0, 0x4440u | ((g + 1) & 3)) * g1;
        }
    }
    *value = vs[0] + (vs[1] >> 2) + (vs[2] >> 4) + (vs[3] >> 6);
    *minterm = m;
}

// Q6_K x Q8_K (GGUF layout, a reading): value = sum_g sc_g * sum_{i in g} q_i a_i
// with the stored codes q in 0..63, min = sum_g sc_g * bsum_g; the signed-code
// sum is value - 32*min.  210-byte blocks: only 2-byte aligned.
__device__ __forceinline__ void q6_K_isums(const SmemBytes& w, uint32_t o, const ActView& a, int u, int* value,
                                           int* minterm, uint32_t* d_bits) {
    uint32_t scw[4];
    w.words<4>(o + 192, scw);
    *d_bits = w.u16(o + 208);
    int m = 0, v = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {  // sum_g sc_g * bsum_g: signed scale bytes against the bsum pairs
        m = dp2a_lo(a.bpair(u, 2 * k), scw[k], m);
        m = dp2a_hi(a.bpair(u, 2 * k + 1), scw[k], m);
    }
#pragma unroll
    for (int n = 0; n < 2; n++) {
        uint32_t A[8], B[8], H[8];
        w.words<8>(o + 64 * n, A);
        w.words<8>(o + 64 * n + 32, B);
        w.words<8>(o + 128 + 32 * n, H);
#pragma unroll
        for (int k = 0; k < 4; k++) {
            // elements 128n + 32k + 4i: chunks 8n + 2k (i < 4) and 8n + 2k + 1 (i >= 4)
            const uint4 c0 = a.chunk(u, 8 * n + 2 * k), c1 = a.chunk(u, 8 * n + 2 * k + 1);
            const uint32_t av[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            int acc0 = 0, acc1 = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                uint32_t q;
                if (k == 0) q = (A[i] & 0x0F0F0F0Fu) | ((H[i] << 4) & 0x30303030u);
                else if (k == 1) q = (B[i] & 0x0F0F0F0Fu) | ((H[i] << 2) & 0x30303030u);
                else if (k == 2) q = ((A[i] >> 4) & 0x0F0F0F0Fu) | (H[i] & 0x30303030u);
                else q = ((B[i] >> 4) & 0x0F0F0F0Fu) | ((H[i] >> 2) & 0x30303030u);
                if (i < 4) acc0 = dp4a(q, av[i], acc0);
                else acc1 = dp4a(q, av[i], acc1);
            }
            const int g = 8 * n + 2 * k;
            v += (int)(int8_t)byte_of(scw[g >> 2], g & 3) * acc0;
            v += (int)(int8_t)byte_of(scw[(g + 1) >> 2], (g + 1) & 3) * acc1;
        }
    }
    *value = v;
    *minterm = m;
}

// ---------------------------------------------------------------- formats with a fifth bit or a min
// GGUF layouts (readings; the pages give the 22/24/176-byte sizes and that the
// five-bit types add a plane of high bits):
//   Q4_1  f16 d, f16 m, qs[16]           value d*q + m
//   Q5_0  f16 d, qh[4], qs[16]           value d*(q - 16)
//   Q5_1  f16 d, f16 m, qh[4], qs[16]    value d*q + m
//   Q5_K  f16 d, f16 dmin, scales[12], qh[32], qs[128]   value d*sc_s*q - dmin*m_s
// Nibbles as in Q4_0; bit i of the 32-bit qh is the fifth bit of element i.

// bits 0..3 of x moved to bit 0 of bytes 0..3 (the four partial products of the
// multiply land on disjoint bit ranges, so nothing carries)
__device__ __forceinline__ uint32_t spread4(uint32_t x) { return ((x & 15u) * 0x00204081u) & 0x01010101u; }

// sum_j q_j * a_j of a 32-value block given its four nibble words and (for the
// five-bit types) the 32-bit plane of fifth bits
template <bool FIVE>
__device__ __forceinline__ int nib_isum(const uint32_t qs[4], uint32_t qh, const ActView& a, int b) {
    const uint4 lo = a.chunk(b, 0), hi = a.chunk(b, 1);
    const uint32_t al[4] = {lo.x, lo.y, lo.z, lo.w}, ah[4] = {hi.x, hi.y, hi.z, hi.w};
    int s0 = 0, s1 = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t ql = qs[i] & 0x0F0F0F0Fu, qu = (qs[i] >> 4) & 0x0F0F0F0Fu;
        if constexpr (FIVE) {
            ql |= spread4(qh >> (4 * i)) << 4;
            qu |= spread4(qh >> (16 + 4 * i)) << 4;
        }
        s0 = dp4a(ql, al[i], s0);
        s1 = dp4a(qu, ah[i], s1);
    }
    return s0 + s1;
}

// Q4_1 x Q8_0: isum = sum q*a; the caller adds m * dx * sum(a).  20-byte blocks
// in 16-byte aligned rows: 4-byte aligned.
__device__ __forceinline__ int q4_1_isum(const SmemBytes& w, uint32_t o, const ActView& a, int b, uint32_t* dm_bits) {
    *dm_bits = w.w32(o);
    uint32_t qs[4];
    w.words_aligned<4>(o + 4, qs);
    return nib_isum<false>(qs, 0u, a, b);
}

// Q5_0 x Q8_0: isum = sum (q - 16)*a, the -16 applied once as -16*sum(a).
// 22-byte blocks: 2-byte aligned.
__device__ __forceinline__ int q5_0_isum(const SmemBytes& w, uint32_t o, const ActView& a, int b, uint32_t* d_bits) {
    *d_bits = w.u16(o);
    uint32_t v[5];
    w.words<5>(o + 2, v);
    const uint32_t qs[4] = {v[1], v[2], v[3], v[4]};
    return nib_isum<true>(qs, v[0], a, b) - 16 * a.s[b];
}

// Q5_1 x Q8_0: isum = sum q*a; the caller adds m * dx * sum(a).  24-byte blocks:
// 8-byte aligned.
__device__ __forceinline__ int q5_1_isum(const SmemBytes& w, uint32_t o, const ActView& a, int b, uint32_t* dm_bits) {
    *dm_bits = w.w32(o);
    const uint32_t qh = w.w32(o + 4);
    uint32_t qs[4];
    w.words_aligned<4>(o + 8, qs);
    return nib_isum<true>(qs, qh, a, b);
}

// Q5_K x Q8_K: the Q4_K dot with five-bit codes: element 64j + l takes bit 2j
// of qh[l], element 64j + 32 + l bit 2j + 1.  176-byte super-blocks: 16-byte
// aligned.
__device__ __forceinline__ void q5_K_isums(const SmemBytes& w, uint32_t o, const ActView& a, int u, int* value,
                                           int* minterm, uint32_t* d_bits, uint32_t* dmin_bits) {
    const uint4 h = *reinterpret_cast<const uint4*>(w.base + o);
    *d_bits = h.x & 0xFFFFu;
    *dmin_bits = h.x >> 16;
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu;
    const uint32_t mn_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t mn_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
    // m_s * (bsum_2s + bsum_2s+1): pair s against the bytes (m_s, m_s)
    int m = 0;
    m = dp2a_lo(a.bpair(u, 0), __byte_perm(mn_lo, 0, 0x1100), m);
    m = dp2a_hi(a.bpair(u, 1), __byte_perm(mn_lo, 0, 0x1100), m);
    m = dp2a_lo(a.bpair(u, 2), __byte_perm(mn_lo, 0, 0x3322), m);
    m = dp2a_hi(a.bpair(u, 3), __byte_perm(mn_lo, 0, 0x3322), m);
    m = dp2a_lo(a.bpair(u, 4), __byte_perm(mn_hi, 0, 0x1100), m);
    m = dp2a_hi(a.bpair(u, 5), __byte_perm(mn_hi, 0, 0x1100), m);
    m = dp2a_lo(a.bpair(u, 6), __byte_perm(mn_hi, 0, 0x3322), m);
    m = dp2a_hi(a.bpair(u, 7), __byte_perm(mn_hi, 0, 0x3322), m);
    const uint4 h0 = *reinterpret_cast<const uint4*>(w.base + o + 16);
    const uint4 h1 = *reinterpret_cast<const uint4*>(w.base + o + 32);
    const uint32_t qh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    int v = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(w.base + o + 48 + 32 * j);
        const uint4 q1 = *reinterpret_cast<const uint4*>(w.base + o + 64 + 32 * j);
        const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint4 l0 = a.chunk(u, 4 * j), l1 = a.chunk(u, 4 * j + 1);
        const uint4 g0 = a.chunk(u, 4 * j + 2), g1 = a.chunk(u, 4 * j + 3);
        const uint32_t al[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
        const uint32_t ah[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        int s_lo = 0, s_hi = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t lo = (q[i] & 0x0F0F0F0Fu) | (((qh[i] >> (2 * j)) & 0x01010101u) << 4);
            const uint32_t hi = ((q[i] >> 4) & 0x0F0F0F0Fu) | (((qh[i] >> (2 * j + 1)) & 0x01010101u) << 4);
            s_lo = dp4a(lo, al[i], s_lo);
            s_hi = dp4a(hi, ah[i], s_hi);
        }
        const uint32_t scw = j < 2 ? sc_lo : sc_hi;
        v += s_lo * (int)byte_of(scw, (2 * j) & 3) + s_hi * (int)byte_of(scw, (2 * j + 1) & 3);
    }
    *value = v;
    *minterm = m;
}

// ---------------------------------------------------------------- activation unpack
// Unpacks one activation row (Q8_0 or Q8_K blocks in global memory, row base
// at least 2-byte aligned) into the chunk-major ActView arrays, one item per
// call so that any set of threads can share the work; the caller synchronizes
// those threads afterwards.
// block b (f16 scale bits, 32 codes as 8 words) into the chunk-major Q8_0 view
__device__ __forceinline__ void act_put_q8_0_block(const uint32_t w[8], uint32_t dbits, int b, int nb, uint8_t* q,
                                                   float* d, int* s) {
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) sum = dp4a(w[i], 0x01010101u, sum);
    d[b] = h2f(dbits);
    s[b] = sum;
    *reinterpret_cast<uint4*>(q + (uint32_t)b * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(q + ((uint32_t)nb + b) * 16) = make_uint4(w[4], w[5], w[6], w[7]);
}

__device__ __forceinline__ void unpack_q8_0_block(const uint8_t* __restrict__ row, int K, int b, uint8_t* q, float* d,
                                                  int* s) {
    const int nb = K / 32;
    const unsigned short* p = reinterpret_cast<const unsigned short*>(row + 34 * b);
    d[b] = h2f(p[0]);
    uint32_t wv[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        wv[i] = (uint32_t)p[1 + 2 * i] | ((uint32_t)p[2 + 2 * i] << 16);
        sum = dp4a(wv[i], 0x01010101u, sum);
    }
    *reinterpret_cast<uint4*>(q + (uint32_t)b * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    *reinterpret_cast<uint4*>(q + ((uint32_t)nb + b) * 16) = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    s[b] = sum;
}

// The whole Q8_K row by the threads tid, tid + nthr, ...: item t is chunk
// c = t % 16 of super-block u = t / 16 (its 16 code bytes as four words); the
// items c < 8 also carry bsum pair c, item 8 the scale.  A thread takes two
// items and issues all their loads before it stores any, so even a long row
// (K = 12288: 768 items) is one memory round trip.  The 16 items of a
// super-block sit in consecutive lanes and their chunks pitch * 16 bytes apart,
// pitch odd, so a quarter warp's 16-byte stores fall in distinct banks.  Rows
// need 4-byte alignment only (Q8_K rows are 292 bytes).
__device__ __forceinline__ void unpack_q8_K_row_by(const uint8_t* __restrict__ row, int ns, int n, uint8_t* q,
                                                   float* d, int* s, int tid, int nthr) {
    const int total = ns * 16;
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(row);
    for (int t0 = tid; t0 < total; t0 += 2 * nthr) {
        uint32_t v[2][5];
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const int t = t0 + k * nthr;
            const int u = t >> 4, c = t & 15;
            if (t < total) {
                const uint32_t* b = rw + 73 * u;
#pragma unroll
                for (int e = 0; e < 4; e++) v[k][e] = b[1 + 4 * c + e];
                v[k][4] = c < 8 ? b[65 + c] : (c == 8 ? b[0] : 0u);
            }
        }
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const int t = t0 + k * nthr;
            const int u = t >> 4, c = t & 15;
            if (t < total) {
                *reinterpret_cast<uint4*>(q + ((uint32_t)c * n + u) * 16) =
                    make_uint4(v[k][0], v[k][1], v[k][2], v[k][3]);
                if (c < 8) reinterpret_cast<uint32_t*>(s)[c * n + u] = v[k][4];  // pair of groups 2c, 2c + 1
                else if (c == 8) d[u] = __uint_as_float(v[k][4]);
            }
        }
    }
}

__device__ __forceinline__ void unpack_q8_0_row(const uint8_t* __restrict__ row, int K, uint8_t* q, float* d,
                                                int* s) {
    for (int b = threadIdx.x; b < K / 32; b += blockDim.x) unpack_q8_0_block(row, K, b, q, d, s);
}

__device__ __forceinline__ void unpack_q8_K_row(const uint8_t* __restrict__ row, int K, uint8_t* q, float* d,
                                                int* s) {
    const int ns = K / 256;
    unpack_q8_K_row_by(row, ns, q8k_pitch(ns), q, d, s, threadIdx.x, blockDim.x);
}

// ---------------------------------------------------------------- activation quantizers
// The per-block arithmetic of the Q8_0 / Q8_K activation quantizers, shared by
// the standalone quantize kernels and the matvec kernels that quantize their
// own input, so both write the same bytes.  Every float operation is an
// explicitly IEEE-rounded intrinsic (no contraction), as the pages' scalar
// definitions round each step once ([krafla] "Architecture", Numerics).
__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }
__device__ __forceinline__ uint32_t f2h_bits(float f) { return (uint32_t)__half_as_ushort(__float2half_rn(f)); }
// 16-bit stores for every f16 field (a byte store of the low half of a
// __float2half_rn result was seen to store 0 with this toolchain)
__device__ __forceinline__ void st_u16(uint8_t* p, uint32_t v) {
    *reinterpret_cast<unsigned short*>(p) = (unsigned short)(v & 0xFFFFu);
}

// Q8_0 ([minfer] "10 . CPU matmul: quantized weights x Q8_0 activations" s3.2):
// per 32 values amax = max|x|, d = amax/127 stored as f16, inverse 127/amax (0
// for an all-zero block), codes rne(x * inverse) saturated to int8.  Eight
// consecutive lanes (part = lane & 7) hold a block, four values each; all 32
// lanes of the warp call, inactive ones with active = false.  `ob` is the
// block's 34 output bytes.
__device__ __forceinline__ void quant_q8_0_part(float4 v, bool active, int part, uint8_t* ob) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    if (!active) return;
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = amax != 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    const int q0 = clampi(__float2int_rn(__fmul_rn(v.x, id)), -128, 127);
    const int q1 = clampi(__float2int_rn(__fmul_rn(v.y, id)), -128, 127);
    const int q2 = clampi(__float2int_rn(__fmul_rn(v.z, id)), -128, 127);
    const int q3 = clampi(__float2int_rn(__fmul_rn(v.w, id)), -128, 127);
    if (part == 0) st_u16(ob, f2h_bits(d));
    st_u16(ob + 2 + 4 * part, (uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8));
    st_u16(ob + 4 + 4 * part, (uint32_t)(q2 & 0xFF) | ((uint32_t)(q3 & 0xFF) << 8));
}

// Q8_K ([minfer] s3.2, quantize_row_q8_k_buf): per 256 values amax, f32
// d = amax/127, codes saturated to [-128, 127], bsums[g] = exact sum of the 16
// saturated codes of group g.  One warp per super-block, eight values per lane
// (v0, v1 = values 8*lane .. 8*lane+7): lanes 2g and 2g+1 hold group g.  `ob`
// is the super-block's 292 output bytes (4-byte aligned).
// The arithmetic of one lane: its 8 codes as two words, the block's f32 scale,
// and (lanes 4k) the bsum pair of groups 2k, 2k + 1.
__device__ __forceinline__ void quant_q8_K_core(float4 v0, float4 v1, float* d_out, uint32_t* w0_out,
                                                uint32_t* w1_out, uint32_t* pair_out) {
    float amax = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                       fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = amax != 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t w0 = 0, w1 = 0;
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int q = clampi(__float2int_rn(__fmul_rn(vv[i], id)), -128, 127);
        sum += q;
        if (i < 4) w0 |= (uint32_t)(q & 0xFF) << (8 * i);
        else w1 |= (uint32_t)(q & 0xFF) << (8 * (i - 4));
    }
    const int bsum = sum + __shfl_xor_sync(0xffffffffu, sum, 1);   // group lane/2
    const int bsum_next = __shfl_down_sync(0xffffffffu, bsum, 2);  // group lane/2 + 1
    *d_out = d;
    *w0_out = w0;
    *w1_out = w1;
    *pair_out = ((uint32_t)bsum & 0xFFFFu) | ((uint32_t)(bsum_next & 0xFFFF) << 16);
}

// the 292-byte Q8_K block at ob
__device__ __forceinline__ void store_q8_K_block(int lane, float d, uint32_t w0, uint32_t w1, uint32_t pair,
                                                 uint8_t* ob) {
    if (lane == 0) *reinterpret_cast<float*>(ob) = d;
    *reinterpret_cast<uint32_t*>(ob + 4 + 8 * lane) = w0;
    *reinterpret_cast<uint32_t*>(ob + 8 + 8 * lane) = w1;
    if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(ob + 260 + lane) = pair;
}

__device__ __forceinline__ void quant_q8_K_lane(float4 v0, float4 v1, int lane, uint8_t* ob) {
    float d;
    uint32_t w0, w1, pair;
    quant_q8_K_core(v0, v1, &d, &w0, &w1, &pair);
    store_q8_K_block(lane, d, w0, w1, pair, ob);
}

// The same block straight into the decoder's view (block u, pitch n): the codes
// of lane l (8l .. 8l + 7) are half of chunk l / 2; also the 292-byte block at
// ob when ob is not null.
__device__ __forceinline__ void quant_q8_K_lane_put(float4 v0, float4 v1, int lane, int u, int n, uint8_t* q,
                                                    float* dv, int* s, uint8_t* ob) {
    float d;
    uint32_t w0, w1, pair;
    quant_q8_K_core(v0, v1, &d, &w0, &w1, &pair);
    if (lane == 0) dv[u] = d;
    *reinterpret_cast<uint2*>(q + ((uint32_t)(lane >> 1) * n + u) * 16 + (lane & 1) * 8) = make_uint2(w0, w1);
    if ((lane & 3) == 0) reinterpret_cast<uint32_t*>(s)[(lane >> 2) * n + u] = pair;
    if (ob != nullptr) store_q8_K_block(lane, d, w0, w1, pair, ob);
}

// ---------------------------------------------------------------- super-units (Q8_0, Q4_0 weights)
// Eight consecutive 32-value blocks form a "super-unit": 272 bytes for Q8_0
// (17 chunks of 16 B), 144 bytes for Q4_0 (9 chunks).  When a row holds whole
// super-units (K % 256 == 0) every super-unit starts on a 16-byte boundary, so
// one lane can read its super-unit with aligned 16-byte loads and no byte
// shuffling.  Each 4-byte word x of a super-unit holds codes of at most one
// block, namely block (4x + 1) / 34 (Q8_0) or (4x + 1) / 18 (Q4_0): the two
// f16 scale bytes sit between the codes of neighbouring blocks.  The activation
// is laid out in the same byte positions with zeros where the weight has its
// scale, so a word-by-word dp4a over the super-unit yields each block's exact
// integer code dot, the scale bytes contributing nothing.
//
// Activation arrays (chunk-major so that lanes on consecutive super-units read
// consecutive 16-byte words):
//   Q8_0: chunk c of super-unit u at (c*nsu + u)*16: the activation row's own
//         bytes [272u + 16c, +16) with the f16 d fields zeroed.
//   Q4_0: two planes in the weight's byte layout: byte y = 18b + 2 + j of
//         super-unit u holds activation code 32(8u+b) + j (plane 0, paired with
//         the low nibble of weight byte j) or 32(8u+b) + 16 + j (plane 1, the
//         high nibble) ([ggml] "ggml Q4_0 vec_dot Walkthrough" s2: byte j holds
//         elements j and j+16); plane p, chunk c at ((9p + c)*nsu + u)*16.
//   d[b]: f32 activation scale of block b; s[b]: int32 sum of its 32 codes.

// Writes block b of a Q8_0 activation row -- its f16 scale bits and its 32
// codes as 8 little-endian words -- into the super-unit arrays of a Q8_0
// (PLANES = false) or Q4_0 (PLANES = true) weight, with its f32 scale and code
// sum.  Every byte of the arrays belongs to exactly one block, so one call per
// block fills them.  All stores are 16-bit at even offsets within a chunk.
template <bool PLANES>
__device__ __forceinline__ void su_put_block(const uint32_t w[8], uint32_t dbits, int b, int nsu, uint8_t* q,
                                             float* d, int* s) {
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) sum = dp4a(w[i], 0x01010101u, sum);
    d[b] = h2f(dbits);
    s[b] = sum;
    const int u = b >> 3, bb = b & 7;
    if constexpr (!PLANES) {
        // bytes 34bb, 34bb+1: the weight's d field (zero); 34bb + 2 + j: code j
        const int y0 = 34 * bb;
        *reinterpret_cast<unsigned short*>(q + ((uint32_t)(y0 >> 4) * nsu + u) * 16 + (y0 & 15)) = 0;
#pragma unroll
        for (int h = 0; h < 16; h++) {
            const int y = y0 + 2 + 2 * h;
            *reinterpret_cast<unsigned short*>(q + ((uint32_t)(y >> 4) * nsu + u) * 16 + (y & 15)) =
                (unsigned short)((w[h >> 1] >> (16 * (h & 1))) & 0xFFFFu);
        }
    } else {
#pragma unroll
        for (int pl = 0; pl < 2; pl++) {
            const int y0 = 18 * bb;  // the weight's d field: zero in both planes
            *reinterpret_cast<unsigned short*>(q + ((uint32_t)(9 * pl + (y0 >> 4)) * nsu + u) * 16 + (y0 & 15)) = 0;
#pragma unroll
            for (int h = 0; h < 8; h++) {
                const int y = y0 + 2 + 2 * h;
                const int code = 16 * pl + 2 * h;
                *reinterpret_cast<unsigned short*>(q + ((uint32_t)(9 * pl + (y >> 4)) * nsu + u) * 16 + (y & 15)) =
                    (unsigned short)((w[code >> 2] >> (16 * ((code >> 1) & 1))) & 0xFFFFu);
            }
        }
    }
}

// ---------------------------------------------------------------- RMSNorm ahead of the quantizer
// [krafla] "Architecture", "Data flow for one token": h = rmsnorm(x) ; qa =
// quantize_q8(h).  h_i = (x_i * s) * w_i with s = 1/sqrt(ss/K + eps), each step
// rounded once; ss in one fixed order -- 8-value sequential partials, then a
// stride-doubling tree (step 1, 2, 4, ...: p[i] += p[i + step] for i a multiple
// of 2*step) -- so that the codes of h are the same on every run and in the
// scalar implementation of the same steps.
//
// The tree runs as: thread t owns the aligned run of m partials [t*m, t*m + m)
// (m a power of two, m * threads >= K/8) and sums it pairwise; lanes then meet
// by xor shuffles and warps through one shared-memory step.  Partials past K/8
// are zeros, which leaves every sum unchanged (ss >= 0), so this is the same
// tree.  Every thread of the CTA calls it; p: rms_scratch_floats(K, threads)
// floats of shared memory; x 16-byte aligned, K % 8 == 0.
__host__ __device__ inline int rms_run(int K, int nthr) {
    int m = 1;
    while (m * nthr < K / 8) m <<= 1;
    return m;
}
__host__ __device__ inline int rms_scratch_floats(int K, int nthr) { return rms_run(K, nthr) * nthr + 33; }
// a bound for any block of up to max_threads threads: m * threads < 2 * K/8 when m > 1
__host__ __device__ inline int rms_scratch_bound(int K, int max_threads) {
    return (2 * (K / 8) > max_threads ? 2 * (K / 8) : max_threads) + 33;
}

__device__ __forceinline__ float sq8(const float4* x4, int i) {
    const float4 a = x4[2 * i], b = x4[2 * i + 1];
    float s = __fmul_rn(a.x, a.x);
    s = __fadd_rn(s, __fmul_rn(a.y, a.y));
    s = __fadd_rn(s, __fmul_rn(a.z, a.z));
    s = __fadd_rn(s, __fmul_rn(a.w, a.w));
    s = __fadd_rn(s, __fmul_rn(b.x, b.x));
    s = __fadd_rn(s, __fmul_rn(b.y, b.y));
    s = __fadd_rn(s, __fmul_rn(b.z, b.z));
    return __fadd_rn(s, __fmul_rn(b.w, b.w));
}

// the pairwise sum of the run of M partials starting at partial `first`, in
// registers: every load is issued before the first add
template <int M>
__device__ __forceinline__ float rms_run_sum(const float4* x4, int first, int n8) {
    float p[M];
#pragma unroll
    for (int i = 0; i < M; i++) p[i] = first + i < n8 ? sq8(x4, first + i) : 0.0f;
#pragma unroll
    for (int step = 1; step < M; step <<= 1)
#pragma unroll
        for (int i = 0; i < M; i += 2 * step) p[i] = __fadd_rn(p[i], p[i + step]);
    return p[0];
}

__device__ __forceinline__ float rms_scale(const float* x, int K, float* p, float eps) {
    const int n8 = K / 8, nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = rms_run(K, nthr);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float v;
    if (m == 1) {
        v = tid < n8 ? sq8(x4, tid) : 0.0f;
    } else if (m == 2) {
        v = rms_run_sum<2>(x4, tid * 2, n8);
    } else if (m == 4) {
        v = rms_run_sum<4>(x4, tid * 4, n8);
    } else if (m == 8) {
        v = rms_run_sum<8>(x4, tid * 8, n8);
    } else {
        // longer runs through shared memory (here each load waits for the
        // previous partial's store)
        float* pt = p + tid * m;
        for (int i = 0; i < m; i++) pt[i] = tid * m + i < n8 ? sq8(x4, tid * m + i) : 0.0f;
        for (int step = 1; step < m; step <<= 1)
            for (int i = 0; i < m; i += 2 * step) pt[i] = __fadd_rn(pt[i], pt[i + step]);
        v = pt[0];
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    float* wsum = p + m * nthr;
    if (lane == 0) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float u = lane < (nthr >> 5) ? wsum[lane] : 0.0f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) u = __fadd_rn(u, __shfl_xor_sync(0xFFFFFFFFu, u, off));
        if (lane == 0) wsum[32] = u;
    }
    __syncthreads();
    const float mean = __fdiv_rn(wsum[32], (float)K);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

__device__ __forceinline__ float4 norm4(float4 v, float s, float4 w) {
    return make_float4(__fmul_rn(__fmul_rn(v.x, s), w.x), __fmul_rn(__fmul_rn(v.y, s), w.y),
                       __fmul_rn(__fmul_rn(v.z, s), w.z), __fmul_rn(__fmul_rn(v.w, s), w.w));
}

// ---------------------------------------------------------------- super-units of Q4_1, Q5_0, Q5_1
// Eight blocks (160, 176, 192 bytes) start on a 16-byte boundary when K % 256
// == 0.  The activation for them: block bb of super-unit u keeps its codes
// 0..15 in chunk 2bb and 16..31 in chunk 2bb+1, chunk c at (c*nsu + u)*16.
template <int WT> struct SuFmt;
template <> struct SuFmt<QMM_Q8_0> { static constexpr int W = 272, A = 272; };
template <> struct SuFmt<QMM_Q4_0> { static constexpr int W = 144, A = 288; };
template <> struct SuFmt<QMM_Q4_1> { static constexpr int W = 160, A = 256; };
template <> struct SuFmt<QMM_Q5_0> { static constexpr int W = 176, A = 256; };
template <> struct SuFmt<QMM_Q5_1> { static constexpr int W = 192, A = 256; };
template <int WT>
__host__ __device__ constexpr bool has_su() {
    return WT == QMM_Q8_0 || WT == QMM_Q4_0 || WT == QMM_Q4_1 || WT == QMM_Q5_0 || WT == QMM_Q5_1;
}

__device__ __forceinline__ void su_put_halves(const uint32_t w[8], uint32_t dbits, int b, int nsu, uint8_t* q,
                                              float* d, int* s) {
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) sum = dp4a(w[i], 0x01010101u, sum);
    d[b] = h2f(dbits);
    s[b] = sum;
    const int u = b >> 3, bb = b & 7;
    *reinterpret_cast<uint4*>(q + ((uint32_t)(2 * bb) * nsu + u) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(q + ((uint32_t)(2 * bb + 1) * nsu + u) * 16) = make_uint4(w[4], w[5], w[6], w[7]);
}

// the 4 bytes at even byte offset `off` of a super-unit held as words ww[]
template <int OFF>
__device__ __forceinline__ uint32_t su_word(const uint32_t* ww) {
    if constexpr (OFF % 4 == 0) return ww[OFF / 4];
    else return __funnelshift_r(ww[OFF / 4], ww[OFF / 4 + 1], 16);
}

// One block bb of a Q4_1 / Q5_0 / Q5_1 super-unit: its f32 contribution
// (the per-block fold of the per-block decoders above).
template <int WT, int BB>
__device__ __forceinline__ float su_block5(const uint32_t* ww, const uint8_t* q, int nsu, int u, float dx, int asum) {
    constexpr int O = Fmt<WT>::BB * BB;  // byte offset of the block
    constexpr int QS = WT == QMM_Q4_1 ? 4 : (WT == QMM_Q5_0 ? 6 : 8);
    uint32_t qs[4], qh = 0;
    qs[0] = su_word<O + QS>(ww);
    qs[1] = su_word<O + QS + 4>(ww);
    qs[2] = su_word<O + QS + 8>(ww);
    qs[3] = su_word<O + QS + 12>(ww);
    if constexpr (WT == QMM_Q5_0) qh = su_word<O + 2>(ww);
    if constexpr (WT == QMM_Q5_1) qh = su_word<O + 4>(ww);
    const uint4 lo = *reinterpret_cast<const uint4*>(q + ((uint32_t)(2 * BB) * nsu + u) * 16);
    const uint4 hi = *reinterpret_cast<const uint4*>(q + ((uint32_t)(2 * BB + 1) * nsu + u) * 16);
    const uint32_t al[4] = {lo.x, lo.y, lo.z, lo.w}, ah[4] = {hi.x, hi.y, hi.z, hi.w};
    int s0 = 0, s1 = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t ql = qs[i] & 0x0F0F0F0Fu, qu = (qs[i] >> 4) & 0x0F0F0F0Fu;
        if constexpr (WT != QMM_Q4_1) {
            ql |= spread4(qh >> (4 * i)) << 4;
            qu |= spread4(qh >> (16 + 4 * i)) << 4;
        }
        s0 = dp4a(ql, al[i], s0);
        s1 = dp4a(qu, ah[i], s1);
    }
    if constexpr (WT == QMM_Q5_0) {
        const uint32_t db = (O % 4 == 0) ? (ww[O / 4] & 0xFFFFu) : (ww[O / 4] >> 16);
        return (float)(s0 + s1 - 16 * asum) * h2f(db) * dx;
    } else {
        const uint32_t dm = ww[O / 4];  // O % 4 == 0 for the 20- and 24-byte blocks
        return (float)(s0 + s1) * h2f(dm & 0xFFFFu) * dx + (float)asum * h2f(dm >> 16) * dx;
    }
}

// The f32 fold of one Q4_1 / Q5_0 / Q5_1 super-unit: the 8 blocks' contributions
// added in block order.  w: the super-unit in shared memory (16-byte aligned).
template <int WT>
__device__ __forceinline__ float su_q45(const uint8_t* w, const uint8_t* q, int nsu, int u, const float* d,
                                        const int* asum) {
    constexpr int NW = SuFmt<WT>::W / 4;
    uint32_t ww[NW + 1];
#pragma unroll
    for (int c = 0; c < NW / 4; c++) {
        const uint4 v = *reinterpret_cast<const uint4*>(w + 16 * c);
        ww[4 * c] = v.x, ww[4 * c + 1] = v.y, ww[4 * c + 2] = v.z, ww[4 * c + 3] = v.w;
    }
    ww[NW] = 0u;  // never selected: a funnel shift past the last block reads no real byte
    float acc = 0.0f;
    acc += su_block5<WT, 0>(ww, q, nsu, u, d[0], asum[0]);
    acc += su_block5<WT, 1>(ww, q, nsu, u, d[1], asum[1]);
    acc += su_block5<WT, 2>(ww, q, nsu, u, d[2], asum[2]);
    acc += su_block5<WT, 3>(ww, q, nsu, u, d[3], asum[3]);
    acc += su_block5<WT, 4>(ww, q, nsu, u, d[4], asum[4]);
    acc += su_block5<WT, 5>(ww, q, nsu, u, d[5], asum[5]);
    acc += su_block5<WT, 6>(ww, q, nsu, u, d[6], asum[6]);
    acc += su_block5<WT, 7>(ww, q, nsu, u, d[7], asum[7]);
    return acc;
}

// One thread quantizes one Q8_0 block of 32 values v (the same IEEE-rounded
// steps as quant_q8_0_part, so the same bytes): f16 scale bits and the codes as
// 8 little-endian words.
__device__ __forceinline__ void quant_q8_0_block(const float4 v[8], uint32_t* dbits, uint32_t w[8]) {
    // max over the block, seeded with the first values so that it is the same
    // set-maximum (NaN rules included) as the reduction in quant_q8_0_part
    float amax = fmaxf(fmaxf(fabsf(v[0].x), fabsf(v[0].y)), fmaxf(fabsf(v[0].z), fabsf(v[0].w)));
#pragma unroll
    for (int i = 1; i < 8; i++)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = amax != 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    *dbits = f2h_bits(d);
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int q0 = clampi(__float2int_rn(__fmul_rn(v[i].x, id)), -128, 127);
        const int q1 = clampi(__float2int_rn(__fmul_rn(v[i].y, id)), -128, 127);
        const int q2 = clampi(__float2int_rn(__fmul_rn(v[i].z, id)), -128, 127);
        const int q3 = clampi(__float2int_rn(__fmul_rn(v[i].w, id)), -128, 127);
        w[i] = (uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8) | ((uint32_t)(q2 & 0xFF) << 16) |
               ((uint32_t)(q3 & 0xFF) << 24);
    }
}

// One Q8_0 block quantized by LPB consecutive lanes of a warp (8 / LPB float4
// each): the same bytes as quant_q8_0_block (the maximum is exact in any order,
// NaN rules included), with the 8 code words gathered in the group's first lane
// (part 0).  Every lane of the warp calls it.
template <int LPB>
__device__ __forceinline__ void quant_q8_0_block_lanes(const float4* v, int part, uint32_t* dbits, uint32_t w[8]) {
    constexpr int NV = 8 / LPB;
    float amax = fmaxf(fmaxf(fabsf(v[0].x), fabsf(v[0].y)), fmaxf(fabsf(v[0].z), fabsf(v[0].w)));
#pragma unroll
    for (int i = 1; i < NV; i++)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
#pragma unroll
    for (int off = 1; off < LPB; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = amax != 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    *dbits = f2h_bits(d);
    uint32_t mine[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int q0 = clampi(__float2int_rn(__fmul_rn(v[i].x, id)), -128, 127);
        const int q1 = clampi(__float2int_rn(__fmul_rn(v[i].y, id)), -128, 127);
        const int q2 = clampi(__float2int_rn(__fmul_rn(v[i].z, id)), -128, 127);
        const int q3 = clampi(__float2int_rn(__fmul_rn(v[i].w, id)), -128, 127);
        mine[i] = (uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8) | ((uint32_t)(q2 & 0xFF) << 16) |
                  ((uint32_t)(q3 & 0xFF) << 24);
        w[i] = mine[i];
    }
#pragma unroll
    for (int src = 1; src < LPB; src++)
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, mine[i], src);
            if (part == 0) w[src * NV + i] = t;
        }
}

// The f32 fold of one super-unit: for each of its 8 blocks, isum * d_w * d_x
// added in block order ([minfer] "10 . CPU matmul: quantized weights x Q8_0
// activations" s3.2, the Q8_0 kernel).  w: the super-unit in shared memory
// (16-byte aligned); q: the activation array; d: the 8 activation scales.
__device__ __forceinline__ float su_q8_0(const uint8_t* w, const uint8_t* q, int nsu, int u, const float* d) {
    int s[8];
    uint32_t dw[8];
#pragma unroll
    for (int b = 0; b < 8; b++) s[b] = 0;
#pragma unroll
    for (int c = 0; c < 17; c++) {
        const uint4 wc = *reinterpret_cast<const uint4*>(w + 16 * c);
        const uint4 ac = *reinterpret_cast<const uint4*>(q + ((uint32_t)c * nsu + u) * 16);
        const uint32_t ww[4] = {wc.x, wc.y, wc.z, wc.w}, aa[4] = {ac.x, ac.y, ac.z, ac.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int x = 4 * c + j;
            s[(4 * x + 1) / 34] = dp4a(ww[j], aa[j], s[(4 * x + 1) / 34]);
#pragma unroll
            for (int b = 0; b < 8; b++)
                if ((34 * b) / 4 == x) dw[b] = ((34 * b) % 4 == 0) ? (ww[j] & 0xFFFFu) : (ww[j] >> 16);
        }
    }
    float acc = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; b++) acc += (float)s[b] * h2f(dw[b]) * d[b];
    return acc;
}

// Q4_0: isum_b = sum n_lo*a_lo + sum n_hi*a_hi - 8*sum(a) ([ggml] s2).  The
// high nibbles are taken in place (byte & 0xF0 = 16 n) with an unsigned x
// signed dp4a; the block's sum is a multiple of 16, divided out exactly.
__device__ __forceinline__ float su_q4_0(const uint8_t* w, const uint8_t* q, int nsu, int u, const float* d,
                                         const int* asum) {
    int s[8], t[8];
    uint32_t dw[8];
#pragma unroll
    for (int b = 0; b < 8; b++) s[b] = 0, t[b] = 0;
#pragma unroll
    for (int c = 0; c < 9; c++) {
        const uint4 wc = *reinterpret_cast<const uint4*>(w + 16 * c);
        const uint4 lo = *reinterpret_cast<const uint4*>(q + ((uint32_t)c * nsu + u) * 16);
        const uint4 hi = *reinterpret_cast<const uint4*>(q + ((uint32_t)(9 + c) * nsu + u) * 16);
        const uint32_t ww[4] = {wc.x, wc.y, wc.z, wc.w}, al[4] = {lo.x, lo.y, lo.z, lo.w},
                       ah[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int x = 4 * c + j, b = (4 * x + 1) / 18;
            s[b] = dp4a(ww[j] & 0x0F0F0F0Fu, al[j], s[b]);
            t[b] = dp4a_us(ww[j] & 0xF0F0F0F0u, ah[j], t[b]);
#pragma unroll
            for (int bb = 0; bb < 8; bb++)
                if ((18 * bb) / 4 == x) dw[bb] = ((18 * bb) % 4 == 0) ? (ww[j] & 0xFFFFu) : (ww[j] >> 16);
        }
    }
    float acc = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; b++) {
        const int isum = s[b] + (t[b] >> 4) - 8 * asum[b];
        acc += (float)isum * h2f(dw[b]) * d[b];
    }
    return acc;
}

}  // namespace qmm

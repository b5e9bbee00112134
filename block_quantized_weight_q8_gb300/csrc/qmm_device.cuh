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
__device__ __forceinline__ uint32_t byte_of(uint32_t w, int k) { return (w >> (8 * k)) & 0xFFu; }

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
// Bounded wait: gives up after `limit_ns` of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
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

// ---------------------------------------------------------------- unaligned byte reader
// A view of bytes in shared memory at a 2-byte-aligned offset.  word(i) returns
// the 4 bytes at off + 4i (little-endian), assembled from aligned 32-bit loads.
struct SmemBytes {
    uint32_t base;  // shared-memory address of byte 0 of the view
    __device__ __forceinline__ uint32_t u16(uint32_t off) const { return lds16(base + off); }
    __device__ __forceinline__ uint32_t u8(uint32_t off) const {
        uint32_t w = lds32((base + off) & ~3u);
        return (w >> (8 * ((base + off) & 3u))) & 0xFFu;
    }
    // n consecutive words starting at byte `off` (off even), into out[0..n)
    template <int NW>
    __device__ __forceinline__ void words(uint32_t off, uint32_t* out) const {
        const uint32_t a = base + off;
        const uint32_t a0 = a & ~3u;
        const uint32_t sh = (a & 3u) * 8u;
        uint32_t prev = lds32(a0);
#pragma unroll
        for (int i = 0; i < NW; i++) {
            uint32_t next = lds32(a0 + 4u * (i + 1));
            out[i] = __funnelshift_r(prev, next, sh);
            prev = next;
        }
    }
    // the same when `off` is known to be 4-byte aligned
    template <int NW>
    __device__ __forceinline__ void words_aligned(uint32_t off, uint32_t* out) const {
#pragma unroll
        for (int i = 0; i < NW; i++) out[i] = lds32(base + off + 4u * i);
    }
};

// The activation row, unpacked once per CTA into shared memory:
//   q[K]      int8 codes, 16-byte aligned, contiguous
//   d[nb]     f32 block scales (Q8_0: from f16; Q8_K: as stored)
//   s[...]    Q8_0: int32 sum of each block's 32 codes (used for the Q4_0 -8);
//             Q8_K: int32 bsums, 16 per super-block.
struct ActView {
    uint32_t q;  // shared address of the int8 codes
    const float* d;
    const int* s;
    __device__ __forceinline__ uint32_t qword(uint32_t elem) const { return lds32(q + elem); }
    __device__ __forceinline__ uint4 qvec(uint32_t elem) const { return lds128(q + elem); }
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
    const uint4 lo = a.qvec(32u * b), hi = a.qvec(32u * b + 16u);
    const uint32_t al[4] = {lo.x, lo.y, lo.z, lo.w}, ah[4] = {hi.x, hi.y, hi.z, hi.w};
    int s = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        s = dp4a(qs[i] & 0x0F0F0F0Fu, al[i], s);
        s = dp4a((qs[i] >> 4) & 0x0F0F0F0Fu, ah[i], s);
    }
    return s - 8 * a.s[b];
}

// Q8_0 x Q8_0: isum = sum_j w_j * a_j ([minfer] s3.2, the Q8_0 kernel).
__device__ __forceinline__ int q8_0_isum(const SmemBytes& w, uint32_t o, const ActView& a, int b,
                                         uint32_t* d_bits) {
    *d_bits = w.u16(o);
    uint32_t qs[8];
    w.words<8>(o + 2, qs);
    const uint4 lo = a.qvec(32u * b), hi = a.qvec(32u * b + 16u);
    int s = 0;
    s = dp4a(qs[0], lo.x, s); s = dp4a(qs[1], lo.y, s); s = dp4a(qs[2], lo.z, s); s = dp4a(qs[3], lo.w, s);
    s = dp4a(qs[4], hi.x, s); s = dp4a(qs[5], hi.y, s); s = dp4a(qs[6], hi.z, s); s = dp4a(qs[7], hi.w, s);
    return s;
}

// Q4_K x Q8_K ([minfer] s3.2, the K-quant dot walked): for chunk j of 32 nibble
// bytes, low nibbles pair with activations 64j + l, high with 64j + 32 + l;
// value = sum_j s_lo*sc[2j] + s_hi*sc[2j+1]; min = sum_s m_s*(bsum_2s + bsum_2s+1).
// The super-block starts 4-byte aligned (144-byte blocks, 16-byte aligned rows).
__device__ __forceinline__ void q4_K_isums(const SmemBytes& w, uint32_t o, const ActView& a, int u, int* value,
                                           int* minterm, uint32_t* d_bits, uint32_t* dmin_bits) {
    uint32_t h[4];
    w.words_aligned<4>(o, h);
    *d_bits = h[0] & 0xFFFFu;
    *dmin_bits = h[0] >> 16;
    // 6-bit scales and mins (GGUF packing, a reading): bytes b0..b11 = h[1..3]
    const uint32_t sc_lo = h[1] & 0x3F3F3F3Fu;                                   // sc 0..3
    const uint32_t mn_lo = h[2] & 0x3F3F3F3Fu;                                   // m 0..3
    const uint32_t sc_hi = (h[3] & 0x0F0F0F0Fu) | ((h[1] >> 2) & 0x30303030u);   // sc 4..7
    const uint32_t mn_hi = ((h[3] >> 4) & 0x0F0F0F0Fu) | ((h[2] >> 2) & 0x30303030u);  // m 4..7
    const int* bs = a.s + 16 * u;
    int m = 0;
#pragma unroll
    for (int s = 0; s < 4; s++) m += (int)byte_of(mn_lo, s) * (bs[2 * s] + bs[2 * s + 1]);
#pragma unroll
    for (int s = 0; s < 4; s++) m += (int)byte_of(mn_hi, s) * (bs[8 + 2 * s] + bs[8 + 2 * s + 1]);
    int v = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        uint32_t q[8];
        w.words_aligned<8>(o + 16 + 32 * j, q);
        const uint32_t e = 256u * u + 64u * j;
        const uint4 l0 = a.qvec(e), l1 = a.qvec(e + 16), h0 = a.qvec(e + 32), h1 = a.qvec(e + 48);
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
// (GGUF order, a reading).  84-byte blocks in 4-byte aligned rows: aligned.
__device__ __forceinline__ void q2_K_isums(const SmemBytes& w, uint32_t o, const ActView& a, int u, int* value,
                                           int* minterm, uint32_t* d_bits, uint32_t* dmin_bits) {
    uint32_t scw[4];
    w.words_aligned<4>(o, scw);
    const uint32_t dd = lds32(w.base + o + 80);
    *d_bits = dd & 0xFFFFu;
    *dmin_bits = dd >> 16;
    const int* bs = a.s + 16 * u;
    int m = 0, v = 0;
#pragma unroll
    for (int g = 0; g < 16; g++) m += (int)(byte_of(scw[g >> 2], g & 3) >> 4) * bs[g];
#pragma unroll
    for (int h = 0; h < 2; h++) {
        uint32_t q[8];
        w.words_aligned<8>(o + 16 + 32 * h, q);
#pragma unroll
        for (int s = 0; s < 4; s++) {
            const uint32_t e = 256u * u + 128u * h + 32u * s;
            const uint4 a0 = a.qvec(e), a1 = a.qvec(e + 16);
            const uint32_t sh = 2u * s;
            int g0 = 0, g1 = 0;
            g0 = dp4a((q[0] >> sh) & 0x03030303u, a0.x, g0);
            g0 = dp4a((q[1] >> sh) & 0x03030303u, a0.y, g0);
            g0 = dp4a((q[2] >> sh) & 0x03030303u, a0.z, g0);
            g0 = dp4a((q[3] >> sh) & 0x03030303u, a0.w, g0);
            g1 = dp4a((q[4] >> sh) & 0x03030303u, a1.x, g1);
            g1 = dp4a((q[5] >> sh) & 0x03030303u, a1.y, g1);
            g1 = dp4a((q[6] >> sh) & 0x03030303u, a1.z, g1);
            g1 = dp4a((q[7] >> sh) & 0x03030303u, a1.w, g1);
            const int g = 8 * h + 2 * s;
            v += (int)(byte_of(scw[g >> 2], g & 3) & 15u) * g0;
            v += (int)(byte_of(scw[(g + 1) >> 2], (g + 1) & 3) & 15u) * g1;
        }
    }
    *value = v;
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
    const int* bs = a.s + 16 * u;
    int m = 0, v = 0;
#pragma unroll
    for (int g = 0; g < 16; g++) m += (int)(int8_t)byte_of(scw[g >> 2], g & 3) * bs[g];
#pragma unroll
    for (int n = 0; n < 2; n++) {
        uint32_t A[8], B[8], H[8];
        w.words<8>(o + 64 * n, A);
        w.words<8>(o + 64 * n + 32, B);
        w.words<8>(o + 128 + 32 * n, H);
        int acc[4][2];
#pragma unroll
        for (int k = 0; k < 4; k++) acc[k][0] = acc[k][1] = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t q0 = (A[i] & 0x0F0F0F0Fu) | ((H[i] << 4) & 0x30303030u);
            const uint32_t q1 = (B[i] & 0x0F0F0F0Fu) | ((H[i] << 2) & 0x30303030u);
            const uint32_t q2 = ((A[i] >> 4) & 0x0F0F0F0Fu) | (H[i] & 0x30303030u);
            const uint32_t q3 = ((B[i] >> 4) & 0x0F0F0F0Fu) | ((H[i] >> 2) & 0x30303030u);
            const uint32_t e = 256u * u + 128u * n + 4u * i;
            const int half = i >> 2;
            acc[0][half] = dp4a(q0, a.qword(e), acc[0][half]);
            acc[1][half] = dp4a(q1, a.qword(e + 32), acc[1][half]);
            acc[2][half] = dp4a(q2, a.qword(e + 64), acc[2][half]);
            acc[3][half] = dp4a(q3, a.qword(e + 96), acc[3][half]);
        }
#pragma unroll
        for (int k = 0; k < 4; k++) {
#pragma unroll
            for (int hf = 0; hf < 2; hf++) {
                const int g = 8 * n + 2 * k + hf;
                v += (int)(int8_t)byte_of(scw[g >> 2], g & 3) * acc[k][hf];
            }
        }
    }
    *value = v;
    *minterm = m;
}

// ---------------------------------------------------------------- activation unpack
// Unpacks one activation row (Q8_0 or Q8_K blocks in global memory, row base
// at least 2-byte aligned) into the shared-memory ActView arrays.  All threads
// of the CTA take part; the caller synchronizes afterwards.
__device__ __forceinline__ void unpack_q8_0_row(const uint8_t* __restrict__ row, int K, uint8_t* q, float* d,
                                                int* s) {
    const int nb = K / 32;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        const unsigned short* p = reinterpret_cast<const unsigned short*>(row + 34 * b);
        d[b] = h2f(p[0]);
        uint32_t* qo = reinterpret_cast<uint32_t*>(q + 32 * b);
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t wv = (uint32_t)p[1 + 2 * i] | ((uint32_t)p[2 + 2 * i] << 16);
            qo[i] = wv;
            sum = dp4a(wv, 0x01010101u, sum);
        }
        s[b] = sum;
    }
}

__device__ __forceinline__ void unpack_q8_K_row(const uint8_t* __restrict__ row, int K, uint8_t* q, float* d,
                                                int* s) {
    const int ns = K / 256;
    // 73 words per block: d, 64 code words, 8 bsum words
    for (int i = threadIdx.x; i < ns * 73; i += blockDim.x) {
        const int u = i / 73, k = i % 73;
        const uint32_t wv = *reinterpret_cast<const uint32_t*>(row + 292 * u + 4 * k);
        if (k == 0) {
            d[u] = __uint_as_float(wv);
        } else if (k <= 64) {
            *reinterpret_cast<uint32_t*>(q + 256 * u + 4 * (k - 1)) = wv;
        } else {
            const int g = 2 * (k - 65);
            s[16 * u + g] = (int)(int16_t)(wv & 0xFFFFu);
            s[16 * u + g + 1] = (int)(int16_t)(wv >> 16);
        }
    }
}

}  // namespace qmm

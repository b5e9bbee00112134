// quantize.cu -- the activation quantizers (Q8_0, Q8_K) on the hot path, and
// the weight quantizers (Q4_0, Q4_K, Q6_K, Q2_K, Q4_1, Q5_0, Q5_1, Q5_K) used
// to prepare inputs.
//
// Every float operation is written with an explicitly IEEE-rounded intrinsic
// (__fdiv_rn, __fmul_rn, __fadd_rn, __float2int_rn, __float2half_rn), so that
// no multiply-add is contracted and each step rounds once, as the pages'
// scalar definitions do; the codes and scales are therefore bit-identical to a
// scalar implementation of the same steps ([krafla] "Architecture", Numerics:
// "quantize_q8 gives the same bits on every ISA").  The max reductions are
// exact in any order.
#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

static __device__ unsigned int g_quantize_error = 0;  // bounds records of a bounds-checked build

// ---------------------------------------------------------------- Q8_0 activations
// [minfer] "10 . CPU matmul: quantized weights x Q8_0 activations" s3.2 (the
// activation quantizers): per 32 values amax = max|x|, d = amax/127 stored as
// f16, inverse 127/amax (0 for an all-zero block), codes rne(x * inverse)
// saturated to int8.  Eight threads per block, four values each; the flat
// [M][K] input is a flat array of blocks because K is a multiple of 32.
// With pdl set the kernel is a link of a programmatic-dependent-launch chain:
// it lets the consumer launch (and start streaming its weights) at once, and
// waits for the previous grid before it reads x or writes xq.
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float4* __restrict__ x, uint8_t* __restrict__ out,
                                                            int64_t nblocks, int pdl) {
    if (pdl) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t b = gt >> 3;
    const bool active = b < nblocks && QMM_IN_BOUNDS(g_quantize_error, b * 34 + 33, nblocks * 34);
    const float4 v = active ? x[gt] : make_float4(0.f, 0.f, 0.f, 0.f);
    quant_q8_0_part(v, active, (int)(gt & 7), out + (active ? b * 34 : 0));
}

// ---------------------------------------------------------------- Q8_K activations
// [minfer] s3.2 (quantize_row_q8_k_buf): per 256 values amax, f32 d = amax/127,
// codes saturated to [-128, 127], bsums[g] = exact sum of the 16 saturated codes
// of group g.  One warp per super-block, eight values per lane: lanes 2g and
// 2g+1 hold group g.
__global__ void __launch_bounds__(256) quantize_q8_K_kernel(const float4* __restrict__ x, uint8_t* __restrict__ out,
                                                            int64_t nblocks, int pdl) {
    if (pdl) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (b >= nblocks) return;  // whole warps leave together
    if (!QMM_IN_BOUNDS(g_quantize_error, b * 292 + 291, nblocks * 292)) return;
    quant_q8_K_lane(x[b * 64 + 2 * lane], x[b * 64 + 2 * lane + 1], lane, out + b * 292);
}

// ---------------------------------------------------------------- Q4_0 weights
// [ggml] "ggml Q4_0 vec_dot Walkthrough" s1.1 and [kvad] "The scale that wasted
// a code": m = the value of largest magnitude (first on a tie), d = m / -8,
// codes min(15, trunc(x * (1/d) + 8.5)), byte j = code j | code j+16 << 4.
__global__ void quantize_q4_0_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float* xb = x + b * 32;
    float amax = 0.0f, m = 0.0f;
    for (int i = 0; i < 32; i++) {
        const float v = xb[i];
        if (fabsf(v) > amax) { amax = fabsf(v); m = v; }
    }
    const float d = __fdiv_rn(m, -8.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    uint8_t* ob = out + b * 18;
    st_u16(ob, f2h_bits(d));
    for (int j = 0; j < 16; j++) {
        const int c0 = clampi(__float2int_rz(__fadd_rn(__fmul_rn(xb[j], id), 8.5f)), 0, 15);
        const int c1 = clampi(__float2int_rz(__fadd_rn(__fmul_rn(xb[j + 16], id), 8.5f)), 0, 15);
        ob[2 + j] = (uint8_t)(c0 | (c1 << 4));
    }
}

// ---------------------------------------------------------------- Q4_K weights
// A reading (the pages give no K-quant quantizer): per sub-block s of 32,
// min_s = max(0, -min x), scale_s = (max x + min_s)/15; d = max scale_s/63,
// dmin = max min_s/63 stored as f16; 6-bit sc_s = rne(scale_s/d), m_s =
// rne(min_s/dmin); codes rne((x + f16(dmin)*m_s) / (f16(d)*sc_s)) in 0..15.
// Layout ([minfer] s3.2): d @0, dmin @2, packed scales @4 (GGUF packing),
// qs[32j + l] = code(64j + l) | code(64j + 32 + l) << 4.
__global__ void quantize_q4_K_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float* xb = x + b * 256;
    uint8_t* ob = out + b * 144;
    float scl[8], mns[8];
    float maxscl = 0.0f, maxmin = 0.0f;
#pragma unroll
    for (int s = 0; s < 8; s++) {
        float lo = xb[32 * s], hi = xb[32 * s];
        for (int i = 1; i < 32; i++) {
            const float v = xb[32 * s + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        mns[s] = lo < 0.0f ? -lo : 0.0f;
        scl[s] = __fdiv_rn(__fadd_rn(hi, mns[s]), 15.0f);
        if (scl[s] > maxscl) maxscl = scl[s];
        if (mns[s] > maxmin) maxmin = mns[s];
    }
    const float d = __fdiv_rn(maxscl, 63.0f), dmin = __fdiv_rn(maxmin, 63.0f);
    const uint32_t dh = f2h_bits(d), dmh = f2h_bits(dmin);
    st_u16(ob, dh);
    st_u16(ob + 2, dmh);
    int sc[8], mn[8];
#pragma unroll
    for (int s = 0; s < 8; s++) {
        sc[s] = d > 0.0f ? clampi(__float2int_rn(__fdiv_rn(scl[s], d)), 0, 63) : 0;
        mn[s] = dmin > 0.0f ? clampi(__float2int_rn(__fdiv_rn(mns[s], dmin)), 0, 63) : 0;
    }
#pragma unroll
    for (int s = 0; s < 4; s++) {
        ob[4 + s] = (uint8_t)((sc[s] & 63) | ((sc[s + 4] >> 4) << 6));
        ob[8 + s] = (uint8_t)((mn[s] & 63) | ((mn[s + 4] >> 4) << 6));
        ob[12 + s] = (uint8_t)((sc[s + 4] & 15) | ((mn[s + 4] & 15) << 4));
    }
    const float df = h2f(dh), dmf = h2f(dmh);
    float ds[8], dm[8];
#pragma unroll
    for (int s = 0; s < 8; s++) {
        ds[s] = __fmul_rn(df, (float)sc[s]);
        dm[s] = __fmul_rn(dmf, (float)mn[s]);
    }
#pragma unroll
    for (int j = 0; j < 4; j++) {
        for (int l = 0; l < 32; l++) {
            const int s0 = 2 * j, s1 = 2 * j + 1;
            const float v0 = xb[64 * j + l], v1 = xb[64 * j + 32 + l];
            const int c0 = ds[s0] > 0.0f ? clampi(__float2int_rn(__fdiv_rn(__fadd_rn(v0, dm[s0]), ds[s0])), 0, 15) : 0;
            const int c1 = ds[s1] > 0.0f ? clampi(__float2int_rn(__fdiv_rn(__fadd_rn(v1, dm[s1]), ds[s1])), 0, 15) : 0;
            ob[16 + 32 * j + l] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

// ---------------------------------------------------------------- Q2_K weights
// [ggml] s1.2 layout (scales[16] @0 = sc | m << 4, qs[64] @16, d @80, dmin @82);
// quantizer a reading: the Q4_K scheme over 16 groups of 16 with /3 and /15,
// 4-bit sc and m, codes 0..3; element 128h + 32s + l in bits 2s of qs[32h + l].
__global__ void quantize_q2_K_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float* xb = x + b * 256;
    uint8_t* ob = out + b * 84;
    float scl[16], mns[16];
    float maxscl = 0.0f, maxmin = 0.0f;
#pragma unroll
    for (int g = 0; g < 16; g++) {
        float lo = xb[16 * g], hi = xb[16 * g];
        for (int i = 1; i < 16; i++) {
            const float v = xb[16 * g + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        mns[g] = lo < 0.0f ? -lo : 0.0f;
        scl[g] = __fdiv_rn(__fadd_rn(hi, mns[g]), 3.0f);
        if (scl[g] > maxscl) maxscl = scl[g];
        if (mns[g] > maxmin) maxmin = mns[g];
    }
    const float d = __fdiv_rn(maxscl, 15.0f), dmin = __fdiv_rn(maxmin, 15.0f);
    const uint32_t dh = f2h_bits(d), dmh = f2h_bits(dmin);
    st_u16(ob + 80, dh);
    st_u16(ob + 82, dmh);
    const float df = h2f(dh), dmf = h2f(dmh);
    float ds[16], dm[16];
#pragma unroll
    for (int g = 0; g < 16; g++) {
        const int sc = d > 0.0f ? clampi(__float2int_rn(__fdiv_rn(scl[g], d)), 0, 15) : 0;
        const int mn = dmin > 0.0f ? clampi(__float2int_rn(__fdiv_rn(mns[g], dmin)), 0, 15) : 0;
        ob[g] = (uint8_t)(sc | (mn << 4));
        ds[g] = __fmul_rn(df, (float)sc);
        dm[g] = __fmul_rn(dmf, (float)mn);
    }
    for (int h = 0; h < 2; h++) {
        for (int l = 0; l < 32; l++) {
            uint32_t byte = 0;
#pragma unroll
            for (int s = 0; s < 4; s++) {
                const int e = 128 * h + 32 * s + l, g = e >> 4;
                const int c = ds[g] > 0.0f ? clampi(__float2int_rn(__fdiv_rn(__fadd_rn(xb[e], dm[g]), ds[g])), 0, 3) : 0;
                byte |= (uint32_t)c << (2 * s);
            }
            ob[16 + 32 * h + l] = (uint8_t)byte;
        }
    }
}

// ---------------------------------------------------------------- Q6_K weights
// Layout a reading (GGUF): ql[128] @0, qh[64] @128, int8 scales[16] @192, f16 d
// @208.  Quantizer a reading: per group the signed extreme m_g (first on a
// tie), s_g = m_g / -32, d = max|s_g| / 127, sc_g = rne(s_g/d), codes
// rne(x / (f16(d)*sc_g)) in -32..31, stored +32.
__global__ void quantize_q6_K_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float* xb = x + b * 256;
    uint8_t* ob = out + b * 210;
    float sg[16];
    float amax_s = 0.0f;
#pragma unroll
    for (int g = 0; g < 16; g++) {
        float amax = 0.0f, m = 0.0f;
        for (int i = 0; i < 16; i++) {
            const float v = xb[16 * g + i];
            if (fabsf(v) > amax) { amax = fabsf(v); m = v; }
        }
        sg[g] = __fdiv_rn(m, -32.0f);
        if (fabsf(sg[g]) > amax_s) amax_s = fabsf(sg[g]);
    }
    const float d = __fdiv_rn(amax_s, 127.0f);
    const uint32_t dh = f2h_bits(d);
    st_u16(ob + 208, dh);
    const float df = h2f(dh);
    float ds[16];
#pragma unroll
    for (int g = 0; g < 16; g++) {
        const int sc = d > 0.0f ? clampi(__float2int_rn(__fdiv_rn(sg[g], d)), -128, 127) : 0;
        ob[192 + g] = (uint8_t)(int8_t)sc;
        ds[g] = __fmul_rn(df, (float)sc);
    }
    for (int h = 0; h < 2; h++) {
        for (int l = 0; l < 32; l++) {
            int c[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int e = 128 * h + 32 * k + l, g = e >> 4;
                const int q = ds[g] != 0.0f ? clampi(__float2int_rn(__fdiv_rn(xb[e], ds[g])), -32, 31) : 0;
                c[k] = q + 32;
            }
            ob[64 * h + l] = (uint8_t)((c[0] & 15) | ((c[2] & 15) << 4));
            ob[64 * h + l + 32] = (uint8_t)((c[1] & 15) | ((c[3] & 15) << 4));
            ob[128 + 32 * h + l] = (uint8_t)((c[0] >> 4) | ((c[1] >> 4) << 2) | ((c[2] >> 4) << 4) | ((c[3] >> 4) << 6));
        }
    }
}

// ---------------------------------------------------------------- host side
static qmm_status check_quant_args(int t, const float* x, const void* xq, int64_t M, int64_t K) {
    if (!x || !xq) return QMM_E_NULL;
    if (M < 1 || K < 1 || M > kMaxDim || K > kMaxDim) return QMM_E_SHAPE;
    if (K % block_values_of(t)) return QMM_E_SHAPE;
    if (!aligned16(x) || !aligned16(xq)) return QMM_E_ALIGN;
    return QMM_OK;
}

qmm_status quantize_act_launch(int act, const float* x, void* xq, int64_t M, int64_t K, cudaStream_t stream,
                               bool pdl) {
    int64_t grid;
    int64_t nblocks;
    if (act == QMM_Q8_0) {
        nblocks = M * (K / 32);
        grid = (nblocks * 8 + 255) / 256;
    } else {
        nblocks = M * (K / 256);
        grid = (nblocks * 32 + 255) / 256;
    }
    if (grid > 0x7FFFFFFFLL) return QMM_E_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e =
        act == QMM_Q8_0
            ? cudaLaunchKernelEx(&cfg, quantize_q8_0_kernel, (const float4*)x, (uint8_t*)xq, nblocks, pdl ? 1 : 0)
            : cudaLaunchKernelEx(&cfg, quantize_q8_K_kernel, (const float4*)x, (uint8_t*)xq, nblocks, pdl ? 1 : 0);
    return e == cudaSuccess ? QMM_OK : QMM_E_CUDA;
}

// ---------------------------------------------------------------- Q4_1 / Q5_1 weights
// A reading (the pages give no quantizer for them): a min/max grid per block of
// 32, m = min x, d = (max x - m) / levels, codes min(levels, trunc((x - m) *
// (1/d) + 0.5)) with the f32 d and m, both stored as f16.  Layouts (GGUF): Q4_1
// d @0, m @2, nibbles @4; Q5_1 d @0, m @2, fifth bits @4, nibbles @8.
template <int LEVELS, int BB, int QH, int QS>
__global__ void quantize_minmax_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float* xb = x + b * 32;
    float lo = xb[0], hi = xb[0];
    for (int i = 1; i < 32; i++) {
        const float v = xb[i];
        if (v < lo) lo = v;
        if (v > hi) hi = v;
    }
    const float d = __fdiv_rn(__fsub_rn(hi, lo), (float)LEVELS);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    uint8_t* ob = out + b * BB;
    st_u16(ob, f2h_bits(d));
    st_u16(ob + 2, f2h_bits(lo));
    uint32_t qh = 0;
    for (int j = 0; j < 16; j++) {
        const int c0 = clampi(__float2int_rz(__fadd_rn(__fmul_rn(__fsub_rn(xb[j], lo), id), 0.5f)), 0, LEVELS);
        const int c1 = clampi(__float2int_rz(__fadd_rn(__fmul_rn(__fsub_rn(xb[j + 16], lo), id), 0.5f)), 0, LEVELS);
        ob[QS + j] = (uint8_t)((c0 & 15) | ((c1 & 15) << 4));
        qh |= (uint32_t)(c0 >> 4) << j;
        qh |= (uint32_t)(c1 >> 4) << (j + 16);
    }
    if constexpr (QH >= 0) {
        st_u16(ob + QH, qh & 0xFFFFu);
        st_u16(ob + QH + 2, qh >> 16);
    }
}

// ---------------------------------------------------------------- Q5_0 weights
// A reading: the Q4_0 scheme on five bits.  m = the value of largest magnitude
// (first on a tie), d = m / -16, codes min(31, trunc(x * (1/d) + 16.5)).
// Layout (GGUF): d @0, fifth bits @2, nibbles @6.
__global__ void quantize_q5_0_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float* xb = x + b * 32;
    float amax = 0.0f, m = 0.0f;
    for (int i = 0; i < 32; i++) {
        const float v = xb[i];
        if (fabsf(v) > amax) { amax = fabsf(v); m = v; }
    }
    const float d = __fdiv_rn(m, -16.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    uint8_t* ob = out + b * 22;
    st_u16(ob, f2h_bits(d));
    uint32_t qh = 0;
    for (int j = 0; j < 16; j++) {
        const int c0 = clampi(__float2int_rz(__fadd_rn(__fmul_rn(xb[j], id), 16.5f)), 0, 31);
        const int c1 = clampi(__float2int_rz(__fadd_rn(__fmul_rn(xb[j + 16], id), 16.5f)), 0, 31);
        ob[6 + j] = (uint8_t)((c0 & 15) | ((c1 & 15) << 4));
        qh |= (uint32_t)(c0 >> 4) << j;
        qh |= (uint32_t)(c1 >> 4) << (j + 16);
    }
    st_u16(ob + 2, qh & 0xFFFFu);
    st_u16(ob + 4, qh >> 16);
}

// ---------------------------------------------------------------- Q5_K weights
// A reading: the Q4_K scheme with codes 0..31 (scale_s = (max x + min_s)/31).
// Layout (GGUF): d @0, dmin @2, packed scales @4, qh[32] @16, qs[128] @48;
// element 64j + l: low nibble of qs[32j + l], fifth bit 2j of qh[l]; element
// 64j + 32 + l: high nibble, bit 2j + 1.
__global__ void quantize_q5_K_kernel(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float* xb = x + b * 256;
    uint8_t* ob = out + b * 176;
    float scl[8], mns[8];
    float maxscl = 0.0f, maxmin = 0.0f;
#pragma unroll
    for (int s = 0; s < 8; s++) {
        float lo = xb[32 * s], hi = xb[32 * s];
        for (int i = 1; i < 32; i++) {
            const float v = xb[32 * s + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        mns[s] = lo < 0.0f ? -lo : 0.0f;
        scl[s] = __fdiv_rn(__fadd_rn(hi, mns[s]), 31.0f);
        if (scl[s] > maxscl) maxscl = scl[s];
        if (mns[s] > maxmin) maxmin = mns[s];
    }
    const float d = __fdiv_rn(maxscl, 63.0f), dmin = __fdiv_rn(maxmin, 63.0f);
    const uint32_t dh = f2h_bits(d), dmh = f2h_bits(dmin);
    st_u16(ob, dh);
    st_u16(ob + 2, dmh);
    int sc[8], mn[8];
#pragma unroll
    for (int s = 0; s < 8; s++) {
        sc[s] = d > 0.0f ? clampi(__float2int_rn(__fdiv_rn(scl[s], d)), 0, 63) : 0;
        mn[s] = dmin > 0.0f ? clampi(__float2int_rn(__fdiv_rn(mns[s], dmin)), 0, 63) : 0;
    }
#pragma unroll
    for (int s = 0; s < 4; s++) {
        ob[4 + s] = (uint8_t)((sc[s] & 63) | ((sc[s + 4] >> 4) << 6));
        ob[8 + s] = (uint8_t)((mn[s] & 63) | ((mn[s + 4] >> 4) << 6));
        ob[12 + s] = (uint8_t)((sc[s + 4] & 15) | ((mn[s + 4] & 15) << 4));
    }
    const float df = h2f(dh), dmf = h2f(dmh);
    float ds[8], dm[8];
#pragma unroll
    for (int s = 0; s < 8; s++) {
        ds[s] = __fmul_rn(df, (float)sc[s]);
        dm[s] = __fmul_rn(dmf, (float)mn[s]);
    }
    for (int l = 0; l < 32; l++) {
        uint32_t qh = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int s0 = 2 * j, s1 = 2 * j + 1;
            const float v0 = xb[64 * j + l], v1 = xb[64 * j + 32 + l];
            const int c0 = ds[s0] > 0.0f ? clampi(__float2int_rn(__fdiv_rn(__fadd_rn(v0, dm[s0]), ds[s0])), 0, 31) : 0;
            const int c1 = ds[s1] > 0.0f ? clampi(__float2int_rn(__fdiv_rn(__fadd_rn(v1, dm[s1]), ds[s1])), 0, 31) : 0;
            ob[48 + 32 * j + l] = (uint8_t)((c0 & 15) | ((c1 & 15) << 4));
            qh |= (uint32_t)((c0 >> 4) << (2 * j)) | (uint32_t)((c1 >> 4) << (2 * j + 1));
        }
        ob[16 + l] = (uint8_t)qh;
    }
}

// ---------------------------------------------------------------- RMSNorm + quantize
// [krafla] "Architecture", "Data flow for one token": h = rmsnorm(x) ; qa =
// quantize_q8(h).  One CTA per row: the norm's scale (rms_scale, a fixed-order
// sum of squares), then h = (x * s) * w handed to the same per-block quantizer
// arithmetic as quantize_q8_0_kernel / quantize_q8_K_kernel.
__global__ void __launch_bounds__(256) rmsnorm_quantize_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                               float eps, uint8_t* __restrict__ out, int K, int act,
                                                               int pdl) {
    extern __shared__ float rq_part[];
    if (pdl) {
        pdl_launch_dependents();
        pdl_wait();
    }
    const float* xr = x + (int64_t)blockIdx.x * K;
    const float sn = rms_scale(xr, K, rq_part, eps);
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (act == QMM_Q8_0) {
        uint8_t* orow = out + (int64_t)blockIdx.x * (K / 32) * 34;
        const int n4 = K / 4, n4r = (n4 + 31) / 32 * 32;  // whole warps: the 8-lane shuffles need them
        for (int gt = warp * 32 + lane; gt < n4r; gt += blockDim.x) {
            const bool active = gt < n4;
            const float4 v = active ? norm4(x4[gt], sn, w4[gt]) : make_float4(0.f, 0.f, 0.f, 0.f);
            quant_q8_0_part(v, active, gt & 7, orow + (active ? (gt >> 3) * 34 : 0));
        }
    } else {
        uint8_t* orow = out + (int64_t)blockIdx.x * (K / 256) * 292;
        for (int b = warp; b < K / 256; b += blockDim.x >> 5) {
            const float4 v0 = norm4(x4[b * 64 + 2 * lane], sn, w4[b * 64 + 2 * lane]);
            const float4 v1 = norm4(x4[b * 64 + 2 * lane + 1], sn, w4[b * 64 + 2 * lane + 1]);
            quant_q8_K_lane(v0, v1, lane, orow + b * 292);
        }
    }
}

qmm_status rmsnorm_quantize_launch(int act, const float* x, const float* w, float eps, void* xq, int64_t M, int64_t K,
                                   cudaStream_t stream, bool pdl) {
    if (M > 0x7FFFFFFFLL) return QMM_E_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)M);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = (size_t)rms_scratch_floats((int)K, 256) * sizeof(float);
    if (cfg.dynamicSmemBytes > 48 * 1024 &&
        cudaFuncSetAttribute(rmsnorm_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)cfg.dynamicSmemBytes) != cudaSuccess)
        return QMM_E_CUDA;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, rmsnorm_quantize_kernel, x, w, eps, (uint8_t*)xq, (int)K, act, pdl ? 1 : 0);
    return e == cudaSuccess ? QMM_OK : QMM_E_CUDA;
}

template <class Kern>
static qmm_status launch_weight_quant(Kern kern, int t, const float* w, void* wq, int64_t N, int64_t K,
                                      cudaStream_t stream) {
    qmm_status st = check_quant_args(t, w, wq, N, K);
    if (st != QMM_OK) return st;
    const int64_t nblocks = N * (K / block_values_of(t));
    const int64_t grid = (nblocks + 127) / 128;
    if (grid > 0x7FFFFFFFLL) return QMM_E_SHAPE;
    kern<<<(unsigned)grid, 128, 0, stream>>>(w, (uint8_t*)wq, nblocks);
    return launch_status();
}

}  // namespace qmm

using namespace qmm;

extern "C" {

qmm_status qmm_quantize_q8_0(const float* x, void* xq, int64_t M, int64_t K, qmm_stream_t stream) {
    qmm_status st = check_quant_args(QMM_Q8_0, x, xq, M, K);
    if (st != QMM_OK) return st;
    return quantize_act_launch(QMM_Q8_0, x, xq, M, K, (cudaStream_t)stream, false);
}

qmm_status qmm_quantize_q8_K(const float* x, void* xq, int64_t M, int64_t K, qmm_stream_t stream) {
    qmm_status st = check_quant_args(QMM_Q8_K, x, xq, M, K);
    if (st != QMM_OK) return st;
    return quantize_act_launch(QMM_Q8_K, x, xq, M, K, (cudaStream_t)stream, false);
}

qmm_status qmm_rmsnorm_quantize(int act, const float* x, const float* w, float eps, void* xq, int64_t M, int64_t K,
                                qmm_stream_t stream) {
    if (act != QMM_Q8_0 && act != QMM_Q8_K) return QMM_E_TYPE;
    qmm_status st = check_quant_args(act, x, xq, M, K);
    if (st != QMM_OK) return st;
    if (!w) return QMM_E_NULL;
    if (K > kMaxK) return QMM_E_SHAPE;
    if (!aligned16(w)) return QMM_E_ALIGN;
    return rmsnorm_quantize_launch(act, x, w, eps, xq, M, K, (cudaStream_t)stream, false);
}

qmm_status qmm_quantize_q4_0(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_q4_0_kernel, QMM_Q4_0, w, wq, N, K, (cudaStream_t)stream);
}
qmm_status qmm_quantize_q4_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_q4_K_kernel, QMM_Q4_K, w, wq, N, K, (cudaStream_t)stream);
}
qmm_status qmm_quantize_q6_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_q6_K_kernel, QMM_Q6_K, w, wq, N, K, (cudaStream_t)stream);
}
qmm_status qmm_quantize_q2_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_q2_K_kernel, QMM_Q2_K, w, wq, N, K, (cudaStream_t)stream);
}
qmm_status qmm_quantize_q4_1(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_minmax_kernel<15, 20, -1, 4>, QMM_Q4_1, w, wq, N, K, (cudaStream_t)stream);
}
qmm_status qmm_quantize_q5_0(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_q5_0_kernel, QMM_Q5_0, w, wq, N, K, (cudaStream_t)stream);
}
qmm_status qmm_quantize_q5_1(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_minmax_kernel<31, 24, 4, 8>, QMM_Q5_1, w, wq, N, K, (cudaStream_t)stream);
}
qmm_status qmm_quantize_q5_K(const float* w, void* wq, int64_t N, int64_t K, qmm_stream_t stream) {
    return launch_weight_quant(quantize_q5_K_kernel, QMM_Q5_K, w, wq, N, K, (cudaStream_t)stream);
}

unsigned qmm_internal_quantize_error(int clear) {
    unsigned v = 0;
    cudaMemcpyFromSymbol(&v, g_quantize_error, sizeof(v));
    if (clear) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_quantize_error, &z, sizeof(z));
    }
    return v;
}

}  // extern "C"

// getrows.cu -- the embedding lookup: out[r] = the dequantized row ids[r] of a
// block-quantized matrix ([minfer] "10 . CPU matmul: quantized weights x Q8_0
// activations" s3.2, "The embedding 'matmul'": for each token id, walk its row
// block by block and dequantize, scale x code, into the output row).
//
// Every value is computed in f32 with at most one rounding, so it equals the
// exact dequantized value rounded once to f32, the same on every run and on
// every backend:
//   Q4_0  d * (n - 8), Q8_0  d * q                       exact products
//   Q4_K  fma(d*sc, q, -(dmin*m)), Q2_K the same         d*sc and dmin*m exact
//   Q6_K  (d*sc) * (q - 32)                             exact (18 + 6 bits)
//   Q4_1, Q5_1  fma(d, q, m)      Q5_0  d * (q - 16)      Q5_K as Q4_K
// Layouts as in the decoders (GGUF readings for the K-quants and the types
// with a fifth bit or a min).
#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

static __device__ unsigned int g_getrows_error = 0;
constexpr unsigned kErrIndex = 2u;

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) { return *reinterpret_cast<const unsigned short*>(p); }

// 32 values of sub-block s (32-value unit s of the row) from the row's bytes
template <int WT>
__device__ __forceinline__ void dequant32(const uint8_t* __restrict__ row, int s, float* v) {
    if constexpr (WT == QMM_Q4_0) {
        const uint8_t* b = row + 18 * s;
        const float d = h2f(ld_u16(b));
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const uint32_t byte = b[2 + j];
            v[j] = d * (float)((int)(byte & 15u) - 8);
            v[j + 16] = d * (float)((int)(byte >> 4) - 8);
        }
    } else if constexpr (WT == QMM_Q8_0) {
        const uint8_t* b = row + 34 * s;
        const float d = h2f(ld_u16(b));
#pragma unroll
        for (int j = 0; j < 32; j++) v[j] = d * (float)(int8_t)b[2 + j];
    } else if constexpr (WT == QMM_Q4_K) {
        const uint8_t* b = row + 144 * (s >> 3);
        const int sb = s & 7;
        const float d = h2f(ld_u16(b)), dmin = h2f(ld_u16(b + 2));
        const uint8_t* sc = b + 4;
        int scale, mn;
        if (sb < 4) {
            scale = sc[sb] & 63;
            mn = sc[sb + 4] & 63;
        } else {
            scale = (sc[sb + 4] & 15) | ((sc[sb - 4] >> 6) << 4);
            mn = (sc[sb + 4] >> 4) | ((sc[sb] >> 6) << 4);
        }
        const float dl = d * (float)scale, ml = dmin * (float)mn;
        const uint8_t* q = b + 16 + 32 * (sb >> 1);
        const int sh = (sb & 1) * 4;
#pragma unroll
        for (int j = 0; j < 32; j++) v[j] = fmaf(dl, (float)((q[j] >> sh) & 15), -ml);
    } else if constexpr (WT == QMM_Q2_K) {
        const uint8_t* b = row + 84 * (s >> 3);
        const int sb = s & 7;  // values 32sb..32sb+31: groups 2sb, 2sb+1
        const float d = h2f(ld_u16(b + 80)), dmin = h2f(ld_u16(b + 82));
        const int h = sb >> 2, sh = 2 * (sb & 3);
        const uint8_t* q = b + 16 + 32 * h;
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const uint32_t g = b[2 * sb + half];
            const float dl = d * (float)(g & 15u), ml = dmin * (float)(g >> 4);
#pragma unroll
            for (int j = 0; j < 16; j++) v[16 * half + j] = fmaf(dl, (float)((q[16 * half + j] >> sh) & 3), -ml);
        }
    } else if constexpr (WT == QMM_Q4_1 || WT == QMM_Q5_0 || WT == QMM_Q5_1) {
        constexpr int BB = Fmt<WT>::BB;
        constexpr int QS = WT == QMM_Q4_1 ? 4 : (WT == QMM_Q5_0 ? 6 : 8);  // nibbles
        constexpr int QH = WT == QMM_Q5_0 ? 2 : 4;                          // fifth bits
        const uint8_t* b = row + BB * s;
        const float d = h2f(ld_u16(b));
        const float m = WT == QMM_Q5_0 ? 0.0f : h2f(ld_u16(b + 2));
        uint32_t qh = 0;
        if constexpr (WT != QMM_Q4_1) qh = ld_u16(b + QH) | (ld_u16(b + QH + 2) << 16);
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const uint32_t byte = b[QS + j];
            int lo = (int)(byte & 15u), hi = (int)(byte >> 4);
            if constexpr (WT != QMM_Q4_1) {
                lo |= (int)((qh >> j) & 1u) << 4;
                hi |= (int)((qh >> (j + 16)) & 1u) << 4;
            }
            if constexpr (WT == QMM_Q5_0) {
                v[j] = d * (float)(lo - 16);
                v[j + 16] = d * (float)(hi - 16);
            } else {
                v[j] = fmaf(d, (float)lo, m);
                v[j + 16] = fmaf(d, (float)hi, m);
            }
        }
    } else if constexpr (WT == QMM_Q5_K) {
        const uint8_t* b = row + 176 * (s >> 3);
        const int sb = s & 7;
        const float d = h2f(ld_u16(b)), dmin = h2f(ld_u16(b + 2));
        const uint8_t* sc = b + 4;
        int scale, mn;
        if (sb < 4) {
            scale = sc[sb] & 63;
            mn = sc[sb + 4] & 63;
        } else {
            scale = (sc[sb + 4] & 15) | ((sc[sb - 4] >> 6) << 4);
            mn = (sc[sb + 4] >> 4) | ((sc[sb] >> 6) << 4);
        }
        const float dl = d * (float)scale, ml = dmin * (float)mn;
        const uint8_t* q = b + 48 + 32 * (sb >> 1);
        const uint8_t* qh = b + 16;
        const int sh = (sb & 1) * 4;  // sub-block sb: nibble (sb & 1), fifth bit sb of qh[l]
#pragma unroll
        for (int j = 0; j < 32; j++) {
            const int code = ((q[j] >> sh) & 15) | (((qh[j] >> sb) & 1) << 4);
            v[j] = fmaf(dl, (float)code, -ml);
        }
    } else {  // Q6_K
        const uint8_t* b = row + 210 * (s >> 3);
        const int sb = s & 7, n = sb >> 2, part = sb & 3;
        const float d = h2f(ld_u16(b + 208));
        const uint8_t* ql = b + 64 * n + 32 * (part & 1);
        const uint8_t* qh = b + 128 + 32 * n;
        const int lsh = (part >> 1) * 4, hsh = 2 * part;
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const float dl = d * (float)(int8_t)b[192 + 2 * sb + half];
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int l = 16 * half + j;
                const int q = ((ql[l] >> lsh) & 15) | (((qh[l] >> hsh) & 3) << 4);
                v[l] = dl * (float)(q - 32);
            }
        }
    }
}

// One thread per 32-value unit of an output row; consecutive threads write
// consecutive 128-byte pieces of a row.
template <int WT>
__global__ void __launch_bounds__(256) getrows_kernel(const uint8_t* __restrict__ W, const int32_t* __restrict__ ids,
                                                      float* __restrict__ out, int64_t R, int N, int K) {
    const int units = K / 32;
    const uint64_t rb = (uint64_t)(K / Fmt<WT>::BV) * Fmt<WT>::BB;
    const int64_t total = R * units;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / units;
        const int s = (int)(i - r * units);
        const int id = ids[r];
        float v[32];
        if (id < 0 || id >= N) {
            if (s == 0) atomicOr(&g_getrows_error, kErrIndex);
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] = 0.0f;
        } else {
            dequant32<WT>(W + (uint64_t)id * rb, s, v);
        }
        if (!QMM_IN_BOUNDS(g_getrows_error, r * (int64_t)K + 32 * s + 31, R * (int64_t)K)) continue;
        float4* o = reinterpret_cast<float4*>(out + r * (int64_t)K + 32 * s);
#pragma unroll
        for (int j = 0; j < 8; j++) o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
}

template <int WT>
static qmm_status launch_getrows(const void* W, const int32_t* ids, float* out, int64_t R, int64_t N, int64_t K,
                                 cudaStream_t stream) {
    DeviceInfo dev;
    qmm_status st = current_device(&dev);
    if (st != QMM_OK) return st;
    const int64_t total = R * (K / 32);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)dev.sms * 8;
    if (blocks > cap) blocks = cap;
    getrows_kernel<WT><<<(unsigned)blocks, 256, 0, stream>>>((const uint8_t*)W, ids, out, R, (int)N, (int)K);
    return launch_status();
}

}  // namespace qmm

using namespace qmm;

extern "C" {

qmm_status qmm_get_rows(int wtype, const void* W, const int32_t* ids, float* out, int64_t R, int64_t N, int64_t K,
                        qmm_stream_t stream) {
    if (act_type_of(wtype) < 0) return QMM_E_TYPE;
    if (!W || !ids || !out) return QMM_E_NULL;
    qmm_status st = check_shape(wtype, R, N, K);
    if (st != QMM_OK) return st;
    if (N > 0x7FFFFFFF) return QMM_E_SHAPE;
    if (!aligned16(W) || !aligned16(out) || ((uintptr_t)ids & 3u)) return QMM_E_ALIGN;
    cudaStream_t cs = (cudaStream_t)stream;
    switch (wtype) {
    case QMM_Q4_0: return launch_getrows<QMM_Q4_0>(W, ids, out, R, N, K, cs);
    case QMM_Q8_0: return launch_getrows<QMM_Q8_0>(W, ids, out, R, N, K, cs);
    case QMM_Q4_K: return launch_getrows<QMM_Q4_K>(W, ids, out, R, N, K, cs);
    case QMM_Q6_K: return launch_getrows<QMM_Q6_K>(W, ids, out, R, N, K, cs);
    case QMM_Q2_K: return launch_getrows<QMM_Q2_K>(W, ids, out, R, N, K, cs);
    case QMM_Q4_1: return launch_getrows<QMM_Q4_1>(W, ids, out, R, N, K, cs);
    case QMM_Q5_0: return launch_getrows<QMM_Q5_0>(W, ids, out, R, N, K, cs);
    case QMM_Q5_1: return launch_getrows<QMM_Q5_1>(W, ids, out, R, N, K, cs);
    case QMM_Q5_K: return launch_getrows<QMM_Q5_K>(W, ids, out, R, N, K, cs);
    default: return QMM_E_TYPE;
    }
}

unsigned qmm_internal_getrows_error(int clear) {
    unsigned v = 0;
    cudaMemcpyFromSymbol(&v, g_getrows_error, sizeof(v));
    if (clear) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_getrows_error, &z, sizeof(z));
    }
    return v;
}

}  // extern "C"

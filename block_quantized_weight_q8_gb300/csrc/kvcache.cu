// kvcache.cu -- the Q8 KV cache of decode attention ([krafla] "Architecture",
// Attention, "Q8 cache"): each position's K and V are kept per KV head as int8
// codes with one float scale, quantized by the activations' rule; each query
// head is quantized the same way; a score is an integer dot product, and the V
// sum widens the int8 values to float as it goes.
//
// A row is one head vector of hd values: f32 d @0, int8 codes @4 (4 + hd bytes;
// 68 at hd = 64).  The cache holds row (p, kvh) at (p*Hkv + kvh) * (4 + hd), so
// appending a position writes Hkv consecutive rows.  Query head h reads KV head
// h / (Hq/Hkv).
//
//   kv_quantize   one warp per row: amax, d = amax/127, codes rne(x*127/amax)
//   kv_scores     a CTA per (128 positions, KV head): the K rows of the tile and
//                 the group's query rows staged in shared memory, one thread per
//                 position computing the group's G integer dots with dp4a;
//                 score = ((dq*dk) * isum) * scale, each step rounded once
//   kv_wsum       pass 1: a CTA per (128-position chunk, KV head), one thread
//                 per (query head of the group, 4 columns), an f32 FMA chain over
//                 the chunk's positions; pass 2: the chunks' partial sums added
//                 in chunk order.  The chunking is fixed, so the result does not
//                 depend on the GPU it runs on.
#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

constexpr int kKvTile = 128;    // positions per CTA of the score kernel
constexpr int kKvChunk = 128;   // positions per partial sum of the V sum
constexpr int kKvMaxGroup = 8;  // query heads per KV head
constexpr int kKvMaxHd = 256;

__global__ void __launch_bounds__(256) kv_quantize_kernel(const float* __restrict__ x, uint8_t* __restrict__ out,
                                                          int64_t rows, int hd) {
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;  // whole warps leave together
    const float* xr = x + r * hd;
    uint8_t* o = out + r * (4 + hd);
    float amax = 0.0f;
    for (int i = lane; i < hd; i += 32) amax = fmaxf(amax, fabsf(xr[i]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float id = amax != 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    if (lane == 0) *reinterpret_cast<float*>(o) = __fdiv_rn(amax, 127.0f);
    for (int i = lane; i < hd; i += 32) o[4 + i] = (uint8_t)(int8_t)clampi(__float2int_rn(__fmul_rn(xr[i], id)), -128, 127);
}

// grid (tiles of kKvTile positions, Hkv); kKvTile threads
__global__ void __launch_bounds__(kKvTile) kv_scores_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ kc,
                                                            float* __restrict__ scores, int G, int Hkv, int64_t P,
                                                            int hd, float scale) {
    extern __shared__ __align__(16) uint32_t kv_smem[];
    const int nwd = (4 + hd) / 4;  // words per row (odd: hd % 16 == 0)
    uint32_t* qs = kv_smem;              // G rows
    uint32_t* ks = kv_smem + G * nwd;    // kKvTile rows
    const int kvh = blockIdx.y;
    const int64_t p0 = (int64_t)blockIdx.x * kKvTile;
    const int rows = P - p0 < kKvTile ? (int)(P - p0) : kKvTile;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t* qg = reinterpret_cast<const uint32_t*>(q + (int64_t)kvh * G * (4 + hd));
    for (int i = threadIdx.x; i < G * nwd; i += blockDim.x) qs[i] = qg[i];
    for (int r = warp; r < rows; r += kKvTile / 32) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(kc + ((p0 + r) * Hkv + kvh) * (int64_t)(4 + hd));
        for (int w = lane; w < nwd; w += 32) ks[r * nwd + w] = src[w];
    }
    __syncthreads();
    const int r = threadIdx.x;
    if (r >= rows) return;
    const uint32_t* kr = ks + r * nwd;
    int acc[kKvMaxGroup];
#pragma unroll
    for (int g = 0; g < kKvMaxGroup; g++) acc[g] = 0;
    for (int w = 1; w < nwd; w++) {
        const uint32_t kw = kr[w];
#pragma unroll
        for (int g = 0; g < kKvMaxGroup; g++)
            if (g < G) acc[g] = dp4a(kw, qs[g * nwd + w], acc[g]);
    }
    const float dk = __uint_as_float(kr[0]);
#pragma unroll
    for (int g = 0; g < kKvMaxGroup; g++) {
        if (g < G) {
            const float dq = __uint_as_float(qs[g * nwd]);
            const float s = __fmul_rn(__fmul_rn(__fmul_rn(dq, dk), (float)acc[g]), scale);
            scores[(int64_t)(kvh * G + g) * P + p0 + r] = s;
        }
    }
}

// pass 1: grid (chunks, Hkv); one thread per (g, column quad)
__global__ void __launch_bounds__(512) kv_wsum_partial_kernel(const float* __restrict__ w, const uint8_t* __restrict__ vc,
                                                              float* __restrict__ part, int G, int Hkv, int64_t P,
                                                              int hd) {
    const int nq = hd / 4;
    const int t = threadIdx.x;
    if (t >= G * nq) return;
    const int g = t / nq, quad = t - g * nq;
    const int kvh = blockIdx.y;
    const int c = blockIdx.x, nc = gridDim.x;
    const int h = kvh * G + g;
    const int64_t pa = (int64_t)c * kKvChunk;
    const int64_t pb = pa + kKvChunk < P ? pa + kKvChunk : P;
    const int64_t rb = 4 + hd;
    const float* wr = w + (int64_t)h * P;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll 4
    for (int64_t p = pa; p < pb; p++) {
        const uint8_t* row = vc + (p * Hkv + kvh) * rb;
        const float coef = __fmul_rn(wr[p], *reinterpret_cast<const float*>(row));
        const uint32_t v = *reinterpret_cast<const uint32_t*>(row + 4 + 4 * quad);
        a0 = __fmaf_rn(coef, (float)(int8_t)(v & 0xFFu), a0);
        a1 = __fmaf_rn(coef, (float)(int8_t)((v >> 8) & 0xFFu), a1);
        a2 = __fmaf_rn(coef, (float)(int8_t)((v >> 16) & 0xFFu), a2);
        a3 = __fmaf_rn(coef, (float)(int8_t)(v >> 24), a3);
    }
    float4* dst = reinterpret_cast<float4*>(part + (((int64_t)kvh * nc + c) * G + g) * hd + 4 * quad);
    *dst = make_float4(a0, a1, a2, a3);
}

// pass 2: one thread per output (h, i); the chunks in order
__global__ void __launch_bounds__(256) kv_wsum_reduce_kernel(const float* __restrict__ part, float* __restrict__ out,
                                                             int G, int Hq, int nc, int hd) {
    const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= (int64_t)Hq * hd) return;
    const int h = (int)(o / hd), i = (int)(o - (int64_t)h * hd);
    const int kvh = h / G, g = h - kvh * G;
    const float* src = part + ((int64_t)kvh * nc * G + g) * hd + i;
    const int64_t step = (int64_t)G * hd;
    float s = 0.0f;
    for (int c = 0; c < nc; c++) s = __fadd_rn(s, src[c * step]);
    out[o] = s;
}

static bool kv_hd_ok(int64_t hd) { return hd >= 16 && hd <= kKvMaxHd && hd % 16 == 0; }

static qmm_status kv_heads_ok(int64_t Hq, int64_t Hkv, int64_t P) {
    if (Hq < 1 || Hkv < 1 || P < 1 || Hq % Hkv || Hq / Hkv > kKvMaxGroup || Hkv > 65535) return QMM_E_SHAPE;
    if (P > 0x7FFFFFFFLL || P * Hq > ((int64_t)1 << 40)) return QMM_E_SHAPE;
    return QMM_OK;
}

static bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

}  // namespace qmm

using namespace qmm;

extern "C" {

size_t qmm_kv_row_bytes(int64_t hd) { return kv_hd_ok(hd) ? (size_t)(4 + hd) : 0; }

qmm_status qmm_kv_quantize(const float* x, void* out, int64_t rows, int64_t hd, qmm_stream_t stream) {
    if (!x || !out) return QMM_E_NULL;
    if (rows < 1 || !kv_hd_ok(hd) || rows > ((int64_t)1 << 36)) return QMM_E_SHAPE;
    if (!aligned4(x) || !aligned4(out)) return QMM_E_ALIGN;
    const int64_t grid = (rows * 32 + 255) / 256;
    if (grid > 0x7FFFFFFFLL) return QMM_E_SHAPE;
    kv_quantize_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(x, (uint8_t*)out, rows, (int)hd);
    return launch_status();
}

qmm_status qmm_kv_scores(const void* q, const void* kc, float* scores, int64_t Hq, int64_t Hkv, int64_t P, int64_t hd,
                         float scale, qmm_stream_t stream) {
    if (!q || !kc || !scores) return QMM_E_NULL;
    if (!kv_hd_ok(hd)) return QMM_E_SHAPE;
    qmm_status st = kv_heads_ok(Hq, Hkv, P);
    if (st != QMM_OK) return st;
    if (!aligned4(q) || !aligned4(kc) || !aligned4(scores)) return QMM_E_ALIGN;
    const int G = (int)(Hq / Hkv);
    const size_t smem = (size_t)(G + kKvTile) * (size_t)(4 + hd);
    const dim3 grid((unsigned)((P + kKvTile - 1) / kKvTile), (unsigned)Hkv);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kv_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return QMM_E_CUDA;
    kv_scores_kernel<<<grid, kKvTile, smem, (cudaStream_t)stream>>>((const uint8_t*)q, (const uint8_t*)kc, scores, G,
                                                                    (int)Hkv, P, (int)hd, scale);
    return launch_status();
}

size_t qmm_kv_wsum_scratch_bytes(int64_t Hq, int64_t P, int64_t hd) {
    if (Hq < 1 || P < 1 || !kv_hd_ok(hd)) return 0;
    return (size_t)Hq * (size_t)((P + kKvChunk - 1) / kKvChunk) * (size_t)hd * sizeof(float);
}

qmm_status qmm_kv_wsum(const float* w, const void* vc, float* out, void* scratch, size_t scratch_bytes, int64_t Hq,
                       int64_t Hkv, int64_t P, int64_t hd, qmm_stream_t stream) {
    if (!w || !vc || !out || !scratch) return QMM_E_NULL;
    if (!kv_hd_ok(hd)) return QMM_E_SHAPE;
    qmm_status st = kv_heads_ok(Hq, Hkv, P);
    if (st != QMM_OK) return st;
    if (!aligned4(w) || !aligned4(vc) || !aligned4(out) || !aligned16(scratch)) return QMM_E_ALIGN;
    if (scratch_bytes < qmm_kv_wsum_scratch_bytes(Hq, P, hd)) return QMM_E_SCRATCH;
    const int G = (int)(Hq / Hkv);
    const int64_t nc = (P + kKvChunk - 1) / kKvChunk;
    if (nc > 0x7FFFFFFFLL) return QMM_E_SHAPE;
    const int threads = (G * (int)(hd / 4) + 31) / 32 * 32;
    cudaStream_t cs = (cudaStream_t)stream;
    kv_wsum_partial_kernel<<<dim3((unsigned)nc, (unsigned)Hkv), threads, 0, cs>>>(w, (const uint8_t*)vc,
                                                                                  (float*)scratch, G, (int)Hkv, P,
                                                                                  (int)hd);
    st = launch_status();
    if (st != QMM_OK) return st;
    const int64_t outs = Hq * hd;
    kv_wsum_reduce_kernel<<<(unsigned)((outs + 255) / 256), 256, 0, cs>>>((const float*)scratch, out, G, (int)Hq,
                                                                          (int)nc, (int)hd);
    return launch_status();
}

}  // extern "C"

// kvcache.cu -- the Q8 KV cache of decode attention ([krafla] "Architecture",
// Attention, "Q8 cache"): each position's K and V are kept per KV head as int8
// codes with one float scale, quantized by the activations' rule; each query
// head is quantized the same way; a score is an integer dot product, and the V
// sum widens the int8 values to float as it goes.
//
// A row is one head vector of hd values: f32 d @0, int8 codes @4 (4 + hd bytes;
// 68 at hd = 64).  The cache holds row (p, kvh) at (p*Hkv + kvh) * (4 + hd), so
// appending a position writes Hkv consecutive rows.  Query head h reads KV head
// h / (Hq/Hkv) ([krafla] "Architecture", "Data flow for one token").
//
//   kv_quantize   one warp per row: amax, d = amax/127, codes rne(x*127/amax)
//   kv_scores     a CTA per (128 positions, KV head): the K rows of the tile and
//                 the group's query rows staged in shared memory, eight lanes per
//                 position computing the group's G integer dots with dp4a and
//                 meeting through shuffles; score = ((dq*dk) * isum) * scale, each
//                 step rounded once
//   kv_wsum       pass 1: a CTA per (128-position chunk, KV head): the chunk's V
//                 rows and the group's weights staged in shared memory; thread
//                 groups each take every groups-th position of the chunk, one
//                 thread per 4 columns converting each V word once and running
//                 an f32 FMA chain for every query head of the group; the groups'
//                 sums are added in group order; pass 2: a warp per output adds
//                 the chunks' partial sums, lane l taking chunks l, l + 32, ... in
//                 order, then a fixed butterfly.  The grouping depends only on
//                 hd, Hq/Hkv and P, so the result does not depend on the GPU.
// The rows of one KV head sit Hkv rows apart and are only 4-byte aligned, so the
// tiles are staged with 4-byte asynchronous copies (cp.async): every copy of a
// tile is in flight at once, then one wait.
#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

constexpr int kKvRows = 128;    // positions per CTA of the score kernel
constexpr int kKvChunk = 128;   // positions per partial sum of the V sum
constexpr int kKvMaxGroup = 8;  // query heads per KV head
constexpr int kKvMaxHd = 256;

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// rows rows of nwd words, row r at src + r * stride_bytes, into dst with a row
// stride of dst_stride words
__device__ __forceinline__ void stage_rows(uint32_t* dst, int dst_stride, const uint8_t* src, int64_t stride_bytes,
                                           int rows, int nwd) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int r = warp; r < rows; r += nwarps) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(src + r * stride_bytes);
        for (int w = lane; w < nwd; w += 32) cp_async4(dst + r * dst_stride + w, s + w);
    }
}

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

// Shared-memory row stride (words) for rows read by 8 lanes each, 4 rows per
// warp: s = 8 (mod 32) puts the four rows' words in distinct bank octets.
__host__ __device__ inline int kv_smem_stride(int nwd) { return nwd <= 8 ? 8 : 8 + (nwd - 8 + 31) / 32 * 32; }

// grid (tiles of kKvRows positions, Hkv); 8 lanes per position, 256 threads.
// Lane j of a position's octet takes code words j, j + 8, ... (at most 8 of
// them, hd <= 256) and holds the group's query words for them in registers; the
// G partial dots meet through three xor shuffles.  GT is G rounded up to 1, 2,
// 4 or 8.
template <int GT>
__global__ void __launch_bounds__(256) kv_scores_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ kc,
                                                        float* __restrict__ scores, int G, int Hkv, int64_t P, int hd,
                                                        float scale) {
    extern __shared__ __align__(16) uint32_t kv_smem[];
    const int nwd = (4 + hd) / 4, st = kv_smem_stride(nwd);
    uint32_t* qs = kv_smem;            // G rows
    uint32_t* ks = kv_smem + G * st;   // kKvRows rows
    const int kvh = blockIdx.y;
    const int64_t p0 = (int64_t)blockIdx.x * kKvRows;
    const int rows = P - p0 < kKvRows ? (int)(P - p0) : kKvRows;
    const int64_t rb = 4 + hd;
    stage_rows(qs, st, q + (int64_t)kvh * G * rb, rb, G, nwd);
    stage_rows(ks, st, kc + (p0 * Hkv + kvh) * rb, Hkv * rb, rows, nwd);
    cp_async_wait_all();
    __syncthreads();
    const int j = threadIdx.x & 7;
    uint32_t qw[GT][8];
#pragma unroll
    for (int g = 0; g < GT; g++)
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const int w = 1 + j + 8 * k;
            qw[g][k] = (g < G && w < nwd) ? qs[g * st + w] : 0u;
        }
    const float dq = j < G ? __uint_as_float(qs[j * st]) : 0.0f;
    // the 32 octets take rows octet, octet + 32, ...
    for (int r = threadIdx.x >> 3; r - (int)(threadIdx.x >> 3) < kKvRows; r += 32) {
        const uint32_t* kr = ks + r * st;
        int acc[GT];
#pragma unroll
        for (int g = 0; g < GT; g++) acc[g] = 0;
        if (r < rows) {
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int w = 1 + j + 8 * k;
                if (w < nwd) {
                    const uint32_t kw = kr[w];
#pragma unroll
                    for (int g = 0; g < GT; g++) acc[g] = dp4a(kw, qw[g][k], acc[g]);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GT; g++) {
            acc[g] += __shfl_xor_sync(0xFFFFFFFFu, acc[g], 1);
            acc[g] += __shfl_xor_sync(0xFFFFFFFFu, acc[g], 2);
            acc[g] += __shfl_xor_sync(0xFFFFFFFFu, acc[g], 4);
        }
        if (r < rows && j < G) {
            int a = acc[0];
#pragma unroll
            for (int g = 1; g < GT; g++)
                if (g == j) a = acc[g];
            const float dk = __uint_as_float(kr[0]);
            scores[(int64_t)(kvh * G + j) * P + p0 + r] = __fmul_rn(__fmul_rn(__fmul_rn(dq, dk), (float)a), scale);
        }
    }
}

// int8 byte k of v as an exact float: the biased byte (v ^ 0x80 per byte,
// 0..255) placed in the low mantissa bits of 2^23, minus 2^23 + 128.
__device__ __forceinline__ float i8_to_f(uint32_t vb, int k) {
    return __fsub_rn(__uint_as_float(__byte_perm(vb, 0x4B000000u, 0x7640u + (uint32_t)k)), 8388736.0f);
}

// pass 1: grid (chunks, Hkv).  One thread per column quad in each of `groups`
// thread groups; group k walks the chunk's positions k, k + groups, ...,
// converting each V word once and running the G heads' f32 FMA chains; then
// the groups' sums are added in group order.  GT as for the scores.
template <int GT>
__global__ void __launch_bounds__(512) kv_wsum_partial_kernel(const float* __restrict__ w, const uint8_t* __restrict__ vc,
                                                              float* __restrict__ part, int G, int Hkv, int64_t P,
                                                              int hd, int groups, int gthreads) {
    extern __shared__ __align__(16) uint32_t kv_smem[];
    const int nq = hd / 4, nwd = nq + 1;
    const int kvh = blockIdx.y;
    const int c = blockIdx.x, nc = gridDim.x;
    const int64_t pa = (int64_t)c * kKvChunk;
    const int n = P - pa < kKvChunk ? (int)(P - pa) : kKvChunk;
    const int64_t rb = 4 + hd;
    uint32_t* vs = kv_smem;                                         // n rows of nwd words
    float* ws = reinterpret_cast<float*>(kv_smem + kKvChunk * nwd);  // G rows of n weights
    float4* red = reinterpret_cast<float4*>(ws + G * kKvChunk);      // groups x G x nq partial sums
    stage_rows(vs, nwd, vc + (pa * Hkv + kvh) * rb, Hkv * rb, n, nwd);
    for (int g = 0; g < G; g++)
        for (int j = threadIdx.x; j < n; j += blockDim.x) cp_async4(ws + g * kKvChunk + j, w + (kvh * G + g) * P + pa + j);
    cp_async_wait_all();
    __syncthreads();
    const int grp = threadIdx.x / gthreads, quad = threadIdx.x - grp * gthreads;
    if (quad < nq) {
        float4 a[GT];
#pragma unroll
        for (int g = 0; g < GT; g++) a[g] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int j = grp; j < n; j += groups) {
            const uint32_t* row = vs + j * nwd;
            const float dv = __uint_as_float(row[0]);
            const uint32_t vb = row[1 + quad] ^ 0x80808080u;
            const float v0 = i8_to_f(vb, 0), v1 = i8_to_f(vb, 1), v2 = i8_to_f(vb, 2), v3 = i8_to_f(vb, 3);
#pragma unroll
            for (int g = 0; g < GT; g++) {
                if (g < G) {
                    const float coef = __fmul_rn(ws[g * kKvChunk + j], dv);
                    a[g].x = __fmaf_rn(coef, v0, a[g].x);
                    a[g].y = __fmaf_rn(coef, v1, a[g].y);
                    a[g].z = __fmaf_rn(coef, v2, a[g].z);
                    a[g].w = __fmaf_rn(coef, v3, a[g].w);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GT; g++)
            if (g < G) red[(grp * G + g) * nq + quad] = a[g];
    }
    __syncthreads();
    for (int t2 = threadIdx.x; t2 < G * nq; t2 += blockDim.x) {
        float4 sum = red[t2];
        for (int k = 1; k < groups; k++) {
            const float4 v = red[k * G * nq + t2];
            sum.x = __fadd_rn(sum.x, v.x);
            sum.y = __fadd_rn(sum.y, v.y);
            sum.z = __fadd_rn(sum.z, v.z);
            sum.w = __fadd_rn(sum.w, v.w);
        }
        const int g = t2 / nq, quad2 = t2 - g * nq;
        *reinterpret_cast<float4*>(part + (((int64_t)kvh * nc + c) * G + g) * hd + 4 * quad2) = sum;
    }
}

// pass 2: one warp per output (h, i).  Lane l adds chunks l, l + 32, ... in
// order, then the 32 lane sums meet in a fixed butterfly: the order depends on
// the chunk count alone.
__global__ void __launch_bounds__(256) kv_wsum_reduce_kernel(const float* __restrict__ part, float* __restrict__ out,
                                                             int G, int Hq, int nc, int hd) {
    const int64_t o = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (o >= (int64_t)Hq * hd) return;  // whole warps leave together
    const int h = (int)(o / hd), i = (int)(o - (int64_t)h * hd);
    const int kvh = h / G, g = h - kvh * G;
    const float* src = part + ((int64_t)kvh * nc * G + g) * hd + i;
    const int64_t step = (int64_t)G * hd;
    float s = 0.0f;
#pragma unroll 4
    for (int c = lane; c < nc; c += 32) s = __fadd_rn(s, src[c * step]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, off));
    if (lane == 0) out[o] = s;
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
    const size_t smem = (size_t)(G + kKvRows) * (size_t)kv_smem_stride((int)(4 + hd) / 4) * 4;
    const dim3 grid((unsigned)((P + kKvRows - 1) / kKvRows), (unsigned)Hkv);
    cudaStream_t cs = (cudaStream_t)stream;
    const uint8_t *qb = (const uint8_t*)q, *kb = (const uint8_t*)kc;
    if (G == 1) kv_scores_kernel<1><<<grid, 256, smem, cs>>>(qb, kb, scores, G, (int)Hkv, P, (int)hd, scale);
    else if (G == 2) kv_scores_kernel<2><<<grid, 256, smem, cs>>>(qb, kb, scores, G, (int)Hkv, P, (int)hd, scale);
    else if (G <= 4) kv_scores_kernel<4><<<grid, 256, smem, cs>>>(qb, kb, scores, G, (int)Hkv, P, (int)hd, scale);
    else kv_scores_kernel<8><<<grid, 256, smem, cs>>>(qb, kb, scores, G, (int)Hkv, P, (int)hd, scale);
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
    const int nq = (int)(hd / 4);
    const int gthreads = (nq + 31) / 32 * 32;
    int groups = 512 / gthreads;
    if (groups > 16) groups = 16;
    // the staged chunk, its weights and the groups' sums within the default 48 KB
    // (one group always fits: at most 33280 + 4096 + 8192 bytes)
    const size_t base = (size_t)kKvChunk * (size_t)(4 + hd) + (size_t)G * kKvChunk * sizeof(float);
    while (groups > 1 && base + (size_t)groups * G * nq * 16 > 48 * 1024) groups--;
    const size_t smem = base + (size_t)groups * G * nq * 16;
    cudaStream_t cs = (cudaStream_t)stream;
    const dim3 grid((unsigned)nc, (unsigned)Hkv);
    const int nt = groups * gthreads;
    const uint8_t* vb = (const uint8_t*)vc;
    float* pt = (float*)scratch;
    if (G == 1) kv_wsum_partial_kernel<1><<<grid, nt, smem, cs>>>(w, vb, pt, G, (int)Hkv, P, (int)hd, groups, gthreads);
    else if (G == 2) kv_wsum_partial_kernel<2><<<grid, nt, smem, cs>>>(w, vb, pt, G, (int)Hkv, P, (int)hd, groups, gthreads);
    else if (G <= 4) kv_wsum_partial_kernel<4><<<grid, nt, smem, cs>>>(w, vb, pt, G, (int)Hkv, P, (int)hd, groups, gthreads);
    else kv_wsum_partial_kernel<8><<<grid, nt, smem, cs>>>(w, vb, pt, G, (int)Hkv, P, (int)hd, groups, gthreads);
    st = launch_status();
    if (st != QMM_OK) return st;
    const int64_t outs = Hq * hd;
    kv_wsum_reduce_kernel<<<(unsigned)((outs * 32 + 255) / 256), 256, 0, cs>>>((const float*)scratch, out, G, (int)Hq,
                                                                               (int)nc, (int)hd);
    return launch_status();
}

}  // extern "C"

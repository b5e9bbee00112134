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
//   kv_scores     a CTA per range of positions, every KV head: one contiguous,
//                 16-byte aligned range of the cache, fetched by one bulk copy;
//                 eight lanes per row computing the group's G integer dots with
//                 dp4a and meeting through a transposing shuffle reduction;
//                 score = ((dq*dk) * isum) * scale, each step rounded once
//   kv_wsum       pass 1: a CTA per 32-position chunk (every KV head, or a group
//                 of them when the rows do not fit), one bulk copy; one thread
//                 per (KV head, 4 columns) converting each V word once and
//                 running the f32 FMA chains of its query heads over the chunk's
//                 positions in order; pass 2: per output, 8 warps each add every
//                 8th chunk's sum in order, then the 8 in warp order.  The order
//                 depends only on P, so the result does not depend on the GPU.
// A ragged last tile, or a cache that is not 16-byte aligned, is staged with
// 4-byte asynchronous copies (cp.async) instead: all in flight, then one wait.
#include <type_traits>

#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

constexpr int kKvChunk = 32;    // positions per partial sum of the V sum
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
    pdl_wait();
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
    pdl_launch_dependents();
}

static __device__ unsigned int g_kv_error = 0;

// Positions per score CTA: a multiple of 4 (so the tile of TP * Hkv rows of
// 4 + hd bytes is a multiple of 16 bytes) with at least 128 rows.
__host__ __device__ inline int kv_score_positions(int Hkv) {
    int tp = (128 + Hkv - 1) / Hkv;
    tp = (tp + 3) / 4 * 4;
    return tp < 4 ? 4 : tp;
}

// grid: tiles of TP positions, every KV head of them -- one contiguous range of
// the cache, fetched by one bulk copy (or, for a ragged last tile or an
// unaligned cache, by 4-byte asynchronous copies).  256 threads = 32 octets;
// octet o takes the tile's rows o, o + 32, ...; lane j of an octet takes a
// contiguous run of the row's code words and holds the matching query words of
// the row's KV-head group in registers (reloaded when the octet's KV head
// changes, never when Hkv divides 32).  The G partial dots meet through three xor
// shuffles.  GT is G rounded up to 1, 2, 4 or 8; WT the code words per lane,
// ceil(hd/32) rounded up to 1, 2, 4 or 8.
template <int GT, int WT>
__global__ void __launch_bounds__(256) kv_scores_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ kc,
                                                        float* __restrict__ scores, int G, int Hkv, int64_t P, int hd,
                                                        float scale, int TP, int bulk) {
    extern __shared__ __align__(16) uint8_t kv_tile[];
    pdl_wait();
    uint64_t* bar = reinterpret_cast<uint64_t*>(kv_tile);
    uint32_t* ks = reinterpret_cast<uint32_t*>(kv_tile + 16);
    const int nwd = (4 + hd) / 4, nq = hd / 4, wpl = (nq + 7) / 8;
    const int64_t rb = 4 + hd;
    const int64_t p0 = (int64_t)blockIdx.x * TP;
    const int np = P - p0 < TP ? (int)(P - p0) : TP;
    const int R = np * Hkv;
    const uint8_t* src = kc + p0 * Hkv * rb;
    const bool use_bulk = bulk && np == TP;
    if (use_bulk) {
        if (threadIdx.x == 0) {
            mbar_init(smem_u32(bar), 1);
            fence_mbar_init();
            uint32_t bytes = (uint32_t)(R * rb);
            if (!QMM_IN_BOUNDS(g_kv_error, 16 + (int64_t)bytes - 1, dynamic_smem_bytes()) ||
                !QMM_IN_BOUNDS(g_kv_error, (p0 * Hkv * rb) + bytes - 1, P * Hkv * rb))
                bytes = 0;  // the tile must fit the shared buffer and lie inside the cache
            mbar_arrive_expect_tx(smem_u32(bar), bytes);
            if (bytes) bulk_g2s(smem_u32(ks), src, bytes, smem_u32(bar), policy_evict_first());
        }
        __syncthreads();
        const bool ok = mbar_wait_bounded(smem_u32(bar), 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) {  // every thread leaves together, so no shuffle misses a lane
            if (threadIdx.x == 0) atomicOr(&g_kv_error, kErrTimeout);
            return;
        }
    } else {
        const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src);
        for (int i = threadIdx.x; i < R * nwd; i += blockDim.x)
            if (QMM_IN_BOUNDS(g_kv_error, p0 * Hkv * rb + 4 * (int64_t)i + 3, P * Hkv * rb) &&
                QMM_IN_BOUNDS(g_kv_error, 16 + 4 * (int64_t)i + 3, dynamic_smem_bytes()))
                cp_async4(ks + i, s4 + i);
        cp_async_wait_all();
        __syncthreads();
    }
    const int j = threadIdx.x & 7, oct = threadIdx.x >> 3;
    const int w0 = 1 + j * wpl;  // this lane's first code word
    // after the octet's transposing reduction lane j holds the dot of head gl
    // of the group (bit k of j picks the upper half at round k)
    int gl = 0;
#pragma unroll
    for (int m = 1, n = GT; n > 1; m <<= 1, n >>= 1)
        if (j & m) gl += n >> 1;
    uint32_t qw[GT][WT];
    int cur = -1;
    float dq = 0.0f;
    // row r = oct + 32 it: position pl, KV head kvh, stepped without a division per row
    const int dpl = 32 / Hkv, dkv = 32 - dpl * Hkv;
    int pl = oct / Hkv, kvh = oct - pl * Hkv;
    const int iters = (R + 31) / 32;  // the same count for every octet: the shuffles need whole warps
    for (int it = 0; it < iters; it++, pl += dpl, kvh += dkv) {
        if (kvh >= Hkv) kvh -= Hkv, pl += 1;
        const int r = oct + 32 * it;
        const bool live = r < R;
        if (live && kvh != cur) {  // uniform per octet: its rows' KV head
            const uint32_t* qg = reinterpret_cast<const uint32_t*>(q + (int64_t)kvh * G * rb);
#pragma unroll
            for (int g = 0; g < GT; g++)
#pragma unroll
                for (int k = 0; k < WT; k++)
                    qw[g][k] = (g < G && k < wpl && w0 + k < nwd) ? __ldg(qg + g * nwd + w0 + k) : 0u;
            dq = gl < G ? __uint_as_float(__ldg(qg + gl * nwd)) : 0.0f;
            cur = kvh;
        }
        const uint32_t* kr = ks + r * nwd;
        int acc[GT];
#pragma unroll
        for (int g = 0; g < GT; g++) acc[g] = 0;
        if (live) {
#pragma unroll
            for (int k = 0; k < WT; k++) {
                if (k < wpl && w0 + k < nwd) {
                    const uint32_t kw = kr[w0 + k];
#pragma unroll
                    for (int g = 0; g < GT; g++) acc[g] = dp4a(kw, qw[g][k], acc[g]);
                }
            }
        }
        // transposing reduction: at each round a lane keeps half of its sums and
        // trades the other half with its partner, so GT - 1 shuffles leave one
        // sum per lane; the remaining rounds add single values
        int m = 1;
#pragma unroll
        for (int n = GT; n > 1; n >>= 1, m <<= 1) {
            const bool hi = (j & m) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; i++) {
                const int send = hi ? acc[i] : acc[i + n / 2];
                const int keep = hi ? acc[i + n / 2] : acc[i];
                acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
            }
        }
        for (; m < 8; m <<= 1) acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], m);
        if (live && j < GT && gl < G) {
            const float dk = __uint_as_float(kr[0]);
            if (QMM_IN_BOUNDS(g_kv_error, (int64_t)(kvh * G + gl) * P + p0 + pl, (int64_t)Hkv * G * P))
                scores[(int64_t)(kvh * G + gl) * P + p0 + pl] =
                    __fmul_rn(__fmul_rn(__fmul_rn(dq, dk), (float)acc[0]), scale);
        }
    }
    // the next kernel may launch once every CTA is here (or has left): launched
    // earlier, its waiting CTAs would take the slots this grid's later waves need
    pdl_launch_dependents();
}

// int8 byte k of v as an exact float: the biased byte (v ^ 0x80 per byte,
// 0..255) placed in the low mantissa bits of 2^23, minus 2^23 + 128.
__device__ __forceinline__ float i8_to_f(uint32_t vb, int k) {
    return __fsub_rn(__uint_as_float(__byte_perm(vb, 0x4B000000u, 0x7640u + (uint32_t)k)), 8388736.0f);
}

// pass 1: grid (chunks of kKvChunk positions, groups of hg KV heads).  The
// chunk's rows of those heads are staged in shared memory (one bulk copy when
// the group is every head and the range is aligned, else 4-byte asynchronous
// copies of each position's run of hg rows), with the weights of their query
// heads.  One thread per (KV head, column quad) walks the chunk's positions in
// order, converting each V word once and running the f32 FMA chains of the
// group's GT (>= G) query heads.  Partial sums: part[(c * Hq + h) * hd + i].
template <int GT>
__global__ void __launch_bounds__(512) kv_wsum_partial_kernel(const float* __restrict__ w, const uint8_t* __restrict__ vc,
                                                              float* __restrict__ part, int G, int Hkv, int64_t P,
                                                              int hd, int hg, int bulk) {
    extern __shared__ __align__(16) uint8_t kv_tile[];
    pdl_wait();
    uint64_t* bar = reinterpret_cast<uint64_t*>(kv_tile);
    const int nq = hd / 4, nwd = nq + 1;
    const int64_t rb = 4 + hd;
    const int c = blockIdx.x, kv0 = blockIdx.y * hg;
    const int hn = Hkv - kv0 < hg ? Hkv - kv0 : hg;  // KV heads in this group
    const int64_t pa = (int64_t)c * kKvChunk;
    const int n = P - pa < kKvChunk ? (int)(P - pa) : kKvChunk;
    const int Hq = Hkv * G;
    uint32_t* vs = reinterpret_cast<uint32_t*>(kv_tile + 16);                 // n positions x hn rows
    float* ws = reinterpret_cast<float*>(vs + (size_t)kKvChunk * hg * nwd);    // hn*G heads x kKvChunk weights
    const uint8_t* src = vc + (pa * Hkv + kv0) * rb;
    const bool use_bulk = bulk && hn == Hkv && n == kKvChunk;
    if (use_bulk && threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
        uint32_t bytes = (uint32_t)((int64_t)n * Hkv * rb);
        if (!QMM_IN_BOUNDS(g_kv_error, (pa * Hkv + kv0) * rb + bytes - 1, P * Hkv * rb)) bytes = 0;
        mbar_arrive_expect_tx(smem_u32(bar), bytes);
        if (bytes) bulk_g2s(smem_u32(vs), src, bytes, smem_u32(bar), policy_evict_first());
    }
    if (!use_bulk) {  // position p's hn rows are one run of hn * nwd words
        const int run = hn * nwd;
        for (int i = threadIdx.x; i < n * run; i += blockDim.x) {
            const int pp = i / run, k = i - pp * run;
            if (QMM_IN_BOUNDS(g_kv_error, (pa * Hkv + kv0) * rb + (int64_t)pp * Hkv * rb + 4 * k + 3, P * Hkv * rb))
                cp_async4(vs + (size_t)pp * run + k,
                          reinterpret_cast<const uint32_t*>(src + (int64_t)pp * Hkv * rb) + k);
        }
    }
    for (int i = threadIdx.x; i < hn * G * n; i += blockDim.x) {
        const int hh = i / n, j = i - hh * n;
        if (QMM_IN_BOUNDS(g_kv_error, (int64_t)(kv0 * G + hh) * P + pa + j, (int64_t)Hq * P))
            cp_async4(ws + hh * kKvChunk + j, w + (int64_t)(kv0 * G + hh) * P + pa + j);
    }
    cp_async_wait_all();
    __syncthreads();
    if (use_bulk) {
        const bool ok = mbar_wait_bounded(smem_u32(bar), 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) atomicOr(&g_kv_error, kErrTimeout);
            return;
        }
    }
    const int run = hn * nwd;
    for (int t = threadIdx.x; t < hn * nq; t += blockDim.x) {
        const int kh = t / nq, quad = t - kh * nq;
        float4 a[GT];
#pragma unroll
        for (int g = 0; g < GT; g++) a[g] = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t* col = vs + kh * nwd;
        const float* wk = ws + kh * G * kKvChunk;
#pragma unroll 2
        for (int j = 0; j < n; j++) {
            const uint32_t* row = col + j * run;
            const float dv = __uint_as_float(row[0]);
            const uint32_t vb = row[1 + quad] ^ 0x80808080u;
            const float v0 = i8_to_f(vb, 0), v1 = i8_to_f(vb, 1), v2 = i8_to_f(vb, 2), v3 = i8_to_f(vb, 3);
#pragma unroll
            for (int g = 0; g < GT; g++) {
                if (g < G) {
                    const float coef = __fmul_rn(wk[g * kKvChunk + j], dv);
                    a[g].x = __fmaf_rn(coef, v0, a[g].x);
                    a[g].y = __fmaf_rn(coef, v1, a[g].y);
                    a[g].z = __fmaf_rn(coef, v2, a[g].z);
                    a[g].w = __fmaf_rn(coef, v3, a[g].w);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GT; g++) {
            if (g < G) {
                const int h = (kv0 + kh) * G + g;
                *reinterpret_cast<float4*>(part + ((int64_t)c * Hq + h) * hd + 4 * quad) = a[g];
            }
        }
    }
    pdl_launch_dependents();
}

// pass 2: a CTA of 8 warps per 32 consecutive outputs (lane = output, so every
// load is one coalesced 128-byte row of a chunk's sums).  Warp k adds chunks k,
// k + 8, ... in order; then the 8 warp sums are added in warp order.  The order
// depends on the chunk count alone.
__global__ void __launch_bounds__(256) kv_wsum_reduce_kernel(const float* __restrict__ part, float* __restrict__ out,
                                                             int Hq, int nc, int hd) {
    __shared__ float red[8][32];
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t outs = (int64_t)Hq * hd;
    const int64_t o = (int64_t)blockIdx.x * 32 + lane;
    float s = 0.0f;
    if (o < outs) {
#pragma unroll 8
        for (int c = warp; c < nc; c += 8)
            if (QMM_IN_BOUNDS(g_kv_error, (int64_t)c * outs + o, (int64_t)nc * outs))
                s = __fadd_rn(s, part[(int64_t)c * outs + o]);
    }
    red[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && o < outs) {
        float t = red[0][lane];
#pragma unroll
        for (int k = 1; k < 8; k++) t = __fadd_rn(t, red[k][lane]);
        out[o] = t;
    }
    pdl_launch_dependents();
}

static bool kv_hd_ok(int64_t hd) { return hd >= 16 && hd <= kKvMaxHd && hd % 16 == 0; }

static qmm_status kv_heads_ok(int64_t Hq, int64_t Hkv, int64_t P) {
    if (Hq < 1 || Hkv < 1 || P < 1 || Hq % Hkv || Hq / Hkv > kKvMaxGroup || Hkv > 128) return QMM_E_SHAPE;
    if (P > 0x7FFFFFFFLL || P * Hq > ((int64_t)1 << 40)) return QMM_E_SHAPE;
    return QMM_OK;
}

static bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

// A programmatic dependent launch: the kernel waits for its predecessor's
// memory before it reads anything, and lets its successor launch when its own
// work is done.
template <typename... KArgs, typename... Args>
static qmm_status launch_pdl(void (*kern)(KArgs...), dim3 grid, int block, size_t smem, cudaStream_t stream,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess ? QMM_OK : QMM_E_CUDA;
}

}  // namespace qmm

using namespace qmm;

extern "C" {

size_t qmm_kv_row_bytes(int64_t hd) { return kv_hd_ok(hd) ? (size_t)(4 + hd) : 0; }

unsigned qmm_internal_kv_error(int clear) {
    unsigned v = 0;
    cudaMemcpyFromSymbol(&v, g_kv_error, sizeof(v));
    if (clear) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_kv_error, &z, sizeof(z));
    }
    return v;
}

qmm_status qmm_kv_quantize(const float* x, void* out, int64_t rows, int64_t hd, qmm_stream_t stream) {
    if (!x || !out) return QMM_E_NULL;
    if (rows < 1 || !kv_hd_ok(hd) || rows > ((int64_t)1 << 36)) return QMM_E_SHAPE;
    if (!aligned4(x) || !aligned4(out)) return QMM_E_ALIGN;
    const int64_t grid = (rows * 32 + 255) / 256;
    if (grid > 0x7FFFFFFFLL) return QMM_E_SHAPE;
    return launch_pdl(kv_quantize_kernel, dim3((unsigned)grid), 256, 0, (cudaStream_t)stream, x, (uint8_t*)out, rows,
                      (int)hd);
}

qmm_status qmm_kv_scores(const void* q, const void* kc, float* scores, int64_t Hq, int64_t Hkv, int64_t P, int64_t hd,
                         float scale, qmm_stream_t stream) {
    if (!q || !kc || !scores) return QMM_E_NULL;
    if (!kv_hd_ok(hd)) return QMM_E_SHAPE;
    qmm_status st = kv_heads_ok(Hq, Hkv, P);
    if (st != QMM_OK) return st;
    if (!aligned4(q) || !aligned4(kc) || !aligned4(scores)) return QMM_E_ALIGN;
    const int G = (int)(Hq / Hkv);
    const int TP = kv_score_positions((int)Hkv);
    const size_t smem = 16 + (size_t)TP * (size_t)Hkv * (size_t)(4 + hd);
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QMM_OK) return st;
    if (smem > (size_t)dev.max_smem_optin) return QMM_E_SHAPE;
    const int bulk = aligned16(kc) ? 1 : 0;
    const dim3 grid((unsigned)((P + TP - 1) / TP));
    cudaStream_t cs = (cudaStream_t)stream;
    const uint8_t *qb = (const uint8_t*)q, *kb = (const uint8_t*)kc;
    auto go = [&](auto kern) -> qmm_status {
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QMM_E_CUDA;
        return launch_pdl(kern, grid, 256, smem, cs, qb, kb, scores, G, (int)Hkv, P, (int)hd, scale, TP, bulk);
    };
    const int wpl = ((int)hd / 4 + 7) / 8;
    auto by_w = [&](auto g_tag) -> qmm_status {
        constexpr int GT = decltype(g_tag)::value;
        if (wpl <= 1) return go(kv_scores_kernel<GT, 1>);
        if (wpl <= 2) return go(kv_scores_kernel<GT, 2>);
        if (wpl <= 4) return go(kv_scores_kernel<GT, 4>);
        return go(kv_scores_kernel<GT, 8>);
    };
    if (G == 1) return by_w(std::integral_constant<int, 1>());
    if (G == 2) return by_w(std::integral_constant<int, 2>());
    if (G <= 4) return by_w(std::integral_constant<int, 4>());
    return by_w(std::integral_constant<int, 8>());
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
    const int nq = (int)(hd / 4), nwd = nq + 1;
    // KV heads per CTA: all of them when the chunk's rows and weights fit in
    // about 100 KB of shared memory (then one bulk copy fetches the rows)
    const size_t per_head = (size_t)kKvChunk * nwd * 4 + (size_t)G * kKvChunk * 4;
    int hg = (int)((100 * 1024 - 16) / per_head);
    if (hg > Hkv) hg = (int)Hkv;
    if (hg < 1) hg = 1;
    const size_t smem = 16 + (size_t)hg * per_head;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QMM_OK) return st;
    if (smem > (size_t)dev.max_smem_optin) return QMM_E_SHAPE;
    const int bulk = (aligned16(vc) && hg == Hkv) ? 1 : 0;
    int nt = (hg * nq + 31) / 32 * 32;
    if (nt > 512) nt = 512;
    cudaStream_t cs = (cudaStream_t)stream;
    const dim3 grid((unsigned)nc, (unsigned)((Hkv + hg - 1) / hg));
    const uint8_t* vb = (const uint8_t*)vc;
    float* pt = (float*)scratch;
    auto go = [&](auto kern) -> qmm_status {
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QMM_E_CUDA;
        return launch_pdl(kern, grid, nt, smem, cs, w, vb, pt, G, (int)Hkv, P, (int)hd, hg, bulk);
    };
    if (G == 1) st = go(kv_wsum_partial_kernel<1>);
    else if (G == 2) st = go(kv_wsum_partial_kernel<2>);
    else if (G <= 4) st = go(kv_wsum_partial_kernel<4>);
    else st = go(kv_wsum_partial_kernel<8>);
    if (st != QMM_OK) return st;
    const int64_t outs = Hq * hd;
    return launch_pdl(kv_wsum_reduce_kernel, dim3((unsigned)((outs + 31) / 32)), 256, 0, cs, (const float*)scratch, out,
                      (int)Hq, (int)nc, (int)hd);
}

}  // extern "C"

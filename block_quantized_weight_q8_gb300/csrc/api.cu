// api.cu -- format queries, status strings, the quantize+matmul entry points
// with the activation pairing fixed by the weight type, and the device status
// word read-back.
#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {
qmm_status quantize_act_launch(int act, const float* x, void* xq, int64_t M, int64_t K, cudaStream_t stream, bool pdl);
qmm_status matvec_dispatch(int wt, const void* W, const void* xq, float* y, int64_t N, int64_t K, cudaStream_t stream,
                           bool pdl);
qmm_status matvec_fused_dispatch(int wt, const void* W, const float* x, void* xq_out, float* y, int64_t N, int64_t K,
                                 cudaStream_t stream, bool pdl);
qmm_status matvec_group_fused_dispatch(int wt, int G, const void* const* W, const int64_t* N, float* const* y,
                                       const float* x, void* xq_out, int64_t K, cudaStream_t stream, bool pdl);
qmm_status matvec_group_dispatch(int wt, int G, const void* const* W, const int64_t* N, float* const* y,
                                 const void* xq, int64_t K, cudaStream_t stream, bool pdl);
bool prefill_on_tensor_cores(int wt, int64_t M, int64_t K);
qmm_status prefill_launch(int wt, const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                          cudaStream_t stream, bool pdl);
qmm_status rmsnorm_quantize_launch(int act, const float* x, const float* w, float eps, void* xq, int64_t M, int64_t K,
                                   cudaStream_t stream, bool pdl);
qmm_status matvec_group_norm_dispatch(int wt, int G, const void* const* W, const int64_t* N, float* const* y,
                                      const float* x, const float* gamma, float eps, void* xq_out, int64_t K,
                                      cudaStream_t stream, bool pdl);

// [minfer] "10 . CPU matmul: quantized weights x Q8_0 activations" s3.2
// (cpu_quant_matmul_f32): the weight type alone decides the activation format;
// quantize once into the caller's scratch, then multiply.
qmm_status linear_impl(int wt, const void* W, const float* x, void* scratch, size_t scratch_bytes, float* y,
                       int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    if (!W || !x || !scratch || !y) return QMM_E_NULL;
    qmm_status st = check_shape(wt, M, N, K);
    if (st != QMM_OK) return st;
    if (!aligned16(W) || !aligned16(x) || !aligned16(scratch) || !aligned16(y)) return QMM_E_ALIGN;
    const int act = act_type_of(wt);
    const size_t xrb = row_bytes_of(act, K);
    if (scratch_bytes < (size_t)M * xrb) return QMM_E_SCRATCH;
    if (prefill_on_tensor_cores(wt, M, K)) {  // quantize all rows once, then the tensor-core prefill
        st = quantize_act_launch(act, x, scratch, M, K, stream, true);
        if (st != QMM_OK) return st;
        return prefill_launch(wt, W, scratch, y, M, N, K, stream, true);
    }
    // one launch per token that quantizes its row and multiplies; a row too
    // large for that kernel's shared memory is quantized by its own kernel first
    st = matvec_fused_dispatch(wt, W, x, scratch, y, N, K, stream, true);
    if (st == QMM_OK) {
        for (int64_t t = 1; t < M; t++) {
            st = matvec_fused_dispatch(wt, W, x + t * K, (uint8_t*)scratch + t * xrb, y + t * N, N, K, stream, true);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    if (st != QMM_E_SHAPE) return st;
    st = quantize_act_launch(act, x, scratch, M, K, stream, true);
    if (st != QMM_OK) return st;
    for (int64_t t = 0; t < M; t++) {
        st = matvec_dispatch(wt, W, (const uint8_t*)scratch + t * xrb, y + t * N, N, K, stream, true);
        if (st != QMM_OK) return st;
    }
    return QMM_OK;
}

// G matrices on the same token rows: one launch per token, each CTA quantizing
// the row it needs; the separate quantizer first when the row does not fit.
static qmm_status linear_group(int wt, int G, const void* const* W, const int64_t* N, const float* x, void* scratch,
                               size_t scratch_bytes, float* const* y, int64_t M, int64_t K, cudaStream_t stream) {
    const int act = act_type_of(wt);
    if (act < 0) return QMM_E_TYPE;
    if (G < 1 || G > 8) return QMM_E_SHAPE;
    if (!W || !N || !x || !scratch || !y) return QMM_E_NULL;
    for (int g = 0; g < G; g++) {
        if (!W[g] || !y[g]) return QMM_E_NULL;
        const qmm_status st = check_shape(wt, M, N[g], K);
        if (st != QMM_OK) return st;
        if (!aligned16(W[g]) || !aligned16(y[g])) return QMM_E_ALIGN;
    }
    if (!aligned16(x) || !aligned16(scratch)) return QMM_E_ALIGN;
    const size_t xrb = row_bytes_of(act, K);
    if (scratch_bytes < (size_t)M * xrb) return QMM_E_SCRATCH;
    if (prefill_on_tensor_cores(wt, M, K)) {  // all rows quantized once, then one prefill per matrix
        qmm_status st = quantize_act_launch(act, x, scratch, M, K, stream, true);
        if (st != QMM_OK) return st;
        for (int g = 0; g < G; g++) {
            st = prefill_launch(wt, W[g], scratch, y[g], M, N[g], K, stream, true);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    float* yt[8];
    bool fused = true;
    for (int64_t t = 0; t < M; t++) {
        for (int g = 0; g < G; g++) yt[g] = y[g] + t * N[g];
        qmm_status st = QMM_E_SHAPE;
        if (fused)
            st = matvec_group_fused_dispatch(wt, G, W, N, yt, x + t * K, (uint8_t*)scratch + t * xrb, K, stream, true);
        if (st == QMM_E_SHAPE && t == 0) {
            fused = false;
            st = quantize_act_launch(act, x, scratch, M, K, stream, true);
            if (st != QMM_OK) return st;
        }
        if (!fused) st = matvec_group_dispatch(wt, G, W, N, yt, (const uint8_t*)scratch + t * xrb, K, stream, true);
        if (st != QMM_OK) return st;
    }
    return QMM_OK;
}

// [krafla] "Architecture", "Data flow for one token": h = rmsnorm(x) ; qa =
// quantize_q8(h) ; then the matvecs that read qa.  A token is one launch (each
// CTA norms and quantizes the row itself); a prefill that takes the tensor-core
// matmul norms and quantizes all rows first; a row too large for the fused
// kernel's shared memory is normed and quantized by its own kernel.
static qmm_status linear_norm(int wt, int G, const void* const* W, const int64_t* N, const float* x, const float* w,
                              float eps, void* scratch, size_t scratch_bytes, float* const* y, int64_t M, int64_t K,
                              cudaStream_t stream) {
    const int act = act_type_of(wt);
    if (act < 0) return QMM_E_TYPE;
    if (G < 1 || G > 8) return QMM_E_SHAPE;
    if (!W || !N || !x || !w || !scratch || !y) return QMM_E_NULL;
    for (int g = 0; g < G; g++) {
        if (!W[g] || !y[g]) return QMM_E_NULL;
        const qmm_status st = check_shape(wt, M, N[g], K);
        if (st != QMM_OK) return st;
        if (!aligned16(W[g]) || !aligned16(y[g])) return QMM_E_ALIGN;
    }
    if (!aligned16(x) || !aligned16(w) || !aligned16(scratch)) return QMM_E_ALIGN;
    const size_t xrb = row_bytes_of(act, K);
    if (scratch_bytes < (size_t)M * xrb) return QMM_E_SCRATCH;
    qmm_status st;
    if (prefill_on_tensor_cores(wt, M, K)) {
        st = rmsnorm_quantize_launch(act, x, w, eps, scratch, M, K, stream, true);
        if (st != QMM_OK) return st;
        for (int g = 0; g < G; g++) {
            st = prefill_launch(wt, W[g], scratch, y[g], M, N[g], K, stream, true);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    float* yt[8];
    bool fused = true;
    for (int64_t t = 0; t < M; t++) {
        for (int g = 0; g < G; g++) yt[g] = y[g] + t * N[g];
        st = QMM_E_SHAPE;
        if (fused)
            st = matvec_group_norm_dispatch(wt, G, W, N, yt, x + t * K, w, eps, (uint8_t*)scratch + t * xrb, K,
                                            stream, true);
        if (st == QMM_E_SHAPE && t == 0) {
            fused = false;
            st = rmsnorm_quantize_launch(act, x, w, eps, scratch, M, K, stream, true);
            if (st != QMM_OK) return st;
        }
        if (!fused) st = matvec_group_dispatch(wt, G, W, N, yt, (const uint8_t*)scratch + t * xrb, K, stream, true);
        if (st != QMM_OK) return st;
    }
    return QMM_OK;
}

// The device address of a pinned (page-locked, mapped) host buffer, or null for
// pageable, managed or device memory.
static const void* mapped_host(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the error this query may leave behind
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

static __device__ unsigned int g_test_error = 0;

// The failure-path test: one thread waits on an mbarrier that nothing arrives
// at, with the library's bounded wait, and records the timeout.
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns)) atomicOr(&g_test_error, kErrTimeout);
    }
}

// Outputs (M * N f32 values) up to which qmm_linear_host writes y straight into
// the caller's pinned host buffer: 256 KB.
constexpr int64_t kDirectHostOutputs = 65536;

}  // namespace qmm

using namespace qmm;

extern "C" {
unsigned qmm_internal_matvec_error(int clear);
unsigned qmm_internal_matmul_kq_error(int clear);
unsigned qmm_internal_getrows_error(int clear);
unsigned qmm_internal_kv_error(int clear);
unsigned qmm_internal_quantize_error(int clear);

qmm_status qmm_linear_group(int wtype, int G, const void* const* W, const int64_t* N, const float* x, void* xq_scratch,
                            size_t scratch_bytes, float* const* y, int64_t M, int64_t K, qmm_stream_t stream) {
    return linear_group(wtype, G, W, N, x, xq_scratch, scratch_bytes, y, M, K, (cudaStream_t)stream);
}
unsigned qmm_internal_matmul_error(int clear);

// qmm_linear_<wtype> with host buffers: x from the caller's (pinned) host
// memory in, y back out, all queued on one stream.
qmm_status qmm_linear_host(int wtype, const void* W, const float* x_host, float* x_dev, void* xq_scratch,
                           size_t scratch_bytes, float* y_dev, float* y_host, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    if (!x_host || !y_host) return QMM_E_NULL;
    qmm_status st = check_shape(wtype, M, N, K);
    if (st != QMM_OK) return st;
    const int act = act_type_of(wtype);
    if (act < 0) return QMM_E_TYPE;
    cudaStream_t cs = (cudaStream_t)stream;
    // Pinned host buffers are mapped into the device's address space: for a small
    // output the quantizer reads x over the host link and the multiply writes y
    // there, with no copy-engine transfer (each of which costs several
    // microseconds of latency on the stream for a few kilobytes).
    const float* xm = static_cast<const float*>(mapped_host(x_host));
    float* ym = static_cast<float*>(const_cast<void*>(mapped_host(y_host)));
    if (xm && ym && M * N <= kDirectHostOutputs && aligned16(xm) && aligned16(ym)) {
        if (!W || !xq_scratch) return QMM_E_NULL;
        if (!aligned16(W) || !aligned16(xq_scratch)) return QMM_E_ALIGN;
        const size_t xrb = row_bytes_of(act, K);
        if (scratch_bytes < (size_t)M * xrb) return QMM_E_SCRATCH;
        st = quantize_act_launch(act, xm, xq_scratch, M, K, cs, true);
        if (st != QMM_OK) return st;
        if (prefill_on_tensor_cores(wtype, M, K)) return prefill_launch(wtype, W, xq_scratch, ym, M, N, K, cs, true);
        for (int64_t t = 0; t < M; t++) {
            st = matvec_dispatch(wtype, W, (const uint8_t*)xq_scratch + t * xrb, ym + t * N, N, K, cs, true);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    if (!x_dev || !y_dev) return QMM_E_NULL;
    if (cudaMemcpyAsync(x_dev, x_host, (size_t)M * (size_t)K * sizeof(float), cudaMemcpyHostToDevice, cs) !=
        cudaSuccess)
        return QMM_E_CUDA;
    st = linear_impl(wtype, W, x_dev, xq_scratch, scratch_bytes, y_dev, M, N, K, cs);
    if (st != QMM_OK) return st;
    if (cudaMemcpyAsync(y_host, y_dev, (size_t)M * (size_t)N * sizeof(float), cudaMemcpyDeviceToHost, cs) !=
        cudaSuccess)
        return QMM_E_CUDA;
    return QMM_OK;
}

qmm_status qmm_linear_norm(int wtype, int G, const void* const* W, const int64_t* N, const float* x, const float* w,
                           float eps, void* xq_scratch, size_t scratch_bytes, float* const* y, int64_t M, int64_t K,
                           qmm_stream_t stream) {
    return linear_norm(wtype, G, W, N, x, w, eps, xq_scratch, scratch_bytes, y, M, K, (cudaStream_t)stream);
}

size_t qmm_block_bytes(int type) { return block_bytes_of(type); }
int qmm_block_values(int type) { return block_values_of(type); }
size_t qmm_row_bytes(int type, int64_t K) { return row_bytes_of(type, K); }
int qmm_act_type(int wtype) { return act_type_of(wtype); }

const char* qmm_status_str(qmm_status s) {
    switch (s) {
    case QMM_OK: return "ok";
    case QMM_E_NULL: return "a required pointer is NULL";
    case QMM_E_SHAPE: return "M, N or K out of range, or K not a multiple of the block size";
    case QMM_E_TYPE: return "unknown block type";
    case QMM_E_ALIGN: return "a base pointer is not 16-byte aligned";
    case QMM_E_SCRATCH: return "the scratch buffer is too small";
    case QMM_E_CUDA: return "a CUDA runtime call or kernel launch failed";
    case QMM_E_TIMEOUT: return "a bounded device wait ran out";
    case QMM_E_BOUNDS: return "a kernel index fell outside its buffer (bounds-checked build)";
    default: return "unknown status";
    }
}

qmm_status qmm_linear_q4_0(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q4_0, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}
qmm_status qmm_linear_q8_0(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q8_0, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}
qmm_status qmm_linear_q4_K(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q4_K, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}
qmm_status qmm_linear_q6_K(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q6_K, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}
qmm_status qmm_linear_q2_K(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q2_K, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}

qmm_status qmm_linear_q4_1(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q4_1, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}
qmm_status qmm_linear_q5_0(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q5_0, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}
qmm_status qmm_linear_q5_1(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q5_1, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}
qmm_status qmm_linear_q5_K(const void* W, const float* x, void* s, size_t sb, float* y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    return linear_impl(QMM_Q5_K, W, x, s, sb, y, M, N, K, (cudaStream_t)stream);
}

qmm_status qmm_test_wait_timeout(uint64_t limit_ns, qmm_stream_t stream) {
    const uint64_t lim = limit_ns < 1000ull ? 1000ull : (limit_ns > 100000000ull ? 100000000ull : limit_ns);
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(lim);
    return launch_status();
}

qmm_status qmm_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return QMM_E_CUDA;
    unsigned e = qmm_internal_matvec_error(clear) | qmm_internal_matmul_error(clear) |
                 qmm_internal_matmul_kq_error(clear) | qmm_internal_getrows_error(clear) |
                 qmm_internal_kv_error(clear) | qmm_internal_quantize_error(clear);
    {
        unsigned v = 0;
        if (cudaMemcpyFromSymbol(&v, g_test_error, sizeof(v)) != cudaSuccess) return QMM_E_CUDA;
        e |= v;
        const unsigned z = 0;
        if (clear && cudaMemcpyToSymbol(g_test_error, &z, sizeof(z)) != cudaSuccess) return QMM_E_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return QMM_E_CUDA;
    if (e & kErrTimeout) return QMM_E_TIMEOUT;  // a device wait ran out of time
    if (e & kErrBounds) return QMM_E_BOUNDS;    // an index check of a bounds-checked build failed
    if (e & 2u) return QMM_E_SHAPE;             // qmm_get_rows met an index outside [0, N)
    return QMM_OK;
}

}  // extern "C"

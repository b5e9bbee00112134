// linear_noalloc.cu -- quantize + multiply for callers that cannot hand the
// library a workspace.
//
// qmm_linear_<type> needs a caller-provided device buffer for the quantized
// activation rows.  Some callers cannot provide one: code that runs where device
// allocation is not allowed or not possible (a plugin living inside a host
// application that owns all device memory and passes in only the input and
// output buffers; a latency-critical loop that must never call cudaMalloc,
// which can block on the device and can fail at run time; a caller with a fixed
// memory budget decided before this library is loaded).  For them the
// activation scratch lives here, in one fixed-size array in device global
// memory that every GPU which loads the library holds until the process exits.
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

qmm_status quantize_act_launch(int act, const float* x, void* xq, int64_t M, int64_t K, cudaStream_t stream, bool pdl);
qmm_status matvec_dispatch(int wt, const void* W, const void* xq, float* y, int64_t N, int64_t K, cudaStream_t stream,
                           bool pdl);
qmm_status matvec_fused_dispatch(int wt, const void* W, const float* x, void* xq_out, float* y, int64_t N, int64_t K,
                                 cudaStream_t stream, bool pdl);
bool prefill_on_tensor_cores(int wt, int64_t M, int64_t K);
qmm_status prefill_launch(int wt, const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                          cudaStream_t stream, bool pdl);

// 1 MiB: room for 240 Q8_0 rows or 224 Q8_K rows at K = 4096.
constexpr size_t kNoAllocScratchBytes = (size_t)1 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The array's name on the host is only a stand-in; the kernels need its device
// address, looked up once per device with that device current.
static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[64];

static qmm_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QMM_E_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QMM_E_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return QMM_OK;
}

}  // namespace qmm

using namespace qmm;

extern "C" {

// See include/qmm.h.  The activation rows are quantized into the library's own
// device array (every byte the multiply reads is written first, so nothing has
// to start at zero), then multiplied exactly as qmm_linear_<type> does.
qmm_status qmm_linear_noalloc(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t N, int64_t K,
                              qmm_stream_t stream) {
    const int act = act_type_of(wtype);
    if (act < 0) return QMM_E_TYPE;
    if (!W || !x || !y) return QMM_E_NULL;
    qmm_status st = check_shape(wtype, M, N, K);
    if (st != QMM_OK) return st;
    if (!aligned16(W) || !aligned16(x) || !aligned16(y)) return QMM_E_ALIGN;
    const size_t xrb = row_bytes_of(act, K);
    if ((uint64_t)M > kNoAllocScratchBytes / xrb) return QMM_E_SCRATCH;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != QMM_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    if (prefill_on_tensor_cores(wtype, M, K)) {  // quantize all rows once, then the tensor-core prefill
        st = quantize_act_launch(act, x, scratch, M, K, cs, true);
        if (st != QMM_OK) return st;
        return prefill_launch(wtype, W, scratch, y, M, N, K, cs, true);
    }
    // one launch per token that quantizes its row and multiplies; a row too
    // large for that kernel's shared memory is quantized by its own kernel first
    st = matvec_fused_dispatch(wtype, W, x, scratch, y, N, K, cs, true);
    if (st == QMM_OK) {
        for (int64_t t = 1; t < M; t++) {
            st = matvec_fused_dispatch(wtype, W, x + t * K, (uint8_t*)scratch + t * xrb, y + t * N, N, K, cs, true);
            if (st != QMM_OK) return st;
        }
        return QMM_OK;
    }
    if (st != QMM_E_SHAPE) return st;
    st = quantize_act_launch(act, x, scratch, M, K, cs, true);
    if (st != QMM_OK) return st;
    for (int64_t t = 0; t < M; t++) {
        st = matvec_dispatch(wtype, W, (const uint8_t*)scratch + t * xrb, y + t * N, N, K, cs, true);
        if (st != QMM_OK) return st;
    }
    return QMM_OK;
}

}  // extern "C"

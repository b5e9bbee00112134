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
// to start at zero), then multiplied by the same code as qmm_linear_<type>;
// more rows than the array holds give QMM_E_SCRATCH before any launch.
qmm_status qmm_linear_noalloc(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t N, int64_t K,
                              qmm_stream_t stream) {
    if (act_type_of(wtype) < 0) return QMM_E_TYPE;
    if (!W || !x || !y) return QMM_E_NULL;
    void* scratch = nullptr;
    const qmm_status st = noalloc_scratch(&scratch);
    if (st != QMM_OK) return st;
    const NoWorkspaceAllocScope no_alloc;  // the K-quant prefill keeps its in-kernel conversion
    return linear_impl(wtype, W, x, scratch, kNoAllocScratchBytes, y, M, N, K, (cudaStream_t)stream);
}

}  // extern "C"

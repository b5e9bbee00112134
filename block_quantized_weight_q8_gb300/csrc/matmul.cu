// matmul.cu -- the prefill matmul Y[M][N] = xq[M] . W^T for Q4_0 weights.
#include "qmm_device.cuh"
#include "qmm_host.h"

namespace qmm {

static __device__ unsigned int g_matmul_error = 0;

qmm_status matvec_dispatch(int wt, const void* W, const void* xq, float* y, int64_t N, int64_t K, cudaStream_t stream,
                           bool pdl);

qmm_status matmul_q4_0_launch(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                              cudaStream_t stream, bool pdl) {
    const size_t xrb = row_bytes_of(QMM_Q8_0, K);
    for (int64_t t = 0; t < M; t++) {
        qmm_status st = matvec_dispatch(QMM_Q4_0, W, (const uint8_t*)xq + t * xrb, Y + t * N, N, K, stream, pdl);
        if (st != QMM_OK) return st;
    }
    return QMM_OK;
}

}  // namespace qmm

using namespace qmm;

extern "C" {

qmm_status qmm_matmul_q4_0(const void* W, const void* xq, float* Y, int64_t M, int64_t N, int64_t K,
                           qmm_stream_t stream) {
    if (!W || !xq || !Y) return QMM_E_NULL;
    qmm_status st = check_shape(QMM_Q4_0, M, N, K);
    if (st != QMM_OK) return st;
    if (!aligned16(W) || !aligned16(xq) || !aligned16(Y)) return QMM_E_ALIGN;
    return matmul_q4_0_launch(W, xq, Y, M, N, K, (cudaStream_t)stream, false);
}

unsigned qmm_internal_matmul_error(int clear) {
    unsigned v = 0;
    cudaMemcpyFromSymbol(&v, g_matmul_error, sizeof(v));
    if (clear) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_matmul_error, &z, sizeof(z));
    }
    return v;
}

}  // extern "C"

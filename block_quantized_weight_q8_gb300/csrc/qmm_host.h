// qmm_host.h -- host-side helpers shared by the libqmm translation units:
// argument validation, device properties, and launch utilities.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "qmm.h"

namespace qmm {

constexpr int64_t kMaxK = 65536;
constexpr int64_t kMaxDim = 2147483647LL;

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline int block_values_of(int t) {
    switch (t) {
    case QMM_Q4_0: case QMM_Q8_0: case QMM_Q4_1: case QMM_Q5_0: case QMM_Q5_1: return 32;
    case QMM_Q4_K: case QMM_Q6_K: case QMM_Q2_K: case QMM_Q8_K: case QMM_Q5_K: return 256;
    default: return 0;
    }
}
inline size_t block_bytes_of(int t) {
    switch (t) {
    case QMM_Q4_0: return 18;
    case QMM_Q8_0: return 34;
    case QMM_Q4_K: return 144;
    case QMM_Q6_K: return 210;
    case QMM_Q2_K: return 84;
    case QMM_Q8_K: return 292;
    case QMM_Q4_1: return 20;
    case QMM_Q5_0: return 22;
    case QMM_Q5_1: return 24;
    case QMM_Q5_K: return 176;
    default: return 0;
    }
}
inline int act_type_of(int wt) {
    switch (wt) {
    case QMM_Q4_0: case QMM_Q8_0: case QMM_Q4_1: case QMM_Q5_0: case QMM_Q5_1: return QMM_Q8_0;
    case QMM_Q4_K: case QMM_Q6_K: case QMM_Q2_K: case QMM_Q5_K: return QMM_Q8_K;
    default: return -1;
    }
}
inline size_t row_bytes_of(int t, int64_t K) {
    const int bv = block_values_of(t);
    if (bv == 0 || K <= 0 || K % bv) return 0;
    return (size_t)(K / bv) * block_bytes_of(t);
}

// Shape check shared by the calls: M, N, K in range, K a multiple of the
// block of type t, K within the shared-memory activation limit.
inline qmm_status check_shape(int t, int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxK) return QMM_E_SHAPE;
    const int bv = block_values_of(t);
    if (bv == 0) return QMM_E_TYPE;
    if (K % bv) return QMM_E_SHAPE;
    return QMM_OK;
}

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int max_smem_optin = 0;
    int smem_per_sm = 0;    // shared memory of one SM, all resident CTAs together
    int smem_reserved = 0;  // shared memory the system keeps per resident CTA
};

// Properties of the current device (cached per device id).
qmm_status current_device(DeviceInfo* info);

// Per-device one-time set-up (kernel attributes, cached device properties)
// that host threads may reach concurrently: the first caller on a device runs
// it under a lock, later callers see the finished flag; a set-up that fails is
// tried again on the next call.
class PerDeviceOnce {
  public:
    template <class F>
    qmm_status run(int dev, F&& setup) {
        if (dev < 0 || dev >= kDevices) return QMM_E_CUDA;
        if (done_[dev].load(std::memory_order_acquire)) return QMM_OK;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev].load(std::memory_order_relaxed)) return QMM_OK;
        const qmm_status st = setup();
        if (st == QMM_OK) done_[dev].store(true, std::memory_order_release);
        return st;
    }

  private:
    static constexpr int kDevices = 64;
    std::atomic<bool> done_[kDevices] = {};
    std::mutex mu_;
};

// The quantize + multiply with a caller scratch buffer (qmm_linear_<wtype>),
// also used by the entry points that supply their own scratch.  wt must be a
// weight type.
qmm_status linear_impl(int wt, const void* W, const float* x, void* scratch, size_t scratch_bytes, float* y,
                       int64_t M, int64_t N, int64_t K, cudaStream_t stream);

// A 2-D TMA map over `rows` rows of `row_bytes` bytes, viewed as elements of
// `elem_bytes` (2 or 8) bytes, with boxes of `box_bytes` x 128 rows; reads past
// the end of a row or below the last row return zeros.  False if the driver
// rejects the map (or has no cuTensorMapEncodeTiled).
bool make_row_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                  int elem_bytes);

// True while an entry point that promises no allocation runs on this thread:
// the K-quant prefill then converts the activation in its kernel instead of in
// a pre-pass with a stream-ordered workspace.
extern thread_local bool tl_no_workspace_alloc;
struct NoWorkspaceAllocScope {
    bool prev;
    NoWorkspaceAllocScope() : prev(tl_no_workspace_alloc) { tl_no_workspace_alloc = true; }
    ~NoWorkspaceAllocScope() { tl_no_workspace_alloc = prev; }
};

inline qmm_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_E_CUDA;
}

}  // namespace qmm

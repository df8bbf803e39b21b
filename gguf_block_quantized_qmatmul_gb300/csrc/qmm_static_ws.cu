// qmm_static_ws.cu -- qmm_matmul for callers that cannot allocate device memory.
//
// Some callers of this library never get to call cudaMalloc: a host engine
// that owns every device allocation (for its own accounting or pooling) and
// only hands plugins finished input and output buffers, or a latency-critical
// loop that must not hit the allocator's implicit synchronization.  For the
// shapes where qmm_matmul needs a workspace (K split across CTAs), this entry
// point takes its scratch from one array in the library's own device memory
// instead of from the caller.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/qmm.h"

namespace {

// The scratch: one array per device that loads the library, kept until exit.
static __device__ __align__(256) unsigned char g_static_workspace[QMM_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDev = 64;
std::atomic<void*> g_static_ws_addr[kMaxDev];  // device address of the array, per device

// Set-up, once per device, with that device current: in host code the array's
// name is only a stand-in, so the device address has to be looked up.  Host
// threads racing on a device's first call look up the same address; the
// cache is atomic.
qmm_status static_workspace_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QMM_ERR_CUDA;
    void* p = g_static_ws_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return QMM_ERR_CUDA;
        g_static_ws_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return QMM_OK;
}

}  // namespace

extern "C" qmm_status qmm_matmul_static_workspace(qmm_type wtype, qmm_act_mode mode, const void* wq, const float* x,
                                                  float* y, int64_t M, int64_t N, int64_t K, qmm_stream_t stream) {
    // sizes beyond the array are refused before anything is launched
    const size_t need = qmm_matmul_workspace(wtype, mode, M, N, K);
    if (need > (size_t)QMM_STATIC_WORKSPACE_BYTES) return QMM_ERR_WORKSPACE;
    void* ws = nullptr;
    const qmm_status st = static_workspace_address(&ws);
    if (st != QMM_OK) return st;
    // qmm_matmul clears on `stream` the part of the workspace that must start
    // at zero (the K-split arrival counters of the streaming and tcgen05
    // kernels) before its launch; partial sums are overwritten and need no
    // clearing.
    return qmm_matmul(wtype, mode, wq, x, y, M, N, K, ws, (size_t)QMM_STATIC_WORKSPACE_BYTES, stream);
}

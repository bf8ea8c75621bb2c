// qmm_noalloc: qmm() for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or cudaMallocAsync) on the path where they run the matmul: a host
// framework that plans every device buffer ahead of time and forbids allocations during its execution
// step (plugins of inference engines are typical), code with hard latency limits where an allocation
// may synchronize the device or take the driver's allocation lock, or code capturing work into a CUDA
// graph under a capture mode that rejects allocation calls. For them this entry point runs exactly what
// qmm_ws() runs, with the scratch of the tensor-core path (the bfloat16 copy of binary32 activations that
// wide plans read) placed in one statically sized device array that belongs to this library.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds it until the
// process exits, so its size is kept modest (QMM_NOALLOC_SCRATCH_BYTES). Host code cannot use the name
// of a __device__ variable as a device address (on the host it denotes a stand-in object), so the
// device address is looked up once per device with cudaGetSymbolAddress, with that device current, and
// passed on as the workspace pointer.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/qmm.h"

namespace wqk {
int check_qmm_args(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, const float *y);
}

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[QMM_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device (looked up on the first call per device; host
// threads that race on the first lookup all store the same address).
void *scratch_ptr() {
    static std::atomic<void *> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    void *p = cache[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        cache[dev].store(p, std::memory_order_relaxed);
    }
    return p;
}

}  // namespace

extern "C" int qmm_noalloc(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                           void *stream) {
    // Arguments first (the same checks and codes as qmm), then the array's address (so that the first call
    // on a device sets it up whatever path it takes), then the scratch this call needs, refused before
    // anything is launched when it does not fit.
    const int rc = wqk::check_qmm_args(wq, qtype, N, K, x, M, y);
    if (rc) return rc;
    void *ws = scratch_ptr();
    if (!ws) return QMM_ECUDA;
    const size_t need = qmm_workspace_size(qtype, N, K, M);
    if (need > (size_t)QMM_NOALLOC_SCRATCH_BYTES) return QMM_EWORKSPACE;
    return qmm_ws(wq, qtype, N, K, x, M, y, need ? ws : nullptr, need ? (size_t)QMM_NOALLOC_SCRATCH_BYTES : 0,
                  stream);
}

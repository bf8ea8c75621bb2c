// qmm_noalloc: qmm() for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or cudaMallocAsync) on the path where they run the matmul: a host
// framework that plans every device buffer ahead of time and forbids allocations during its execution
// step (plugins of inference engines are typical), code with hard latency limits where an allocation
// may synchronize the device or take the driver's allocation lock, or code capturing work into a CUDA
// graph under a capture mode that rejects allocation calls. For them this entry point runs exactly what
// qmm_ws() runs, with the scratch of the tensor-core path (the bfloat16 copy of the activations and the
// split-K partial sums) placed in one statically sized device array that belongs to this library.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds it until the
// process exits, so its size is kept modest (QMM_NOALLOC_SCRATCH_BYTES). Host code cannot use the name
// of a __device__ variable as a device address (on the host it denotes a stand-in object), so the
// device address is looked up once per device with cudaGetSymbolAddress, with that device current, and
// passed on as the workspace pointer.
#include <cuda_runtime.h>

#include "../../include/qmm.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[QMM_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device (set up on the first call per device).
void *scratch_ptr() {
    static void *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        cache[dev] = p;
    }
    return cache[dev];
}

}  // namespace

extern "C" int qmm_noalloc(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                           void *stream) {
    // The shapes decide how much scratch the call needs; refuse what does not fit before touching the GPU.
    const size_t need = qmm_workspace_size(qtype, N, K, M);
    if (need > (size_t)QMM_NOALLOC_SCRATCH_BYTES) return QMM_EWORKSPACE;
    if (need == 0) return qmm_ws(wq, qtype, N, K, x, M, y, nullptr, 0, stream);
    void *ws = scratch_ptr();
    if (!ws) return QMM_ECUDA;
    return qmm_ws(wq, qtype, N, K, x, M, y, ws, (size_t)QMM_NOALLOC_SCRATCH_BYTES, stream);
}

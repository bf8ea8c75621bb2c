// Tensor-core path for larger token counts: y = x * dequant(W)^T on tcgen05 with a TMEM accumulator.
//
// The method (candle PR 4056, "Metal: 64-token tile for the quantized matrix-matrix kernel", section "Why
// the tile sets the weight reuse"): a thread block owns a slab of weight rows; at every step along K it
// reads those rows' quantized blocks, dequantizes them into shared memory and multiplies them by every
// token of its tile, so each weight is fetched and dequantized once per token tile. Here:
//   - a CTA owns BM = 128 weight rows (the MMA's M) and one token tile of T = 32, 64 or 128 tokens (the
//     MMA's N);
//   - each K step of 64 columns: the CTA's threads decode the 128 x 64 weight slab to bf16 (round to
//     nearest even) straight into the 128-byte-swizzled K-major layout; one thread loads the T x 64 bf16
//     activation tile by TMA (rows past M read as zero) and issues four K=16 tcgen05.mma into TMEM;
//   - stages are recycled through mbarriers signalled by tcgen05.commit;
//   - the epilogue reads TMEM with tcgen05.ld (one TMEM lane per weight row) and writes y as binary32.
// Bit-identity across T: every output element sees the same K steps and the same K=16 MMAs in the same
// order whatever T is (candle PR 4056, section "Same results, bit for bit"); T only changes how many
// token columns share one decoded slab.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "qmm_common.cuh"

namespace wqk {
namespace mm {

constexpr int BM = 128;            // weight rows per CTA
constexpr int BK = 64;             // columns per K step: one 128-byte swizzle row of bf16
constexpr int STAGES = 3;
constexpr int A_STAGE = BM * BK * 2;   // 16 KB
constexpr int THREADS = 128;

__host__ __device__ constexpr int b_stage_bytes(int T) { return T * BK * 2; }
__host__ __device__ constexpr int smem_bytes(int T) {
    return 1024 /* alignment slack */ + STAGES * (A_STAGE + b_stage_bytes(T)) + 256 /* barriers */;
}

// Byte offset of the 16-byte piece p (bf16 columns 8p .. 8p+7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int p) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((p ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int QT, int T>
__global__ void __launch_bounds__(THREADS, 1)
    mm_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint8_t *__restrict__ wq, int N, int64_t K,
              int64_t rowbytes, int M, float *__restrict__ y, unsigned int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * b_stage_bytes(T));
    uint64_t *done = full + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + STAGES);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * T;
    constexpr uint32_t TMEM_COLS = T < 32 ? 32 : T;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&done[s], 1);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int nsteps = (int)((K + BK - 1) / BK);
    const int nchunks = (int)(K / 32);      // K is a multiple of 32 on this path
    const int row = n0 + tid;               // the weight row this thread decodes
    const uint8_t *wrow = wq + (int64_t)(row < N ? row : 0) * rowbytes;
    const uint32_t sA_u32 = ptx::smem_u32(sA), sB_u32 = ptx::smem_u32(sB);
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, T);
    int issued = 0;          // steps whose MMAs thread 0 committed
    int loaded = 0;          // steps whose activation tile thread 0 requested
    bool aborted = false;

    for (int i = 0; i < nsteps; ++i) {
        const int s = i % STAGES;
        bool ok = true;
        if (i >= STAGES) ok = ptx::mbar_wait(&done[s], ((i / STAGES) - 1) & 1, status);
        if (tid == 0 && ok) {
            ptx::mbar_arrive_expect_tx(&full[s], (uint32_t)b_stage_bytes(T));
            ptx::tma_load_2d(sB + s * b_stage_bytes(T), &tmap_x, i * BK, m0, &full[s]);
            loaded = i + 1;
        }
        // Decode this thread's row: two 32-weight chunks = 64 bf16 = eight 16-byte pieces.
        const uint32_t a_base = sA_u32 + s * A_STAGE;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = 2 * i + h;
            float w[32];
            if (row < N && c < nchunks) {
                decode_chunk<QT>(wrow, c, K, w);
            } else {
#pragma unroll
                for (int l = 0; l < 32; ++l) w[l] = 0.0f;
            }
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                ptx::st_shared_v4(a_base + sw128_off(tid, 4 * h + p), pack_bf16x2(w[8 * p + 0], w[8 * p + 1]),
                                  pack_bf16x2(w[8 * p + 2], w[8 * p + 3]), pack_bf16x2(w[8 * p + 4], w[8 * p + 5]),
                                  pack_bf16x2(w[8 * p + 6], w[8 * p + 7]));
            }
        }
        ptx::fence_proxy_async_smem();
        if (__syncthreads_or(!ok || *abort_flag)) {
            aborted = true;
            break;
        }
        if (tid == 0) {
            if (ptx::mbar_wait(&full[s], (i / STAGES) & 1, status)) {
                ptx::tc_fence_after();
                const uint64_t adesc = ptx::sw128_desc(a_base);
                const uint64_t bdesc = ptx::sw128_desc(sB_u32 + s * b_stage_bytes(T));
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    // advancing 16 bf16 = 32 bytes inside the swizzle row moves the start address by 2 units
                    ptx::mma_bf16(tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (i | kk) != 0);
                }
                ptx::mma_commit(&done[s]);
                issued = i + 1;
            } else {
                *abort_flag = 1;
            }
        }
    }

    // Wait for the last committed MMAs (they cover every earlier one). Broadcast thread 0's view.
    __shared__ int s_issued, s_loaded;
    if (tid == 0) {
        s_issued = issued;
        s_loaded = loaded;
    }
    __syncthreads();
    const int last_issued = s_issued, last_loaded = s_loaded;
    bool ok = true;
    if (last_issued > 0) {
        const int li = last_issued - 1;
        ok = ptx::mbar_wait(&done[li % STAGES], (li / STAGES) & 1, status);
    }
    if (tid == 0 && last_loaded > last_issued) {
        // an activation tile was requested but never consumed (abort path): let it land before exiting
        const int li = last_loaded - 1;
        ptx::mbar_wait(&full[li % STAGES], (li / STAGES) & 1, status);
    }
    ptx::tc_fence_after();
    const bool good = !__syncthreads_or(aborted || !ok || *abort_flag);

    if (good) {
        const int r = n0 + warp * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
        for (int c0 = 0; c0 < T; c0 += 16) {
            uint32_t v[16];
            ptx::tmem_ld_32x32b_x16(lane_base + c0, v);
            ptx::tmem_ld_wait();
            if (r < N) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int tok = m0 + c0 + j;
                    if (tok < M) y[(int64_t)tok * N + r] = __uint_as_float(v[j]);
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// binary32 -> bfloat16 (round to nearest even), 8 elements per thread; n is a multiple of 8.
__global__ void x_to_bf16_kernel(const float4 *__restrict__ x, uint4 *__restrict__ out, int64_t n8) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = x[2 * i], b = x[2 * i + 1];
        out[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                            pack_bf16x2(b.z, b.w));
    }
}

}  // namespace mm

// ------------------------------------------------------------------------------------------ host side

// cuTensorMapEncodeTiled through the runtime's driver entry-point lookup, so that the library does not
// link libcuda directly (it loads on machines without a driver; calls then fail with QMM_ECUDA).
static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

static bool make_x_tmap(CUtensorMap *map, const void *xb, int64_t M, int64_t K, int T) {
    auto enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)mm::BK, (cuuint32_t)T};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(xb), dims,
                                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int QT, int T>
static int launch_mm_t(const void *wq, int64_t N, int64_t K, const void *xb, int64_t M, float *y,
                       unsigned int *status, cudaStream_t st) {
    CUtensorMap map;
    if (!make_x_tmap(&map, xb, M, K, T)) return -6;
    auto kern = mm::mm_kernel<QT, T>;
    const int smem = mm::smem_bytes(T);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -6;
    dim3 grid((unsigned)((N + mm::BM - 1) / mm::BM), (unsigned)((M + T - 1) / T));
    kern<<<grid, mm::THREADS, smem, st>>>(map, static_cast<const uint8_t *>(wq), (int)N, K, row_bytes(QT, K),
                                          (int)M, y, status);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

namespace {
struct MmLaunch {
    int tile;
    const void *wq;
    int64_t N, K;
    const void *xb;
    int64_t M;
    float *y;
    unsigned int *status;
    cudaStream_t st;
    template <int QT> int operator()() {
        switch (tile) {
        case 32: return launch_mm_t<QT, 32>(wq, N, K, xb, M, y, status, st);
        case 64: return launch_mm_t<QT, 64>(wq, N, K, xb, M, y, status, st);
        case 128: return launch_mm_t<QT, 128>(wq, N, K, xb, M, y, status, st);
        default: return -7;
        }
    }
};
}  // namespace

// x_bf16: M x K bf16, row stride K*2 bytes (16-byte multiple), 16-byte aligned.
int launch_mm(int qt, int tile, const void *wq, int64_t N, int64_t K, const void *x_bf16, int64_t M, float *y,
              unsigned int *status, cudaStream_t st) {
    MmLaunch f{tile, wq, N, K, x_bf16, M, y, status, st};
    return dispatch_type(qt, f);
}

int launch_x_to_bf16(const float *x, void *out, int64_t n, cudaStream_t st) {
    const int64_t n8 = n / 8;
    const int threads = 256;
    int64_t blocks = (n8 + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    mm::x_to_bf16_kernel<<<(unsigned)blocks, threads, 0, st>>>(reinterpret_cast<const float4 *>(x),
                                                               static_cast<uint4 *>(out), n8);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

}  // namespace wqk

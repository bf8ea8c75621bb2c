// Tensor-core path for larger token counts: y = x * dequant(W)^T on tcgen05 with a TMEM accumulator.
//
// The method (candle PR 4056, "Metal: 64-token tile for the quantized matrix-matrix kernel", section "Why
// the tile sets the weight reuse"): a thread block owns a slab of weight rows; at every step along K it
// reads those rows' quantized blocks, dequantizes them into shared memory and multiplies them by every
// token it holds, so each weight is fetched and dequantized once per token tile. Here:
//   - a CTA owns BM = 128 weight rows (the MMA's M) and J token tiles of T = 32, 64 or 128 tokens (the
//     MMA's N), J*T <= 256; the J tiles share every decoded slab;
//   - warp 0 loads the J*T x 64 bf16 activation tile of each K step by TMA (rows past M read as zero);
//   - warps 2..9 decode the 128 x 64 weight slab of each step to bf16 (round to nearest even of the
//     binary32 value) straight into the 128-byte-swizzled K-major layout tcgen05 reads;
//   - warp 1 issues, per step, 4 (K = 16) x J tcgen05.mma into TMEM and commits them to the stage's
//     "empty" barrier, which hands the stage back to the producer and the decoders;
//   - the decoder warps then read TMEM with tcgen05.ld and write y (or, when K is split over CTAs, a
//     binary32 partial that a second kernel adds up in a fixed order).
// Bit-identity across T: every output element sees the same K steps, the same K=16 MMAs in the same
// order and the same K split whatever T is (candle PR 4056, section "Same results, bit for bit").
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "qmm_common.cuh"

namespace wqk {
namespace mm {

constexpr int BM = 128;            // weight rows per CTA
constexpr int BK = 64;             // columns per K step: one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;   // 16 KB
constexpr int NDEC = 8;                // decoder / epilogue warps
constexpr int THREADS = 32 * (2 + NDEC);

__host__ __device__ constexpr int b_stage_bytes(int TN) { return TN * BK * 2; }
__host__ __device__ constexpr int smem_bytes(int TN) {
    return 1024 /* alignment slack */ + STAGES * (A_STAGE + b_stage_bytes(TN)) + 256 /* barriers */;
}

// Byte offset of the 16-byte piece p (bf16 columns 8p .. 8p+7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int p) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((p ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

struct Smem {
    uint64_t full_b[STAGES], full_a[STAGES], empty[STAGES], done;
    uint32_t tmem;
    int abort;
};

// out = y (S == 1) or the partial buffer of this K split (S > 1), both M x N binary32 row-major.
template <int QT, int T, int J>
__global__ void __launch_bounds__(THREADS, 1)
    mm_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint8_t *__restrict__ wq, int N, int64_t K,
              int64_t rowbytes, int M, float *__restrict__ out, int64_t split_stride, int ksteps_per_split,
              unsigned int *status) {
    constexpr int TN = T * J;
    constexpr uint32_t TMEM_COLS = TN <= 32 ? 32 : (TN <= 64 ? 64 : (TN <= 128 ? 128 : 256));
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, T);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    Smem *sm = reinterpret_cast<Smem *>(sB + STAGES * b_stage_bytes(TN));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * TN;
    const int split = blockIdx.z;
    const int ktotal = (int)((K + BK - 1) / BK);
    const int kbeg = split * ksteps_per_split;
    const int kend = (kbeg + ksteps_per_split < ktotal) ? kbeg + ksteps_per_split : ktotal;
    const int nsteps = kend > kbeg ? kend - kbeg : 0;
    float *y = out + (int64_t)split * split_stride;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&sm->full_b[s], 1);
            ptx::mbar_init(&sm->full_a[s], NDEC);
            ptx::mbar_init(&sm->empty[s], 1);
        }
        ptx::mbar_init(&sm->done, 1);
        sm->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&sm->tmem, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm->tmem;

    if (warp == 0) {
        // ---------------- activation producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nsteps; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !ptx::mbar_wait(&sm->empty[s], ((i / STAGES) - 1) & 1, status)) {
                    sm->abort = 1;
                    break;
                }
                if (*(volatile int *)&sm->abort) break;
                ptx::mbar_arrive_expect_tx(&sm->full_b[s], (uint32_t)b_stage_bytes(TN));
                ptx::tma_load_2d(sB + s * b_stage_bytes(TN), &tmap_x, (kbeg + i) * BK, m0, &sm->full_b[s]);
                issued = i + 1;
            }
            // every requested tile lands before the CTA may exit
            for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
                ptx::mbar_wait(&sm->full_b[i % STAGES], (i / STAGES) & 1, status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t sA_u32 = ptx::smem_u32(sA), sB_u32 = ptx::smem_u32(sB);
            for (int i = 0; i < nsteps; ++i) {
                const int s = i % STAGES;
                const uint32_t par = (i / STAGES) & 1;
                if (!ptx::mbar_wait(&sm->full_a[s], par, status) || !ptx::mbar_wait(&sm->full_b[s], par, status)) {
                    sm->abort = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t adesc = ptx::sw128_desc(sA_u32 + s * A_STAGE);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
                    for (int jj = 0; jj < J; ++jj) {
                        const uint64_t bdesc = ptx::sw128_desc(sB_u32 + s * b_stage_bytes(TN) + jj * T * 128);
                        // advancing 16 bf16 = 32 bytes inside the swizzle row moves the start address by 2 units
                        ptx::mma_bf16(tmem + jj * T, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (i | kk) != 0);
                    }
                }
                ptx::mma_commit(&sm->empty[s]);
            }
            ptx::mma_commit(&sm->done);   // tracks every MMA issued above
        }
    } else {
        // ---------------- decoders: warp d handles rows 16d .. 16d+15 of the slab; lane -> (row, chunk)
        const int d = warp - 2;
        const int r_local = 16 * d + (lane >> 1), h = lane & 1;
        const int row = n0 + r_local;
        const uint8_t *wrow = wq + (int64_t)(row < N ? row : N - 1) * rowbytes;
        const int nchunks = (int)((K + 31) / 32);
        const uint32_t sA_u32 = ptx::smem_u32(sA);
        for (int i = 0; i < nsteps; ++i) {
            const int s = i % STAGES;
            if (i >= STAGES && !ptx::mbar_wait(&sm->empty[s], ((i / STAGES) - 1) & 1, status)) {
                sm->abort = 1;
                break;
            }
            if (*(volatile int *)&sm->abort) break;
            const int c = 2 * (kbeg + i) + h;
            float w[32];
            if (row < N && c < nchunks) {
                decode_chunk<QT>(wrow, c, K, w);
            } else {
#pragma unroll
                for (int l = 0; l < 32; ++l) w[l] = 0.0f;
            }
            const uint32_t a_base = sA_u32 + s * A_STAGE;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                ptx::st_shared_v4(a_base + sw128_off(r_local, 4 * h + p), pack_bf16x2(w[8 * p + 0], w[8 * p + 1]),
                                  pack_bf16x2(w[8 * p + 2], w[8 * p + 3]), pack_bf16x2(w[8 * p + 4], w[8 * p + 5]),
                                  pack_bf16x2(w[8 * p + 6], w[8 * p + 7]));
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm->full_a[s]);
        }
        // ---------------- epilogue: TMEM lanes = weight rows, columns = tokens
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;       // two warps per quarter split the columns
        const int r = n0 + 32 * q + lane;
        if (nsteps > 0) {
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(&sm->done, 0, status) && !*(volatile int *)&sm->abort);
            ptx::tc_fence_after();
            if (ok) {
                const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll
                for (int c0 = half * (TN / 2); c0 < (half + 1) * (TN / 2); c0 += 16) {
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
        } else {
            // an empty K split contributes zeros
            for (int c0 = half * (TN / 2); c0 < (half + 1) * (TN / 2); ++c0) {
                const int tok = m0 + c0;
                if (r < N && tok < M) y[(int64_t)tok * N + r] = 0.0f;
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// y[i] = sum over s of part[s][i], s ascending (deterministic K-split reduction).
__global__ void splitk_reduce_kernel(const float4 *__restrict__ part, int64_t stride4, int S, float4 *__restrict__ y,
                                     int64_t n4) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = part[i];
        for (int s = 1; s < S; ++s) {
            const float4 b = part[i + s * stride4];
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        y[i] = a;
    }
}
__global__ void splitk_reduce_tail_kernel(const float *__restrict__ part, int64_t stride, int S, float *__restrict__ y,
                                          int64_t beg, int64_t n) {
    for (int64_t i = beg + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float a = part[i];
        for (int s = 1; s < S; ++s) a += part[i + s * stride];
        y[i] = a;
    }
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

static bool make_x_tmap(CUtensorMap *map, const void *xb, int64_t M, int64_t K, int rows) {
    auto enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)mm::BK, (cuuint32_t)rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(xb), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// Token tiles per CTA: as many as fit 256 columns, but not more than the tokens need (a power of two).
inline int tiles_per_cta(int T, int64_t M) {
    int j = 256 / T;
    const int64_t need = (M + T - 1) / T;
    while (j > 1 && j / 2 >= need) j /= 2;
    return j;
}

template <int QT, int T, int J>
int launch_mm_t(const void *wq, int64_t N, int64_t K, const void *xb, int64_t M, float *out, int S, int kps,
                int64_t split_stride, unsigned int *status, cudaStream_t st) {
    CUtensorMap map;
    if (!make_x_tmap(&map, xb, M, K, T * J)) return -6;
    auto kern = mm::mm_kernel<QT, T, J>;
    const int smem = mm::smem_bytes(T * J);
    static bool attr_set = false;   // once per kernel instance
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -6;
        attr_set = true;
    }
    dim3 grid((unsigned)((N + mm::BM - 1) / mm::BM), (unsigned)((M + T * J - 1) / (T * J)), (unsigned)S);
    kern<<<grid, mm::THREADS, smem, st>>>(map, static_cast<const uint8_t *>(wq), (int)N, K, row_bytes(QT, K),
                                          (int)M, out, split_stride, kps, status);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

struct MmLaunch {
    int tile, J;
    const void *wq;
    int64_t N, K;
    const void *xb;
    int64_t M;
    float *out;
    int S, kps;
    int64_t split_stride;
    unsigned int *status;
    cudaStream_t st;
    template <int QT, int T, int JJ> int go_j() {
        if constexpr (T * JJ <= 256) return launch_mm_t<QT, T, JJ>(wq, N, K, xb, M, out, S, kps, split_stride, status, st);
        else return -7;
    }
    template <int QT, int T> int go() {
        switch (J) {
        case 1: return go_j<QT, T, 1>();
        case 2: return go_j<QT, T, 2>();
        case 4: return go_j<QT, T, 4>();
        case 8: return go_j<QT, T, 8>();
        default: return -7;
        }
    }
    template <int QT> int operator()() {
        switch (tile) {
        case 32: return go<QT, 32>();
        case 64: return go<QT, 64>();
        case 128: return go<QT, 128>();
        default: return -7;
        }
    }
};

}  // namespace

// K split of the tensor-core path, a function of (N, K, M) only (never of the token tile), so that every
// tile variant adds the same partial sums: split while CTAs of 128 rows x 256 tokens leave more than
// half the SMs idle, keeping at least 8 K steps per split.
int mm_ksplit(int64_t N, int64_t K, int64_t M) {
    const int64_t ksteps = (K + mm::BK - 1) / mm::BK;
    const int64_t ctas = ((N + mm::BM - 1) / mm::BM) * ((M + 255) / 256);
    int64_t S = 1;
    while (ctas * S * 2 <= 148 && ksteps / (S * 2) >= 8 && S < 16) S *= 2;
    return (int)S;
}

// Partial buffers of the K splits are M*N binary32 each, padded to a multiple of 4 elements so that every
// split starts 16-byte aligned.
static inline int64_t split_stride_of(int64_t M, int64_t N) { return (M * N + 3) & ~(int64_t)3; }

// Bytes of split-K partials needed (0 when the K dimension is not split).
size_t mm_partial_bytes(int64_t N, int64_t K, int64_t M) {
    const int S = mm_ksplit(N, K, M);
    return S > 1 ? (size_t)S * (size_t)split_stride_of(M, N) * 4 : 0;
}

// x_bf16: M x K bf16, row stride K*2 bytes (16-byte multiple), 16-byte aligned. `part` (when the K
// dimension is split) holds S * M * N binary32.
int launch_mm(int qt, int tile, const void *wq, int64_t N, int64_t K, const void *x_bf16, int64_t M, float *y,
              float *part, unsigned int *status, cudaStream_t st) {
    const int S = mm_ksplit(N, K, M);
    const int64_t ksteps = (K + mm::BK - 1) / mm::BK;
    const int kps = (int)((ksteps + S - 1) / S);
    float *out = S > 1 ? part : y;
    const int64_t sstride = split_stride_of(M, N);
    MmLaunch f{tile, tiles_per_cta(tile, M), wq, N, K, x_bf16, M, out, S, kps, sstride, status, st};
    int rc = dispatch_type(qt, f);
    if (rc || S == 1) return rc;
    const int64_t n = M * N, n4 = n / 4;
    if (n4 > 0) {
        int64_t blocks = (n4 + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        mm::splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(part),
                                                                   sstride / 4, S, reinterpret_cast<float4 *>(y), n4);
    }
    if (n % 4) mm::splitk_reduce_tail_kernel<<<1, 32, 0, st>>>(part, sstride, S, y, n4 * 4, n);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
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

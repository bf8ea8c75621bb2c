// Binary32 CUDA-core mat-vec path for small token counts (M <= 16), y[m, n] = sum_k w[n, k] x[m, k]: the
// plain weight types (F32, F16, BF16; the quantized types run on the tensor-core mat-vec kernel). Rows whose
// bytes are whole 16-byte runs (K a multiple of 8) take the row-streaming kernel gemv_plain_kernel below;
// other K take the chunk kernel described here, which also decodes every block format.
//
// Lane mapping. A warp works on weight rows; its lanes take the row's 32-weight chunks (nb32 = K/32 of
// them), decode each chunk once to binary32 and multiply it by every token's activations, keeping one
// accumulator per token. Two idle-lane fixes from the pages are built in:
//   - narrow K (llama.cpp PR 28086, "metal : fix idle threads in mul_mv_iq3_xxs for ne00 < 1024",
//     section "Overview"): when nb32 < 32 and nb32 divides 32, the warp splits into 32/nb32 lane groups
//     that each take a different row, so no lane idles; otherwise the plain mapping (lane = chunk) is kept,
//     exactly the pages' fallback for nb32 = 24;
//   - small M (tiny-llm PR 122, "perf: Optimize quantized matmul for small decode batches", section
//     "Summary"): no lane is ever assigned to a token. Every lane walks weights and loops over the M
//     tokens itself, which is the pages' x_size shift taken to x_size = 1; kernels are specialised per
//     M bucket 1, 2, 4, 8, 16 (the pages' buckets) so that a bucket keeps only as many accumulators as it
//     needs.
// The per-token partial sums of a row are combined with warp shuffles within the row's lane group.
#include <cuda_runtime.h>

#include "qmm_common.cuh"

namespace wqk {
namespace gemv {

constexpr int WARPS = 8;

template <bool XBF16>
__device__ __forceinline__ void load_x32(const void *x, int64_t off, float (&v)[32]) {
    if constexpr (XBF16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 q = __ldg(p + i);
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
                v[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
            }
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + off);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 q = __ldg(p + i);
            v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
        }
    }
}

// Activations of one chunk with a K tail (plain weight types with K not a multiple of 32).
template <bool XBF16>
__device__ __forceinline__ void load_x32_tail(const void *x, int64_t rowoff, int64_t k0, int64_t K, float (&v)[32]) {
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        const int64_t k = k0 + l;
        if (k < K) {
            if constexpr (XBF16) v[l] = __uint_as_float((uint32_t)static_cast<const uint16_t *>(x)[rowoff + k] << 16);
            else v[l] = static_cast<const float *>(x)[rowoff + k];
        } else {
            v[l] = 0.0f;
        }
    }
}

// split = rows per warp pass (32 / nb32 on the narrow-K path, else 1); lanes per row L = 32 / split.
template <int QT, int MB, bool XBF16>
__global__ void __launch_bounds__(WARPS * 32)
    gemv_kernel(const uint8_t *__restrict__ wq, int64_t N, int64_t K, int64_t rowbytes, const void *__restrict__ x,
                int M, float *__restrict__ y, int split) {
    const int lane = threadIdx.x & 31;
    const int L = 32 / split;
    const int sub = lane / L, cl = lane % L;
    const int nchunks = (int)((K + 31) / 32);
    const bool vec_x = (K % 32) == 0;
    const int64_t groups = (N + split - 1) / split;
    const int64_t warp0 = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
    const int64_t wstride = (int64_t)gridDim.x * WARPS;

    for (int64_t g = warp0; g < groups; g += wstride) {
        const int64_t n = g * split + sub;
        const bool valid = n < N;
        const uint8_t *row = wq + (valid ? n : 0) * rowbytes;
        float acc[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.0f;
        if (valid) {
            for (int c = cl; c < nchunks; c += L) {
                float w[32];
                decode_chunk<QT>(row, c, K, w);
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    if (m < M) {
                        float xv[32];
                        if (vec_x) load_x32<XBF16>(x, (int64_t)m * K + 32 * (int64_t)c, xv);
                        else load_x32_tail<XBF16>(x, (int64_t)m * K, 32 * (int64_t)c, K, xv);
                        float s = acc[m];
#pragma unroll
                        for (int l = 0; l < 32; ++l) s = fmaf(w[l], xv[l], s);
                        acc[m] = s;
                    }
                }
            }
        }
        // reduce within the row's lane group (L is a power of two)
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            float v = acc[m];
            for (int off = L >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            acc[m] = v;
        }
        if (valid && cl == 0) {
#pragma unroll
            for (int m = 0; m < MB; ++m)
                if (m < M) y[(int64_t)m * N + n] = acc[m];
        }
    }
}

// Plain weight types (F32, F16, BF16) with 16-byte-aligned rows (K a multiple of 8): a warp owns R rows and
// walks all of K; lane l takes the 4 consecutive weights 4l, 4l + 128, ... of each of its rows (one 16- or
// 8-byte load per row per step, so a warp reads whole 512- or 256-byte runs of each row) and multiplies them
// by the same 4 activations of every token, keeping R x M binary32 accumulators; the 32 lanes' sums of a
// (row, token) are then added by a butterfly of shuffles. The products are exact (binary16/bfloat16 weights
// and bfloat16 activations widen exactly), so the result stays in the binary32 class. R trades the
// activation reloads (M loads per R weight loads, served by L1) against registers.
template <int QT> __device__ __forceinline__ void load_w4(const uint8_t *row, int64_t k, float (&w)[4]) {
    if constexpr (QT == T_F32) {
        const float4 q = __ldcs(reinterpret_cast<const float4 *>(row) + k / 4);
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    } else {
        const uint2 q = __ldcs(reinterpret_cast<const uint2 *>(row) + k / 4);
        if constexpr (QT == T_F16) {
            w[0] = h2f(q.x & 0xffffu); w[1] = h2f(q.x >> 16); w[2] = h2f(q.y & 0xffffu); w[3] = h2f(q.y >> 16);
        } else {
            w[0] = bf2f(q.x & 0xffffu); w[1] = bf2f(q.x >> 16); w[2] = bf2f(q.y & 0xffffu); w[3] = bf2f(q.y >> 16);
        }
    }
}
template <bool XBF16> __device__ __forceinline__ void load_x4(const void *x, int64_t off, float (&v)[4]) {
    if constexpr (XBF16) {
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(x) + off));
        v[0] = bf2f(q.x & 0xffffu); v[1] = bf2f(q.x >> 16); v[2] = bf2f(q.y & 0xffffu); v[3] = bf2f(q.y >> 16);
    } else {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(x) + off));
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
}
constexpr int PLAIN_WARPS = 4;
// Rows per warp: one up to 2 tokens, two above (measured on GB300, 9728 x 2560: more warps in flight beat
// fewer activation reloads; 8 rows per warp streamed at a third of the rate at one token).
template <int MB> __host__ __device__ constexpr int plain_rows() { return MB <= 2 ? 1 : 2; }

template <int QT, int MB, bool XBF16>
__global__ void __launch_bounds__(PLAIN_WARPS * 32)
    gemv_plain_kernel(const uint8_t *__restrict__ wq, int64_t N, int64_t K, const void *__restrict__ x, int M,
                      float *__restrict__ y) {
    constexpr int R = plain_rows<MB>();
    constexpr int ES = QT == T_F32 ? 4 : 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row0 = ((int64_t)blockIdx.x * PLAIN_WARPS + warp) * R;
    if (row0 >= N) return;                                    // whole warp
    const uint8_t *rows[R];
#pragma unroll
    for (int r = 0; r < R; ++r) rows[r] = wq + (row0 + r < N ? row0 + r : N - 1) * K * ES;
    float acc[R][MB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[r][m] = 0.0f;
#pragma unroll 4
    for (int64_t k = 4 * lane; k < K; k += 128) {
        float w[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) load_w4<QT>(rows[r], k, w[r]);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            if (m < M) {
                float v[4];
                load_x4<XBF16>(x, (int64_t)m * K + k, v);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float a = acc[r][m];
                    a = fmaf(w[r][0], v[0], a);
                    a = fmaf(w[r][1], v[1], a);
                    a = fmaf(w[r][2], v[2], a);
                    a = fmaf(w[r][3], v[3], a);
                    acc[r][m] = a;
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            acc[r][m] = v;
        }
    // lane (r * MB + m) % 32 stores (row r, token m)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m)
            if (lane == (r * MB + m) % 32 && m < M && row0 + r < N) y[(int64_t)m * N + row0 + r] = acc[r][m];
}

// Rows per warp pass for a row of nb32 chunks.
__host__ __device__ inline int row_split(int64_t nb32) {
    return (nb32 < 32 && nb32 > 0 && (32 % nb32) == 0) ? (int)(32 / nb32) : 1;
}

}  // namespace gemv

template <int QT, int MB, bool XBF16>
static int launch_gemv_b(const void *wq, int64_t N, int64_t K, const void *x, int M, float *y, cudaStream_t st) {
    const int split = gemv::row_split((K + 31) / 32);
    const int64_t groups = (N + split - 1) / split;
    int64_t blocks = (groups + gemv::WARPS - 1) / gemv::WARPS;
    if (blocks > 65535) blocks = 65535;
    gemv::gemv_kernel<QT, MB, XBF16><<<(unsigned)blocks, gemv::WARPS * 32, 0, st>>>(
        static_cast<const uint8_t *>(wq), N, K, row_bytes(QT, K), x, M, y, split);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

template <int QT, int MB, bool XBF16>
static int launch_gemv_plain(const void *wq, int64_t N, int64_t K, const void *x, int M, float *y, cudaStream_t st) {
    constexpr int R = gemv::plain_rows<MB>();
    const int64_t blocks = (N + R * gemv::PLAIN_WARPS - 1) / (R * gemv::PLAIN_WARPS);
    if (blocks > 0x7fffffff) return -3;
    gemv::gemv_plain_kernel<QT, MB, XBF16><<<(unsigned)blocks, gemv::PLAIN_WARPS * 32, 0, st>>>(
        static_cast<const uint8_t *>(wq), N, K, x, M, y);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

namespace {
struct GemvLaunch {
    bool xbf16;
    const void *wq;
    int64_t N, K;
    const void *x;
    int M;
    float *y;
    cudaStream_t st;
    template <int QT, int MB> int go() {
        if constexpr (is_plain(QT)) {
            // whole 16-byte runs of every weight and activation row: the row-streaming kernel
            if (K % 8 == 0)
                return xbf16 ? launch_gemv_plain<QT, MB, true>(wq, N, K, x, M, y, st)
                             : launch_gemv_plain<QT, MB, false>(wq, N, K, x, M, y, st);
        }
        return xbf16 ? launch_gemv_b<QT, MB, true>(wq, N, K, x, M, y, st)
                     : launch_gemv_b<QT, MB, false>(wq, N, K, x, M, y, st);
    }
    template <int QT> int operator()() {
        if (M <= 1) return go<QT, 1>();
        if (M <= 2) return go<QT, 2>();
        if (M <= 4) return go<QT, 4>();
        if (M <= 8) return go<QT, 8>();
        return go<QT, 16>();
    }
};
}  // namespace

// Tokens are processed 16 at a time; each group picks the smallest M bucket that holds it.
int launch_gemv(int qt, bool xbf16, const void *wq, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                cudaStream_t st) {
    const int esz = xbf16 ? 2 : 4;
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        const int mg = (int)((M - m0) < 16 ? (M - m0) : 16);
        GemvLaunch f{xbf16, wq, N, K, static_cast<const uint8_t *>(x) + m0 * K * esz, mg, y + m0 * N, st};
        const int rc = dispatch_type(qt, f);
        if (rc != 0) return rc;
    }
    return 0;
}

}  // namespace wqk

// Expert-indexed mat-vec for mixture-of-experts layers (the pages' MUL_MAT_ID; llama.cpp PR 28086,
// "metal : fix idle threads in mul_mv_iq3_xxs for ne00 < 1024", sections "Overview" and "Test
// methodology": one mat-vec per routed (token, expert) pair during speculative verify, n = 1..24 tokens,
// top-8 routing, narrow K).
//
// Grouped gather: every CTA reads all M*topk expert ids into shared memory and builds the sorted list of
// distinct experts that occur, with the (token, slot) pairs routed to each. CTA (row block rb, rank u)
// serves the u-th distinct expert: it streams that expert's rows of block rb once and multiplies each
// decoded chunk by the activations of every token routed to the expert. So each expert's weights are read
// once per call however many tokens chose it; CTAs whose rank exceeds the number of distinct experts exit
// at once.
// Lane mapping inside a warp is the mat-vec path's: lane = 32-weight chunk, and when nb32 = K/32 < 32
// divides 32 the warp takes 32/nb32 rows at a time (K = 512 -> 2 rows, K = 256 -> 4); K = 768 (nb32 = 24)
// keeps the plain mapping (the pages' fallback).
#include <cuda_runtime.h>

#include "../../include/qmm.h"
#include "qmm_common.cuh"

namespace wqk {
namespace mvid {

constexpr int WARPS = 8;
constexpr int ROWS_PER_CTA = 64;
constexpr int TOKG = 8;   // tokens per accumulator group

struct Experts {
    const uint8_t *p[QMM_MAX_EXPERTS];
};

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

template <int QT, bool XBF16>
__global__ void __launch_bounds__(WARPS * 32)
    mvid_kernel(const __grid_constant__ Experts ex, int E, int64_t N, int64_t K, int64_t rowbytes,
                const void *__restrict__ x, int xdiv, const int32_t *__restrict__ ids, int M, int topk,
                float *__restrict__ y, int split, unsigned int *status) {
    __shared__ int s_ids[QMM_MAX_ID_SLOTS];
    __shared__ int s_slots[QMM_MAX_ID_SLOTS];   // slots routed to this CTA's expert, ascending
    __shared__ int s_rank[QMM_MAX_EXPERTS];
    __shared__ unsigned char s_used[QMM_MAX_EXPERTS];
    __shared__ int s_nexp, s_expert, s_nslots;

    const int tid = threadIdx.x;
    const int nslot = M * topk;
    for (int i = tid; i < QMM_MAX_EXPERTS; i += blockDim.x) s_used[i] = 0;
    __syncthreads();
    for (int i = tid; i < nslot; i += blockDim.x) {
        const int e = ids[i];
        s_ids[i] = e;
        if (e >= 0 && e < E) s_used[e] = 1;
    }
    __syncthreads();
    if (tid < 32) {
        // ranks of used experts in ascending expert order (E <= 256: 8 ballots)
        int base = 0;
        for (int w0 = 0; w0 < QMM_MAX_EXPERTS; w0 += 32) {
            const bool u = s_used[w0 + tid] != 0;
            const unsigned b = __ballot_sync(0xffffffffu, u);
            s_rank[w0 + tid] = u ? base + __popc(b & ((1u << tid) - 1u)) : -1;
            base += __popc(b);
        }
        if (tid == 0) s_nexp = base;
    }
    __syncthreads();
    const int u = blockIdx.y;
    const int64_t r0 = (int64_t)blockIdx.x * ROWS_PER_CTA;

    if (u == 0) {
        // slots with an id outside [0, E): NaN rows and a status bit (one CTA column does it)
        bool bad = false;
        for (int p = 0; p < nslot; ++p) {
            const int e = s_ids[p];
            if (e < 0 || e >= E) {
                bad = true;
                for (int64_t n = r0 + tid; n < r0 + ROWS_PER_CTA && n < N; n += blockDim.x)
                    y[(int64_t)p * N + n] = __int_as_float(0x7fc00000);
            }
        }
        if (bad && tid == 0 && blockIdx.x == 0) atomicOr(status, kStatusBadId);
    }
    if (u >= s_nexp) return;
    if (tid < QMM_MAX_EXPERTS && s_rank[tid] == u) s_expert = tid;
    __syncthreads();
    const int e = s_expert;
    if (tid == 0) {
        int c = 0;
        for (int p = 0; p < nslot; ++p)
            if (s_ids[p] == e) s_slots[c++] = p;
        s_nslots = c;
    }
    __syncthreads();
    const int ns = s_nslots;
    const uint8_t *wbase = ex.p[e];

    const int lane = tid & 31, warp = tid >> 5;
    const int L = 32 / split;
    const int sub = lane / L, cl = lane % L;
    const int nchunks = (int)(K / 32);
    const int rows_here = (int)((N - r0) < ROWS_PER_CTA ? (N - r0) : ROWS_PER_CTA);
    const int groups = (rows_here + split - 1) / split;

    for (int g = warp; g < groups; g += WARPS) {
        const int64_t n = r0 + (int64_t)g * split + sub;
        const bool valid = (g * split + sub) < rows_here;
        const uint8_t *row = wbase + (valid ? n : 0) * rowbytes;
        for (int t0 = 0; t0 < ns; t0 += TOKG) {
            float acc[TOKG];
#pragma unroll
            for (int j = 0; j < TOKG; ++j) acc[j] = 0.0f;
            if (valid) {
                for (int c = cl; c < nchunks; c += L) {
                    float w[32];
                    decode_chunk<QT>(row, c, K, w);
#pragma unroll
                    for (int j = 0; j < TOKG; ++j) {
                        if (t0 + j < ns) {
                            const int tok = s_slots[t0 + j] / xdiv;   // the token's row, or the slot's
                            float xv[32];
                            load_x32<XBF16>(x, (int64_t)tok * K + 32 * (int64_t)c, xv);
                            float s = acc[j];
#pragma unroll
                            for (int l = 0; l < 32; ++l) s = fmaf(w[l], xv[l], s);
                            acc[j] = s;
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < TOKG; ++j) {
                float v = acc[j];
                for (int off = L >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                acc[j] = v;
            }
            if (valid && cl == 0) {
#pragma unroll
                for (int j = 0; j < TOKG; ++j)
                    if (t0 + j < ns) y[(int64_t)s_slots[t0 + j] * N + n] = acc[j];
            }
        }
    }
}

}  // namespace mvid

namespace {
struct MvidLaunch {
    bool xbf16;
    const mvid::Experts *ex;
    int E;
    int64_t N, K;
    const void *x;
    int xdiv;
    const int32_t *ids;
    int M, topk;
    float *y;
    int split;
    dim3 grid;
    unsigned int *status;
    cudaStream_t st;
    template <int QT> int operator()() {
        const int64_t rb = row_bytes(QT, K);
        if (xbf16)
            mvid::mvid_kernel<QT, true><<<grid, mvid::WARPS * 32, 0, st>>>(*ex, E, N, K, rb, x, xdiv, ids, M, topk,
                                                                          y, split, status);
        else
            mvid::mvid_kernel<QT, false><<<grid, mvid::WARPS * 32, 0, st>>>(*ex, E, N, K, rb, x, xdiv, ids, M,
                                                                           topk, y, split, status);
        return cudaGetLastError() == cudaSuccess ? 0 : -6;
    }
};
}  // namespace

int launch_mvid(int qt, bool xbf16, const void *const *wq, int64_t E, int64_t N, int64_t K, const void *x,
                bool x_per_slot, const int32_t *ids, int64_t M, int topk, float *y, unsigned int *status,
                cudaStream_t st) {
    mvid::Experts ex;
    for (int e = 0; e < QMM_MAX_EXPERTS; ++e) ex.p[e] = e < E ? static_cast<const uint8_t *>(wq[e]) : nullptr;
    const int64_t nb32 = K / 32;
    const int split = (nb32 < 32 && nb32 > 0 && (32 % nb32) == 0) ? (int)(32 / nb32) : 1;
    const int64_t slots = M * topk;
    const int64_t maxexp = slots < E ? slots : E;
    dim3 grid((unsigned)((N + mvid::ROWS_PER_CTA - 1) / mvid::ROWS_PER_CTA), (unsigned)maxexp);
    MvidLaunch f{xbf16, &ex, (int)E, N, K, x, x_per_slot ? 1 : topk, ids, (int)M, topk, y, split, grid, status, st};
    return dispatch_type(qt, f);
}

}  // namespace wqk

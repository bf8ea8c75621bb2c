// Stand-alone dequantization (blocks -> binary32) and the device encoder (binary32 -> blocks).
//
// Dequantization uses the same per-format chunk decoders as the matmul kernels, so a bit-exact match
// with the CPU oracle here pins the decoders the matmul paths run.
//
// The encoder is the block-format specification's deterministic round-to-nearest encoder: every decision
// is taken in binary32 with IEEE operations (correctly rounded division, no contraction), so that it agrees
// bit for bit with any other implementation of the same rules. It is not on the matmul path; it gives
// users (and the benchmark) a way to produce weights on the device.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qmm_common.cuh"

namespace wqk {
namespace deq {

template <int QT>
__global__ void dequant_kernel(const uint8_t *__restrict__ wq, int64_t N, int64_t K, int64_t rowbytes,
                               float *__restrict__ out) {
    const int64_t nchunks = (K + 31) / 32;
    const int64_t total = N * nchunks;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = t / nchunks;
        const int c = (int)(t % nchunks);
        float w[32];
        decode_chunk<QT>(wq + n * rowbytes, c, K, w);
        float *o = out + n * K + 32 * (int64_t)c;
        if constexpr (QT == T_F32) {
            // keep the stored bits (NaN payloads included)
            const uint32_t *src = reinterpret_cast<const uint32_t *>(wq + n * rowbytes);
            for (int l = 0; l < 32 && 32 * (int64_t)c + l < K; ++l)
                reinterpret_cast<uint32_t *>(o)[l] = src[32 * (int64_t)c + l];
        } else if (QT <= T_BF16) {
            for (int l = 0; l < 32 && 32 * (int64_t)c + l < K; ++l) o[l] = w[l];
        } else {
            float4 *o4 = reinterpret_cast<float4 *>(o);
#pragma unroll
            for (int i = 0; i < 8; ++i) o4[i] = make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
    }
}

// ------------------------------------------------------------------------------------------ encoder
__device__ __forceinline__ int rne_clamp(float t, float a, float b) {
    return (int)rintf(fminf(fmaxf(t, a), b));
}
__device__ __forceinline__ uint32_t f16_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }
__device__ __forceinline__ uint32_t bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// amax, min, max of n weights, scanned in order with strict comparisons (first occurrence wins).
__device__ __forceinline__ void stats(const float *w, int n, float &amax, float &lo, float &hi) {
    float am = 0.0f, l = w[0], h = w[0];
    for (int i = 0; i < n; ++i) {
        const float a = fabsf(w[i]);
        if (a > am) am = a;
        if (w[i] < l) l = w[i];
        if (w[i] > h) h = w[i];
    }
    amax = am; lo = l; hi = h;
}

__device__ __forceinline__ void put16(uint8_t *b, int off, uint32_t v) {
    b[off] = (uint8_t)(v & 255u);
    b[off + 1] = (uint8_t)(v >> 8);
}
__device__ __forceinline__ void put_bits(uint8_t *b, int off, int pos, int width, uint32_t v) {
    for (int t = 0; t < width; ++t) {
        const int p = pos + t;
        const uint8_t bit = (uint8_t)(1u << (p & 7));
        if ((v >> t) & 1u) b[off + (p >> 3)] |= bit;
        else b[off + (p >> 3)] &= (uint8_t)~bit;
    }
}

// Encode one block (QK weights at w) into b (BYTES, written in full).
template <int QT>
__device__ void encode_block(const float *w, uint8_t *b) {
    constexpr int BYTES = TypeInfo<QT>::BYTES;
    for (int i = 0; i < BYTES; ++i) b[i] = 0;
    if constexpr (QT == T_F32) {
        const uint32_t u = __float_as_uint(w[0]);
        for (int i = 0; i < 4; ++i) b[i] = (uint8_t)(u >> (8 * i));
    } else if constexpr (QT == T_F16) {
        put16(b, 0, f16_bits(w[0]));
    } else if constexpr (QT == T_BF16) {
        put16(b, 0, bf16_bits(w[0]));
    } else if constexpr (QT == T_Q4_0 || QT == T_Q5_0 || QT == T_Q8_0) {
        float amax, lo, hi;
        stats(w, 32, amax, lo, hi);
        const float top = QT == T_Q4_0 ? 7.0f : (QT == T_Q5_0 ? 15.0f : 127.0f);
        const float bot = QT == T_Q4_0 ? -8.0f : (QT == T_Q5_0 ? -16.0f : -127.0f);
        const uint32_t dh = f16_bits(__fdiv_rn(amax, top));
        const float D = h2f(dh);
        put16(b, 0, dh);
        for (int i = 0; i < 32; ++i) {
            const int q = D == 0.0f ? 0 : rne_clamp(__fdiv_rn(w[i], D), bot, top);
            if (QT == T_Q4_0) {
                const uint32_t u = (uint32_t)(q + 8);
                if (i < 16) b[2 + i] |= (uint8_t)u;
                else b[2 + i - 16] |= (uint8_t)(u << 4);
            } else if (QT == T_Q5_0) {
                const uint32_t u = (uint32_t)(q + 16);
                if (i < 16) b[6 + i] |= (uint8_t)(u & 15u);
                else b[6 + i - 16] |= (uint8_t)((u & 15u) << 4);
                if (u >> 4) b[2 + i / 8] |= (uint8_t)(1u << (i % 8));
            } else {
                b[2 + i] = (uint8_t)(int8_t)q;
            }
        }
    } else if constexpr (QT == T_Q4_1 || QT == T_Q5_1) {
        float amax, lo, hi;
        stats(w, 32, amax, lo, hi);
        const float top = QT == T_Q4_1 ? 15.0f : 31.0f;
        const uint32_t dh = f16_bits(__fdiv_rn(__fsub_rn(hi, lo), top)), mh = f16_bits(lo);
        const float D = h2f(dh), Mv = h2f(mh);
        put16(b, 0, dh);
        put16(b, 2, mh);
        for (int i = 0; i < 32; ++i) {
            const uint32_t q = D == 0.0f ? 0u : (uint32_t)rne_clamp(__fdiv_rn(__fsub_rn(w[i], Mv), D), 0.0f, top);
            const int qo = QT == T_Q4_1 ? 4 : 8;
            if (i < 16) b[qo + i] |= (uint8_t)(q & 15u);
            else b[qo + i - 16] |= (uint8_t)((q & 15u) << 4);
            if (QT == T_Q5_1 && (q >> 4)) b[4 + i / 8] |= (uint8_t)(1u << (i % 8));
        }
    } else if constexpr (QT == T_A4G64) {
        float amax, lo, hi;
        stats(w, 64, amax, lo, hi);
        const uint32_t sh = bf16_bits(__fdiv_rn(__fsub_rn(hi, lo), 15.0f)), bh = bf16_bits(lo);
        const float S = bf2f(sh), B = bf2f(bh);
        put16(b, 0, sh);
        put16(b, 2, bh);
        for (int i = 0; i < 64; ++i) {
            const uint32_t q = S == 0.0f ? 0u : (uint32_t)rne_clamp(__fdiv_rn(__fsub_rn(w[i], B), S), 0.0f, 15.0f);
            if (i < 32) b[4 + i] |= (uint8_t)q;
            else b[4 + i - 32] |= (uint8_t)(q << 4);
        }
    } else if constexpr (QT == T_Q2_K || QT == T_Q4_K || QT == T_Q5_K) {
        constexpr int SUB = QT == T_Q2_K ? 16 : 32, NS = 256 / SUB;
        const float levels = QT == T_Q2_K ? 3.0f : (QT == T_Q4_K ? 15.0f : 31.0f);
        const float smax = QT == T_Q2_K ? 15.0f : 63.0f;
        float r[NS], nn[NS], rmax = 0.0f, nmax = 0.0f;
        for (int s = 0; s < NS; ++s) {
            float amax, lo, hi;
            stats(w + s * SUB, SUB, amax, lo, hi);
            const float l = lo < 0.0f ? lo : 0.0f;
            r[s] = __fdiv_rn(__fsub_rn(hi, l), levels);
            nn[s] = -l;
            if (r[s] > rmax) rmax = r[s];
            if (nn[s] > nmax) nmax = nn[s];
        }
        const uint32_t dh = f16_bits(__fdiv_rn(rmax, smax)), mh = f16_bits(__fdiv_rn(nmax, smax));
        const float D = h2f(dh), Dm = h2f(mh);
        const int doff = QT == T_Q2_K ? 80 : 0;
        put16(b, doff, dh);
        put16(b, doff + 2, mh);
        for (int s = 0; s < NS; ++s) {
            const int sc = D == 0.0f ? 0 : rne_clamp(__fdiv_rn(r[s], D), 0.0f, smax);
            const int mn = Dm == 0.0f ? 0 : rne_clamp(__fdiv_rn(nn[s], Dm), 0.0f, smax);
            if (QT == T_Q2_K) {
                b[s] = (uint8_t)(sc | (mn << 4));
            } else {
                put_bits(b, 4, 6 * s, 6, (uint32_t)sc);
                put_bits(b, 4, 48 + 6 * s, 6, (uint32_t)mn);
            }
            const float S = __fmul_rn(D, (float)sc), Bm = __fmul_rn(Dm, (float)mn);
            for (int t = 0; t < SUB; ++t) {
                const int i = s * SUB + t;
                const uint32_t q =
                    S == 0.0f ? 0u : (uint32_t)rne_clamp(__fdiv_rn(__fadd_rn(w[i], Bm), S), 0.0f, levels);
                if (QT == T_Q2_K) {
                    const int h = i / 128, g = (i % 128) / 32, l = i % 32;
                    b[16 + 32 * h + l] |= (uint8_t)(q << (2 * g));
                } else {
                    const int c = i / 64, l = i % 32, qoff = QT == T_Q4_K ? 16 : 48;
                    if ((i % 64) < 32) b[qoff + 32 * c + l] |= (uint8_t)(q & 15u);
                    else b[qoff + 32 * c + l] |= (uint8_t)((q & 15u) << 4);
                    if (QT == T_Q5_K && (q >> 4)) b[16 + i % 32] |= (uint8_t)(1u << (i / 32));
                }
            }
        }
    } else if constexpr (QT == T_Q3_K || QT == T_Q6_K) {
        const float top = QT == T_Q3_K ? 3.0f : 31.0f, smax = QT == T_Q3_K ? 31.0f : 127.0f;
        const float bot = QT == T_Q3_K ? -4.0f : -32.0f;
        float r[16], rmax = 0.0f;
        for (int s = 0; s < 16; ++s) {
            float amax, lo, hi;
            stats(w + 16 * s, 16, amax, lo, hi);
            r[s] = __fdiv_rn(amax, top);
            if (r[s] > rmax) rmax = r[s];
        }
        const uint32_t dh = f16_bits(__fdiv_rn(rmax, smax));
        const float D = h2f(dh);
        put16(b, QT == T_Q3_K ? 108 : 208, dh);
        for (int s = 0; s < 16; ++s) {
            const int sc = D == 0.0f ? 0 : rne_clamp(__fdiv_rn(r[s], D), 0.0f, smax);
            if (QT == T_Q3_K) put_bits(b, 96, 6 * s, 6, (uint32_t)(sc + 32));
            else b[192 + s] = (uint8_t)(int8_t)sc;
            const float S = __fmul_rn(D, (float)sc);
            for (int t = 0; t < 16; ++t) {
                const int i = 16 * s + t;
                const int q = S == 0.0f ? 0 : rne_clamp(__fdiv_rn(w[i], S), bot, top);
                if (QT == T_Q3_K) {
                    const uint32_t u = (uint32_t)(q + 4);
                    const int h = i / 128, g = (i % 128) / 32, l = i % 32;
                    b[32 + 32 * h + l] |= (uint8_t)((u & 3u) << (2 * g));
                    if (u >> 2) b[i % 32] |= (uint8_t)(1u << (i / 32));
                } else {
                    const uint32_t u = (uint32_t)(q + 32);
                    const int h = i / 128, j = i % 128;
                    b[64 * h + j % 64] |= (uint8_t)((u & 15u) << (4 * (j / 64)));
                    b[128 + 32 * h + j % 32] |= (uint8_t)((u >> 4) << (2 * (j / 32)));
                }
            }
        }
    }
}

// One thread per block: the block's weights are copied to a local array, encoded into a local byte
// buffer, then written out as 16-bit words (every block size is even and every block 2-byte aligned).
template <int QT>
__global__ void quantize_kernel(const float *__restrict__ w, int64_t N, int64_t K, uint8_t *__restrict__ out) {
    constexpr int QK = TypeInfo<QT>::QK, BYTES = TypeInfo<QT>::BYTES;
    const int64_t nb = K / QK;
    const int64_t total = N * nb;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = t / nb, bi = t % nb;
        float wl[QK];
        const float *src = w + n * K + bi * QK;
        for (int i = 0; i < QK; ++i) wl[i] = src[i];
        uint8_t bl[BYTES];
        encode_block<QT>(wl, bl);
        uint16_t *dst = reinterpret_cast<uint16_t *>(out + t * BYTES);
        for (int i = 0; i < BYTES / 2; ++i) dst[i] = (uint16_t)(bl[2 * i] | ((uint32_t)bl[2 * i + 1] << 8));
    }
}

// Plain types: one element per thread, stored in the output's own width.
template <int QT>
__global__ void quantize_plain_kernel(const float *__restrict__ w, int64_t n, uint8_t *__restrict__ out) {
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
        const float v = w[t];
        if constexpr (QT == T_F32) reinterpret_cast<uint32_t *>(out)[t] = __float_as_uint(v);
        else if constexpr (QT == T_F16) reinterpret_cast<uint16_t *>(out)[t] = (uint16_t)f16_bits(v);
        else reinterpret_cast<uint16_t *>(out)[t] = (uint16_t)bf16_bits(v);
    }
}

}  // namespace deq

namespace {
struct DequantLaunch {
    const void *wq;
    int64_t N, K;
    float *out;
    cudaStream_t st;
    template <int QT> int operator()() {
        const int64_t total = N * ((K + 31) / 32);
        int64_t blocks = (total + 255) / 256;
        if (blocks > 152 * 32) blocks = 152 * 32;
        if (blocks < 1) blocks = 1;
        deq::dequant_kernel<QT><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint8_t *>(wq), N, K,
                                                                row_bytes(QT, K), out);
        return cudaGetLastError() == cudaSuccess ? 0 : -6;
    }
};
struct QuantizeLaunch {
    const float *w;
    int64_t N, K;
    void *out;
    cudaStream_t st;
    template <int QT> int operator()() {
        const int64_t total = N * (K / TypeInfo<QT>::QK);
        const int threads = 128;
        int64_t blocks = (total + threads - 1) / threads;
        if (blocks > 152 * 64) blocks = 152 * 64;
        if (blocks < 1) blocks = 1;
        if constexpr (QT <= T_BF16)
            deq::quantize_plain_kernel<QT><<<(unsigned)blocks, threads, 0, st>>>(w, N * K, static_cast<uint8_t *>(out));
        else
            deq::quantize_kernel<QT><<<(unsigned)blocks, threads, 0, st>>>(w, N, K, static_cast<uint8_t *>(out));
        return cudaGetLastError() == cudaSuccess ? 0 : -6;
    }
};
}  // namespace

int launch_dequant(int qt, const void *wq, int64_t N, int64_t K, float *out, cudaStream_t st) {
    DequantLaunch f{wq, N, K, out, st};
    return dispatch_type(qt, f);
}

int launch_quantize(int qt, const float *w, int64_t N, int64_t K, void *out, cudaStream_t st) {
    QuantizeLaunch f{w, N, K, out, st};
    return dispatch_type(qt, f);
}

}  // namespace wqk

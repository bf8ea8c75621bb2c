// Shared device-side definitions of libqmm: the weight-type table and the per-format decoders.
//
// Every decoder turns 32 consecutive weights of a row (a "chunk", the pages' 32-element lane unit,
// llama.cpp PR 28086, section "Overview": nb32 = K/32 chunks per row) into binary32 values equal to the
// exact value of the type's formula rounded once to nearest-even. Every product in the formulas is exact
// in binary32 (at most 24 significant bits), so a product followed by one fused multiply-add or one add
// gives exactly that rounding.
//
// Block layouts (little-endian; element i of a block is weight b*QK + i of its row):
//   Q4_0  18 B: d f16 @0; qs[16] @2, element j<16 = qs[j] & 15, element j+16 = qs[j] >> 4;  w = d(q-8)
//   Q4_1  20 B: d f16 @0; m f16 @2; qs[16] @4 as Q4_0;                                      w = d q + m
//   Q5_0  22 B: d @0; qh u32 @2 (bit i = high bit of element i); qs[16] @6;                  w = d(q-16)
//   Q5_1  24 B: d @0; m @2; qh u32 @4; qs[16] @8;                                           w = d q + m
//   Q8_0  34 B: d @0; int8 q[32] @2;                                                         w = d q
//   Q2_K  84 B: scales[16] @0 (low nibble sc, high nibble mn, per 16 weights); qs[64] @16; d @80; dmin @82
//               element i: q = (qs[32(i/128) + i%32] >> 2((i%128)/32)) & 3;            w = d sc q - dmin mn
//   Q3_K 110 B: hmask[32] @0; qs[64] @32; scales: 16 six-bit fields of a 96-bit LE integer @96; d @108
//               q = (2 low bits as Q2_K) + 4 * ((hmask[i%32] >> (i/32)) & 1);          w = d(sc-32)(q-4)
//   Q4_K 144 B: d @0; dmin @2; 96-bit LE scale field @4: sc_s = bits 6s.., mn_s = bits 48+6s.. (s = i/32);
//               qs[128] @16: byte 32(i/64) + i%32, low nibble if i%64 < 32 else high; w = d sc q - dmin mn
//   Q5_K 176 B: as Q4_K, plus qh[32] @16 (high bit (qh[i%32] >> (i/32)) & 1), qs[128] @48
//   Q6_K 210 B: ql[128] @0; qh[64] @128; int8 scales[16] @192 (per 16 weights); d @208. For h = i/128,
//               j = i%128: low = (ql[64h + j%64] >> 4(j/64)) & 15, high = (qh[32h + j%32] >> 2(j/32)) & 3,
//               q = low + 16 high;                                                       w = d sc (q-32)
//   A4G64 36 B: s bf16 @0; b bf16 @2; qs[32] @4, element i<32 low nibble of qs[i], i>=32 high nibble of
//               qs[i-32];                                                                w = s q + b
//   F32 / F16 / BF16: plain row-major values.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wqk {

// ------------------------------------------------------------------------------------------ per-device state
// Kernel attributes and launch-planning caches are kept per device (a process may drive several GPUs).
constexpr int kMaxDevices = 16;
// Index of the current device for those caches (0 when it cannot be queried).
inline int current_device_index() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) d = 0;
    return d;
}
// SMs of the current device (148 when there is no device to ask, e.g. host-only planning).
inline int device_sm_count() {
    static int nsm[kMaxDevices] = {};
    const int d = current_device_index();
    if (!nsm[d]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0) return 152;   // no device: plan for a GB300
        nsm[d] = v;
    }
    return nsm[d];
}

enum : int {
    T_F32 = 0, T_F16 = 1, T_BF16 = 2, T_Q4_0 = 3, T_Q4_1 = 4, T_Q5_0 = 5, T_Q5_1 = 6, T_Q8_0 = 7,
    T_Q2_K = 8, T_Q3_K = 9, T_Q4_K = 10, T_Q5_K = 11, T_Q6_K = 12, T_A4G64 = 13, T_COUNT = 14
};

template <int QT> struct TypeInfo;
#define QMM_TYPEINFO(T, QK_, BYTES_) \
    template <> struct TypeInfo<T> { static constexpr int QK = QK_; static constexpr int BYTES = BYTES_; };
QMM_TYPEINFO(T_F32, 1, 4)
QMM_TYPEINFO(T_F16, 1, 2)
QMM_TYPEINFO(T_BF16, 1, 2)
QMM_TYPEINFO(T_Q4_0, 32, 18)
QMM_TYPEINFO(T_Q4_1, 32, 20)
QMM_TYPEINFO(T_Q5_0, 32, 22)
QMM_TYPEINFO(T_Q5_1, 32, 24)
QMM_TYPEINFO(T_Q8_0, 32, 34)
QMM_TYPEINFO(T_Q2_K, 256, 84)
QMM_TYPEINFO(T_Q3_K, 256, 110)
QMM_TYPEINFO(T_Q4_K, 256, 144)
QMM_TYPEINFO(T_Q5_K, 256, 176)
QMM_TYPEINFO(T_Q6_K, 256, 210)
QMM_TYPEINFO(T_A4G64, 64, 36)
#undef QMM_TYPEINFO

// Host-side table (same numbers).
static constexpr int kQK[T_COUNT] = {1, 1, 1, 32, 32, 32, 32, 32, 256, 256, 256, 256, 256, 64};
static constexpr int kBytes[T_COUNT] = {4, 2, 2, 18, 20, 22, 24, 34, 84, 110, 144, 176, 210, 36};

__host__ __device__ constexpr bool is_plain(int qt) { return qt <= T_BF16; }

// Kernels that can fail at run time (a bad expert id, a bounded wait that gave up) OR a bit into a
// device status word whose address the host passes in; qmm_get_status() reads and clears it.
constexpr unsigned int kStatusBadId = 0x1u;
constexpr unsigned int kStatusTimeout = 0x2u;

// ------------------------------------------------------------------------------------------ loads
__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }
__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint4 ld_u128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }
// Four bytes at a 2-byte aligned address.
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t *p) { return ld_u16(p) | (ld_u16(p + 2) << 16); }

__device__ __forceinline__ float h2f(uint32_t bits) { return __half2float(__ushort_as_half((unsigned short)bits)); }
// Exact integer -> binary32 for small magnitudes through the 2^23 (resp. 1.5 * 2^23) bias trick, which
// runs on the full-rate ALU/FMA pipes instead of the conversion unit.
__device__ __forceinline__ float u2f_small(uint32_t v) { return __int_as_float(0x4B000000 | v) - 8388608.0f; }  // v < 2^23
__device__ __forceinline__ float i2f_small(int v) { return __int_as_float(0x4B400000 + v) - 12582912.0f; }    // |v| < 2^22
__device__ __forceinline__ float bf2f(uint32_t bits) { return __uint_as_float(bits << 16); }

// Load 32 consecutive bytes starting at a 2-byte aligned address into 8 words.
__device__ __forceinline__ void ld32_a2(const uint8_t *p, uint32_t (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = ld_u32_a2(p + 4 * i);
}
__device__ __forceinline__ void ld32_a4(const uint8_t *p, uint32_t (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = ld_u32(p + 4 * i);
}
__device__ __forceinline__ void ld32_a16(const uint8_t *p, uint32_t (&v)[8]) {
    uint4 a = ld_u128(p), b = ld_u128(p + 16);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// 16 bytes at a 2-byte aligned address.
__device__ __forceinline__ void ld16_a2(const uint8_t *p, uint32_t (&v)[4]) {
#pragma unroll
    for (int i = 0; i < 4; i++) v[i] = ld_u32_a2(p + 4 * i);
}

// Byte e (0..31) of 32 bytes held in 8 words.
__device__ __forceinline__ uint32_t byte_of(const uint32_t (&v)[8], int e) { return (v[e >> 2] >> (8 * (e & 3))) & 255u; }
__device__ __forceinline__ uint32_t byte16(const uint32_t (&v)[4], int e) { return (v[e >> 2] >> (8 * (e & 3))) & 255u; }

// Six-bit field number f of a 96-bit little-endian integer held in three words.
__device__ __forceinline__ uint32_t six_bits(uint32_t s0, uint32_t s1, uint32_t s2, int f) {
    const int pos = 6 * f;
    const uint64_t lo = ((uint64_t)s1 << 32) | s0;
    const uint64_t hi = ((uint64_t)s2 << 32) | s1;
    return (uint32_t)((pos < 58 ? (lo >> pos) : (hi >> (pos - 32))) & 63u);
}

// ------------------------------------------------------------------------------------------ decoders
// decode_chunk<QT>(row, c, w): weights 32c .. 32c+31 of the row starting at `row` (the row's first block)
// into w[0..31]. `row` is 2-byte aligned at least; types whose block size is a multiple of 4 or 16 bytes
// use wider loads, which the row alignment then guarantees (rows start at multiples of the row stride
// from a 16-byte aligned base).
template <int QT> struct Dec;

template <> struct Dec<T_Q4_0> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 18 * c;
        const float d = h2f(ld_u16(b));
        uint32_t q[4];
        ld16_a2(b + 2, q);
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const uint32_t v = byte16(q, j);
            w[j] = __fmul_rn(d, i2f_small((int)(v & 15u) - 8));
            w[j + 16] = __fmul_rn(d, i2f_small((int)(v >> 4) - 8));
        }
    }
};

template <> struct Dec<T_Q4_1> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 20 * c;
        const uint32_t dm = ld_u32(b);
        const float d = h2f(dm & 0xffffu), m = h2f(dm >> 16);
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; i++) q[i] = ld_u32(b + 4 + 4 * i);
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const uint32_t v = byte16(q, j);
            w[j] = __fmaf_rn(d, (float)(v & 15u), m);
            w[j + 16] = __fmaf_rn(d, (float)(v >> 4), m);
        }
    }
};

template <> struct Dec<T_Q5_0> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 22 * c;
        const float d = h2f(ld_u16(b));
        const uint32_t qh = ld_u32_a2(b + 2);
        uint32_t q[4];
        ld16_a2(b + 6, q);
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const uint32_t v = byte16(q, j);
            const int lo = (int)((v & 15u) | (((qh >> j) & 1u) << 4));
            const int hi = (int)((v >> 4) | (((qh >> (j + 16)) & 1u) << 4));
            w[j] = __fmul_rn(d, (float)(lo - 16));
            w[j + 16] = __fmul_rn(d, (float)(hi - 16));
        }
    }
};

template <> struct Dec<T_Q5_1> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 24 * c;
        const uint32_t dm = ld_u32(b);
        const float d = h2f(dm & 0xffffu), m = h2f(dm >> 16);
        const uint32_t qh = ld_u32(b + 4);
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; i++) q[i] = ld_u32(b + 8 + 4 * i);
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const uint32_t v = byte16(q, j);
            const uint32_t lo = (v & 15u) | (((qh >> j) & 1u) << 4);
            const uint32_t hi = (v >> 4) | (((qh >> (j + 16)) & 1u) << 4);
            w[j] = __fmaf_rn(d, (float)lo, m);
            w[j + 16] = __fmaf_rn(d, (float)hi, m);
        }
    }
};

template <> struct Dec<T_Q8_0> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 34 * c;
        const float d = h2f(ld_u16(b));
        uint32_t q[8];
        ld32_a2(b + 2, q);
#pragma unroll
        for (int i = 0; i < 32; i++) w[i] = __fmul_rn(d, (float)(int8_t)byte_of(q, i));
    }
};

template <> struct Dec<T_Q2_K> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 84 * (c >> 3);
        const int t = c & 7, h = t >> 2, g = t & 3;
        const uint32_t dd = ld_u32(b + 80);
        const float d = h2f(dd & 0xffffu), dmin = h2f(dd >> 16);
        const uint32_t sm = ld_u16(b + 2 * t);   // scales[2t], scales[2t+1]
        uint32_t q[8];
        ld32_a4(b + 16 + 32 * h, q);
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const uint32_t s = (sm >> (8 * half)) & 255u;
            const float ds = __fmul_rn(d, (float)(s & 15u));
            const float dm = __fmul_rn(dmin, (float)(s >> 4));
#pragma unroll
            for (int l = 0; l < 16; l++) {
                const uint32_t v = (byte_of(q, 16 * half + l) >> (2 * g)) & 3u;
                w[16 * half + l] = __fmaf_rn(ds, (float)v, -dm);
            }
        }
    }
};

template <> struct Dec<T_Q3_K> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 110 * (c >> 3);
        const int t = c & 7, h = t >> 2, g = t & 3;
        const float d = h2f(ld_u16(b + 108));
        uint32_t hm[8], q[8];
        ld32_a2(b, hm);
        ld32_a2(b + 32 + 32 * h, q);
        const uint32_t s0 = ld_u32_a2(b + 96), s1 = ld_u32_a2(b + 100), s2 = ld_u32_a2(b + 104);
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const int sc = (int)six_bits(s0, s1, s2, 2 * t + half) - 32;
            const float ds = __fmul_rn(d, (float)sc);
#pragma unroll
            for (int l = 0; l < 16; l++) {
                const int e = 16 * half + l;
                const uint32_t lo = (byte_of(q, e) >> (2 * g)) & 3u;
                const uint32_t hi = (byte_of(hm, e) >> t) & 1u;
                w[e] = __fmul_rn(ds, (float)((int)(lo | (hi << 2)) - 4));
            }
        }
    }
};

template <int QT> struct DecQ45K {
    static constexpr bool A16 = true;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        constexpr int BYTES = TypeInfo<QT>::BYTES;
        const uint8_t *b = row + BYTES * (c >> 3);
        const int t = c & 7;                 // sub-block of 32
        const uint4 hd = ld_u128(b);         // d, dmin, 12 scale bytes
        const float d = h2f(hd.x & 0xffffu), dmin = h2f(hd.x >> 16);
        const uint32_t sc = six_bits(hd.y, hd.z, hd.w, t), mn = six_bits(hd.y, hd.z, hd.w, 8 + t);
        const float ds = __fmul_rn(d, u2f_small(sc)), dm = __fmul_rn(dmin, u2f_small(mn));
        uint32_t q[8];
        ld32_a16(b + (QT == T_Q4_K ? 16 : 48) + 32 * (t >> 1), q);
        const int sh = 4 * (t & 1);
        if (QT == T_Q4_K) {
#pragma unroll
            for (int l = 0; l < 32; l++) w[l] = __fmaf_rn(ds, u2f_small((byte_of(q, l) >> sh) & 15u), -dm);
        } else {
            uint32_t qh[8];
            ld32_a16(b + 16, qh);
#pragma unroll
            for (int l = 0; l < 32; l++) {
                const uint32_t v = ((byte_of(q, l) >> sh) & 15u) | (((byte_of(qh, l) >> t) & 1u) << 4);
                w[l] = __fmaf_rn(ds, u2f_small(v), -dm);
            }
        }
    }
};
template <> struct Dec<T_Q4_K> : DecQ45K<T_Q4_K> {};
template <> struct Dec<T_Q5_K> : DecQ45K<T_Q5_K> {};

template <> struct Dec<T_Q6_K> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 210 * (c >> 3);
        const int t = c & 7, h = t >> 2, u = t & 3;   // elements 128h + 32u + l
        const float d = h2f(ld_u16(b + 208));
        const uint32_t sc2 = ld_u16(b + 192 + 2 * t);
        uint32_t ql[8], qh[8];
        ld32_a2(b + 64 * h + 32 * (u & 1), ql);
        ld32_a2(b + 128 + 32 * h, qh);
        const int shl = 4 * (u >> 1), shh = 2 * u;
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const float ds = __fmul_rn(d, i2f_small((int)(int8_t)((sc2 >> (8 * half)) & 255u)));
#pragma unroll
            for (int l = 0; l < 16; l++) {
                const int e = 16 * half + l;
                const uint32_t v = ((byte_of(ql, e) >> shl) & 15u) | (((byte_of(qh, e) >> shh) & 3u) << 4);
                w[e] = __fmul_rn(ds, i2f_small((int)v - 32));
            }
        }
    }
};

template <> struct Dec<T_A4G64> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk(const uint8_t *row, int c, float (&w)[32]) {
        const uint8_t *b = row + 36 * (c >> 1);
        const int sh = 4 * (c & 1);
        const uint32_t sb = ld_u32(b);
        const float s = bf2f(sb & 0xffffu), bias = bf2f(sb >> 16);
        uint32_t q[8];
        ld32_a4(b + 4, q);
#pragma unroll
        for (int l = 0; l < 32; l++) w[l] = __fmaf_rn(s, u2f_small((byte_of(q, l) >> sh) & 15u), bias);
    }
};

// Plain types: chunk c holds elements 32c .. 32c+31 of the row; elements at or past K read as zero.
template <> struct Dec<T_F32> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk_k(const uint8_t *row, int c, int64_t K, float (&w)[32]) {
        const float *r = reinterpret_cast<const float *>(row);
#pragma unroll
        for (int l = 0; l < 32; l++) {
            const int64_t k = 32 * (int64_t)c + l;
            w[l] = k < K ? r[k] : 0.0f;
        }
    }
};
template <> struct Dec<T_F16> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk_k(const uint8_t *row, int c, int64_t K, float (&w)[32]) {
        const uint16_t *r = reinterpret_cast<const uint16_t *>(row);
#pragma unroll
        for (int l = 0; l < 32; l++) {
            const int64_t k = 32 * (int64_t)c + l;
            w[l] = k < K ? h2f(r[k]) : 0.0f;
        }
    }
};
template <> struct Dec<T_BF16> {
    static constexpr bool A16 = false;
    __device__ __forceinline__ static void chunk_k(const uint8_t *row, int c, int64_t K, float (&w)[32]) {
        const uint16_t *r = reinterpret_cast<const uint16_t *>(row);
#pragma unroll
        for (int l = 0; l < 32; l++) {
            const int64_t k = 32 * (int64_t)c + l;
            w[l] = k < K ? bf2f(r[k]) : 0.0f;
        }
    }
};

// One entry point for all types: chunk c of a row with K columns (K only matters for the plain types).
template <int QT>
__device__ __forceinline__ void decode_chunk(const uint8_t *row, int c, int64_t K, float (&w)[32]) {
    if constexpr (QT <= T_BF16) Dec<QT>::chunk_k(row, c, K, w);
    else Dec<QT>::chunk(row, c, w);
}

// Row stride in bytes of an N x K matrix of type qt.
__host__ __device__ __forceinline__ int64_t row_bytes(int qt, int64_t K) {
    constexpr int qk[T_COUNT] = {1, 1, 1, 32, 32, 32, 32, 32, 256, 256, 256, 256, 256, 64};
    constexpr int nb[T_COUNT] = {4, 2, 2, 18, 20, 22, 24, 34, 84, 110, 144, 176, 210, 36};
    return (K / qk[qt]) * nb[qt];
}

// Host-side list of weight matrices of one type and K that share their activations (one mat-vec launch
// serves them all); count = 1 for a single matrix.
constexpr int kMaxBatch = 8;
struct MatSet {
    int count;
    const void *wq[kMaxBatch];
    int64_t N[kMaxBatch];
    float *y[kMaxBatch];
};

// Dispatch a functor templated on the weight type.
template <typename F>
inline int dispatch_type(int qt, F &&f) {
    switch (qt) {
    case T_F32: return f.template operator()<T_F32>();
    case T_F16: return f.template operator()<T_F16>();
    case T_BF16: return f.template operator()<T_BF16>();
    case T_Q4_0: return f.template operator()<T_Q4_0>();
    case T_Q4_1: return f.template operator()<T_Q4_1>();
    case T_Q5_0: return f.template operator()<T_Q5_0>();
    case T_Q5_1: return f.template operator()<T_Q5_1>();
    case T_Q8_0: return f.template operator()<T_Q8_0>();
    case T_Q2_K: return f.template operator()<T_Q2_K>();
    case T_Q3_K: return f.template operator()<T_Q3_K>();
    case T_Q4_K: return f.template operator()<T_Q4_K>();
    case T_Q5_K: return f.template operator()<T_Q5_K>();
    case T_Q6_K: return f.template operator()<T_Q6_K>();
    case T_A4G64: return f.template operator()<T_A4G64>();
    default: return -1;
    }
}

}  // namespace wqk

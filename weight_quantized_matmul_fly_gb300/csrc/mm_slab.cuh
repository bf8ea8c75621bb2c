// Device-side building blocks shared by the tensor-core kernels (the dense one in k_mm.cu and the
// expert-indexed one in k_mm_id.cu): tile constants, shared-memory sizing, the 128-byte swizzle of the
// operand tiles and the per-format slab decoders that turn 32 quantized weights into bf16 pairs.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "qmm_common.cuh"

namespace wqk {
namespace mm {

constexpr int BM = 128;            // weight rows per CTA
constexpr int BK = 64;             // columns per K step: one 128-byte swizzle row of bf16
constexpr int MAX_STAGES = 8;
constexpr int PF = 2;              // K steps of its own group a decoder warp keeps in flight (raw bytes in registers)
// ... per weight type: one for F32, whose 32-weight chunk is 128 bytes
template <int QT> __host__ __device__ constexpr int pf_of() { return QT == T_F32 ? 1 : PF; }
constexpr int A_STAGE = BM * BK * 2;   // 16 KB
constexpr int NDEC = 16;               // decoder / epilogue warps: two groups of 8 taking alternate K steps
constexpr int NGRP = NDEC / 8;         // decoder groups (one slab = 8 warps x 16 rows)
constexpr int THREADS = 32 * (2 + NDEC);

constexpr int MAX_XSLOTS = 6;
constexpr int MAX_SPLIT = 8;       // K splits of one output tile: CTAs of one (portable-size) cluster

__host__ __device__ constexpr int b_stage_bytes(int TN) { return TN * BK * 2; }
__host__ __device__ constexpr int x_slot_bytes(int TN) { return TN * BK * 4; }   // binary32 staging of a K step
// Operand stages: four up to 256 token columns per CTA, two at 512 (80 KB each; there one K step of MMAs
// takes about as long as decoding the step's weights). More stages measured no faster, and the shared memory
// they take comes out of the L1 cache the decoders' weight loads go through. With binary32 activations
// converted in the kernel, staging slots for them take part of the room.
__host__ __device__ constexpr int stages_of(int TN, bool xf32) {
    return xf32 ? (TN > 96 ? 3 : (TN > 32 ? 4 : 8)) : (TN > 256 ? 2 : 4);
}
__host__ __device__ constexpr int xslots_of(int TN, bool xf32) { return xf32 ? (TN > 64 ? 3 : (TN > 32 ? 6 : 4)) : 0; }
__host__ __device__ constexpr int smem_bytes(int TN, bool xf32) {
    return 1024 /* alignment slack */ + stages_of(TN, xf32) * (A_STAGE + b_stage_bytes(TN)) +
           xslots_of(TN, xf32) * x_slot_bytes(TN) + 256 /* barriers */;
}

// Epilogue: which of the NDEC/4 column parts decoder warp `warp` drains (its lane quarter is warp & 3).
__device__ __forceinline__ int part_of(int warp) { return (warp - 2) >> 2; }

// Byte offset of the 16-byte piece p (bf16 columns 8p .. 8p+7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int p) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((p ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------------------------------------------------------ slab decoders
// A decoder lane turns 32 consecutive weights of one row (chunk c) into 16 bf16x2 words, each the bf16
// rounding (nearest even) of the binary32 dequantized weight. Raw bytes are loaded two K steps ahead.
// One byte-permute and one multiply-add per weight: the permute puts code byte j (< 128) under exponent
// byte 0x43, which reads as exactly 128 + q, and the weight ds*q + off is computed as
// ds*(128 + q) + (off - 128*ds) with the second term formed once per chunk. Where off - 128*ds is exact
// (the types without an additive term: -(128 + bias)*ds needs at most 21 significant bits) the result is
// the binary32 weight bit for bit; with an additive term (Q4_K, Q5_K, A4G64) that term is rounded once,
// an absolute error of at most 2^-17 * ds before the bf16 rounding.
__device__ __forceinline__ float code128(uint32_t v4, int j) {   // 128 + byte j of v4, exact for bytes < 128
    return __int_as_float(__byte_perm(v4, 0x43u, 0x4055u | ((uint32_t)j << 8)));
}
// the four codes of v4 -> bf16x2 (lo: codes 0, 1; hi: codes 2, 3) of s * (128 + q) + c
__device__ __forceinline__ void fma4_pack(uint32_t v4, float s, float c, uint32_t &lo, uint32_t &hi) {
    lo = pack_bf16x2(__fmaf_rn(s, code128(v4, 0), c), __fmaf_rn(s, code128(v4, 1), c));
    hi = pack_bf16x2(__fmaf_rn(s, code128(v4, 2), c), __fmaf_rn(s, code128(v4, 3), c));
}

template <int QT> struct Slab {
    static constexpr bool FAST = false;
    struct Raw { int dummy; };
};

// Q4_K / Q5_K: chunk t of a 256-weight super-block = sub-block t; its 32 codes are the low (t even) or
// high (t odd) nibbles of qs[32*(t/2) .. +31], with the fifth bit of Q5_K in bit t of qh[0..31].
template <int QT> struct SlabQ45K {
    static constexpr bool FAST = true;
    struct Raw { uint4 hd, q0, q1, h0, h1; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        constexpr int BY = QT == T_Q4_K ? 144 : 176, QOFF = QT == T_Q4_K ? 16 : 48;
        const uint8_t *b = row + BY * (c >> 3);
        const int t = c & 7;
        r.hd = ld_u128(b);
        r.q0 = ld_u128(b + QOFF + 32 * (t >> 1));
        r.q1 = ld_u128(b + QOFF + 32 * (t >> 1) + 16);
        if (QT == T_Q5_K) { r.h0 = ld_u128(b + 16); r.h1 = ld_u128(b + 32); }
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        const int t = c & 7, sh = 4 * (t & 1);
        const float d = h2f(r.hd.x & 0xffffu), dmin = h2f(r.hd.x >> 16);
        const float ds = __fmul_rn(d, u2f_small(six_bits(r.hd.y, r.hd.z, r.hd.w, t)));
        const float dm = __fmaf_rn(-128.0f, ds, -__fmul_rn(dmin, u2f_small(six_bits(r.hd.y, r.hd.z, r.hd.w, 8 + t))));
        const uint32_t q[8] = {r.q0.x, r.q0.y, r.q0.z, r.q0.w, r.q1.x, r.q1.y, r.q1.z, r.q1.w};
        const uint32_t hh[8] = {r.h0.x, r.h0.y, r.h0.z, r.h0.w, r.h1.x, r.h1.y, r.h1.z, r.h1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t v = (q[i] >> sh) & 0x0F0F0F0Fu;
            if (QT == T_Q5_K) v |= ((hh[i] >> t) & 0x01010101u) << 4;
            fma4_pack(v, ds, dm, o[2 * i], o[2 * i + 1]);
        }
    }
};
template <> struct Slab<T_Q4_K> : SlabQ45K<T_Q4_K> {};
template <> struct Slab<T_Q5_K> : SlabQ45K<T_Q5_K> {};

// Q6_K: chunk t (sub-blocks 2t, 2t+1) takes 32 consecutive ql bytes and 32 consecutive qh bytes. A block
// (210 bytes) starts 4-byte aligned or 2 bytes past it: in the second case each 4-byte word is rebuilt
// from the two aligned words around it.
template <> struct Slab<T_Q6_K> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t ql[9], qh[9]; uint32_t sc; uint32_t d; uint32_t a2; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 210 * (c >> 3);
        const int t = c & 7, h = t >> 2, u = t & 3;
        const uint8_t *pl = b + 64 * h + 32 * (u & 1), *ph = b + 128 + 32 * h;
        r.a2 = (reinterpret_cast<uintptr_t>(b) & 3u) != 0;
        if (!r.a2) {
#pragma unroll
            for (int i = 0; i < 8; ++i) { r.ql[i] = ld_u32(pl + 4 * i); r.qh[i] = ld_u32(ph + 4 * i); }
        } else {
#pragma unroll
            for (int i = 0; i < 9; ++i) { r.ql[i] = ld_u32(pl - 2 + 4 * i); r.qh[i] = ld_u32(ph - 2 + 4 * i); }
        }
        r.sc = ld_u16(b + 192 + 2 * t);
        r.d = ld_u16(b + 208);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        const int t = c & 7, u = t & 3;
        const int shl = 4 * (u >> 1), shh = 2 * u;
        const float d = h2f(r.d);
        const float ds0 = __fmul_rn(d, i2f_small((int)(int8_t)(r.sc & 255u)));
        const float ds1 = __fmul_rn(d, i2f_small((int)(int8_t)(r.sc >> 8)));
        const float c0 = -160.0f * ds0, c1 = -160.0f * ds1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t wl = r.a2 ? __funnelshift_r(r.ql[i], r.ql[i + 1], 16) : r.ql[i];
            const uint32_t wh = r.a2 ? __funnelshift_r(r.qh[i], r.qh[i + 1], 16) : r.qh[i];
            const uint32_t v = ((wl >> shl) & 0x0F0F0F0Fu) | (((wh >> shh) & 0x03030303u) << 4);
            // (q - 32) * ds = ds * (128 + q) - 160 * ds, the last term exact
            const float s = i < 4 ? ds0 : ds1;
            fma4_pack(v, s, i < 4 ? c0 : c1, o[2 * i], o[2 * i + 1]);
        }
    }
};

// A4G64: chunk c is half of a 64-weight block: low (c even) or high (c odd) nibbles of its 32 code bytes.
template <> struct Slab<T_A4G64> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t sb; uint32_t q[8]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 36 * (c >> 1);
        r.sb = ld_u32(b);
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = ld_u32(b + 4 + 4 * i);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        const int sh = 4 * (c & 1);
        const float s = bf2f(r.sb & 0xffffu), bias = bf2f(r.sb >> 16);
        const float cb = __fmaf_rn(-128.0f, s, bias);
#pragma unroll
        for (int i = 0; i < 8; ++i) fma4_pack((r.q[i] >> sh) & 0x0F0F0F0Fu, s, cb, o[2 * i], o[2 * i + 1]);
    }
};

// Q4_0: chunk c is block c (18 bytes, 2-byte aligned): 16 code bytes, low nibbles first.
template <> struct Slab<T_Q4_0> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t q[4]; uint32_t d; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 18 * c;
        r.d = ld_u16(b);
#pragma unroll
        for (int i = 0; i < 4; ++i) r.q[i] = ld_u16(b + 2 + 4 * i) | (ld_u16(b + 4 + 4 * i) << 16);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
        const float d = h2f(r.d);
        const float cb = -136.0f * d;  // (q - 8) * d = d * (128 + q) - 136 * d, the last term exact
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            fma4_pack(r.q[i] & 0x0F0F0F0Fu, d, cb, o[2 * i], o[2 * i + 1]);
            fma4_pack((r.q[i] >> 4) & 0x0F0F0F0Fu, d, cb, o[8 + 2 * i], o[8 + 2 * i + 1]);
        }
    }
};

// ---- legacy 32-weight blocks and the 16-bit plain types: chunk c is block c (resp. weights 32c .. 32c+31).
// Codes 0..15 of a 4-bit block are the low nibbles of its 16 code bytes, 16..31 the high nibbles; the fifth
// bit of weight j (Q5_0, Q5_1) is bit j of the 32-bit field qh.

// The four bits (f >> 4i) & 15 moved to bit 4 of bytes 0..3.
__device__ __forceinline__ uint32_t fifth_bits(uint32_t f, int i) {
    return ((((f >> (4 * i)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
}
// the four codes of v4 (bytes < 128) -> bf16x2 of d * q + m, each the binary32 fma rounded once (exact
// weights: q is recovered exactly as (128 + q) - 128)
__device__ __forceinline__ void fma4_pack_m(uint32_t v4, float d, float m, uint32_t &lo, uint32_t &hi) {
    lo = pack_bf16x2(__fmaf_rn(d, code128(v4, 0) - 128.0f, m), __fmaf_rn(d, code128(v4, 1) - 128.0f, m));
    hi = pack_bf16x2(__fmaf_rn(d, code128(v4, 2) - 128.0f, m), __fmaf_rn(d, code128(v4, 3) - 128.0f, m));
}

// Q4_1: 20-byte blocks (4-byte aligned): d, m (binary16), 16 code bytes.
template <> struct Slab<T_Q4_1> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t dm; uint32_t q[4]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 20 * c;
        r.dm = ld_u32(b);
#pragma unroll
        for (int i = 0; i < 4; ++i) r.q[i] = ld_u32(b + 4 + 4 * i);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
        const float d = h2f(r.dm & 0xffffu), m = h2f(r.dm >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            fma4_pack_m(r.q[i] & 0x0F0F0F0Fu, d, m, o[2 * i], o[2 * i + 1]);
            fma4_pack_m((r.q[i] >> 4) & 0x0F0F0F0Fu, d, m, o[8 + 2 * i], o[8 + 2 * i + 1]);
        }
    }
};

// Q5_0: 22-byte blocks (2-byte aligned): d, qh (32 bits), 16 code bytes; w = d * (q - 16), exact as
// d * (128 + q) - 144 * d (both terms exact).
template <> struct Slab<T_Q5_0> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t d, qh; uint32_t q[4]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 22 * c;
        r.d = ld_u16(b);
        r.qh = ld_u16(b + 2) | (ld_u16(b + 4) << 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) r.q[i] = ld_u16(b + 6 + 4 * i) | (ld_u16(b + 8 + 4 * i) << 16);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
        const float d = h2f(r.d), cb = -144.0f * d;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            fma4_pack((r.q[i] & 0x0F0F0F0Fu) | fifth_bits(r.qh, i), d, cb, o[2 * i], o[2 * i + 1]);
            fma4_pack(((r.q[i] >> 4) & 0x0F0F0F0Fu) | fifth_bits(r.qh >> 16, i), d, cb, o[8 + 2 * i], o[8 + 2 * i + 1]);
        }
    }
};

// Q5_1: 24-byte blocks (8-byte aligned): d, m, qh, 16 code bytes; w = d * q + m.
template <> struct Slab<T_Q5_1> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t dm, qh; uint32_t q[4]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 24 * c;
        r.dm = ld_u32(b);
        r.qh = ld_u32(b + 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) r.q[i] = ld_u32(b + 8 + 4 * i);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
        const float d = h2f(r.dm & 0xffffu), m = h2f(r.dm >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            fma4_pack_m((r.q[i] & 0x0F0F0F0Fu) | fifth_bits(r.qh, i), d, m, o[2 * i], o[2 * i + 1]);
            fma4_pack_m(((r.q[i] >> 4) & 0x0F0F0F0Fu) | fifth_bits(r.qh >> 16, i), d, m, o[8 + 2 * i], o[8 + 2 * i + 1]);
        }
    }
};

// Q8_0: 34-byte blocks (2-byte aligned): d, 32 signed code bytes; w = d * q, exact as d * u - 128 * d with
// u = q + 128 (the byte with its top bit flipped) read as 2^23 + u and the bias subtracted exactly.
template <> struct Slab<T_Q8_0> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t d; uint32_t q[8]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 34 * c;
        r.d = ld_u16(b);
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = ld_u16(b + 2 + 4 * i) | (ld_u16(b + 4 + 4 * i) << 16);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
        const float d = h2f(r.d), cb = -128.0f * d;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t u = r.q[i] ^ 0x80808080u;
            float w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                w[j] = __fmaf_rn(d, __int_as_float(__byte_perm(u, 0x4B000000u, 0x7650u | (uint32_t)j)) - 8388608.0f, cb);
            o[2 * i] = pack_bf16x2(w[0], w[1]);
            o[2 * i + 1] = pack_bf16x2(w[2], w[3]);
        }
    }
};

// Q2_K: 84-byte super-blocks (4-byte aligned); chunk t (sub-blocks 2t, 2t+1 of 16) takes 2-bit field g = t & 3
// of the 32 code bytes at 16 + 32 * (t >> 2), scale bytes 2t and 2t+1 (low nibble scale, high nibble
// minimum), d and dmin at 80; w = d * sc * q - dmin * mn, computed as fma(ds, q, -dm) (exact, as decoded).
template <> struct Slab<T_Q2_K> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t sm, dd; uint32_t q[8]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 84 * (c >> 3);
        const int t = c & 7;
        r.sm = ld_u16(b + 2 * t);
        r.dd = ld_u32(b + 80);
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = ld_u32(b + 16 + 32 * (t >> 2) + 4 * i);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        const int g = c & 3;
        const float d = h2f(r.dd & 0xffffu), dmin = h2f(r.dd >> 16);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t sc = (r.sm >> (8 * half)) & 255u;
            const float ds = __fmul_rn(d, u2f_small(sc & 15u)), dm = __fmul_rn(dmin, u2f_small(sc >> 4));
#pragma unroll
            for (int i = 4 * half; i < 4 * half + 4; ++i)
                fma4_pack_m((r.q[i] >> (2 * g)) & 0x03030303u, ds, -dm, o[2 * i], o[2 * i + 1]);
        }
    }
};

// Q3_K: 110-byte super-blocks (2-byte aligned): 32 high-bit bytes, 64 low-bit bytes, 12 bytes of 6-bit
// scales, d. Chunk t: low 2-bit field g = t & 3 of the 32 bytes at 32 + 32 * (t >> 2), high bit t of the
// high-bit bytes, scales 2t and 2t+1 (offset 32); w = d * (sc - 32) * (q - 4) = ds * (128 + q) - 132 * ds,
// both terms exact.
template <> struct Slab<T_Q3_K> {
    static constexpr bool FAST = true;
    struct Raw { uint32_t hm[8], q[8]; uint32_t s0, s1, s2, d; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 110 * (c >> 3);
        const int t = c & 7;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            r.hm[i] = ld_u32_a2(b + 4 * i);
            r.q[i] = ld_u32_a2(b + 32 + 32 * (t >> 2) + 4 * i);
        }
        r.s0 = ld_u32_a2(b + 96);
        r.s1 = ld_u32_a2(b + 100);
        r.s2 = ld_u32_a2(b + 104);
        r.d = ld_u16(b + 108);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        const int t = c & 7, g = t & 3;
        const float d = h2f(r.d);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const float ds = __fmul_rn(d, i2f_small((int)six_bits(r.s0, r.s1, r.s2, 2 * t + half) - 32));
            const float cb = -132.0f * ds;
#pragma unroll
            for (int i = 4 * half; i < 4 * half + 4; ++i) {
                const uint32_t v = ((r.q[i] >> (2 * g)) & 0x03030303u) | (((r.hm[i] >> t) & 0x01010101u) << 2);
                fma4_pack(v, ds, cb, o[2 * i], o[2 * i + 1]);
            }
        }
    }
};

// F32 weights: each value rounded to bf16, nearest even (128 bytes per chunk, 16-byte aligned). The raw
// buffer is 32 registers, so this type keeps one K step in flight instead of PF (pf_of).
template <> struct Slab<T_F32> {
    static constexpr bool FAST = true;
    struct Raw { uint4 v[8]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 128 * c;
#pragma unroll
        for (int i = 0; i < 8; ++i) r.v[i] = ld_u128(b + 16 * i);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[2 * i] = pack_bf16x2(__uint_as_float(r.v[i].x), __uint_as_float(r.v[i].y));
            o[2 * i + 1] = pack_bf16x2(__uint_as_float(r.v[i].z), __uint_as_float(r.v[i].w));
        }
    }
};

// BF16 weights: the operand itself (64 bytes per chunk, 16-byte aligned).
template <> struct Slab<T_BF16> {
    static constexpr bool FAST = true;
    struct Raw { uint4 v[4]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 64 * c;
#pragma unroll
        for (int i = 0; i < 4; ++i) r.v[i] = ld_u128(b + 16 * i);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[4 * i] = r.v[i].x; o[4 * i + 1] = r.v[i].y; o[4 * i + 2] = r.v[i].z; o[4 * i + 3] = r.v[i].w;
        }
    }
};

// F16 weights: each binary16 value (exact in binary32) rounded to bf16, nearest even.
template <> struct Slab<T_F16> {
    static constexpr bool FAST = true;
    struct Raw { uint4 v[4]; };
    __device__ static void load(Raw &r, const uint8_t *row, int c) {
        const uint8_t *b = row + 64 * c;
#pragma unroll
        for (int i = 0; i < 4; ++i) r.v[i] = ld_u128(b + 16 * i);
    }
    __device__ static void decode(const Raw &r, int c, uint32_t (&o)[16]) {
        (void)c;
        const uint32_t h[16] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w, r.v[1].x, r.v[1].y, r.v[1].z, r.v[1].w,
                                r.v[2].x, r.v[2].y, r.v[2].z, r.v[2].w, r.v[3].x, r.v[3].y, r.v[3].z, r.v[3].w};
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = pack_bf16x2(h2f(h[j] & 0xffffu), h2f(h[j] >> 16));
    }
};

}  // namespace mm
}  // namespace wqk

// Tensor-core mat-vec path for small token counts (M <= 16) and quantized weight types.
//
// Why tensor cores here. At 4-6 bits per weight the HBM stream delivers about one weight per 2-3 CUDA-core
// issue slots, so a binary32 FMA per weight per token cannot keep up beyond M = 1 or 2. The products are
// instead run on mma.sync (m16n8k16, bf16 in, f32 accumulate) fed from registers:
//   - A = the weights' integer codes (q - bias), which are exact in bf16 (|q| <= 32), 16 rows x 16 k;
//   - B = the activations, 8 columns: for binary32 x each token takes two columns, x_hi = bf16(x) and
//     x_lo = bf16(x - x_hi), so the product keeps ~17 bits of x (residual <= 2^-18 |x|) and the result
//     stays in the binary32 tolerance class; bf16 x is exact and takes one column per token;
//   - each scale unit's sum (16, 32 or 64 weights, which never straddle a k16 group) is scaled in binary32
//     on the CUDA cores: y += ds * sum_k q x + off * sum_k x, with off the type's minimum or bias term.
// tcgen05 is not used on this path: its A operand must come from shared or tensor memory, and writing the
// decoded bf16 codes there costs 4 bytes of on-chip traffic per weight against the 0.56 bytes the weight
// costs in HBM; mma.sync takes A straight from the registers the decoder wrote.
//
// Lane mapping. Lane (g, t) = (lane / 4, lane % 4) of a warp decodes rows g and g + 8 of the warp's 16-row
// group, weights 4t .. 4t+3 of every 16-weight group, which mma.sync sees as logical k {2t, 2t+1, 2t+8,
// 2t+9} (the activations are read with the same permutation). Every lane is busy at any K, which is what
// the pages' narrow-K row split was for (llama.cpp PR 28086, "metal : fix idle threads in mul_mv_iq3_xxs
// for ne00 < 1024", section "Overview"); and tokens are MMA columns, so the kernel is specialised on the
// number of 4- or 8-token column groups (tiny-llm PR 122, "perf: Optimize quantized matmul for small
// decode batches": the x_size buckets become column-group buckets).
//
// Work split. A CTA owns 16 rows per row group and one K segment; the K segments of a row block form a
// thread block cluster. Each CTA stores its partial sums into the shared memory of the cluster's first
// CTA, which adds them in rank order after one cluster barrier (so the result is deterministic and no
// global scratch is needed). The weights reach shared memory through bulk copies issued before the
// kernel waits for its predecessor (programmatic dependent launch), so consecutive launches overlap.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/qmm.h"
#include "ptx.cuh"
#include "qmm_common.cuh"

namespace wqk {
namespace gtc {

// ------------------------------------------------------------------------------------------ helpers
__device__ __forceinline__ uint32_t ldw_a2(const uint8_t *p) { return ld_u16(p) | (ld_u16(p + 2) << 16); }

// bf16x2 (lo, hi) of codes byte0/byte1 (lo pair) or byte2/byte3 (hi pair) minus `bias2` (bf16x2 of 128+bias).
__device__ __forceinline__ uint32_t codes_pair(uint32_t codes, uint32_t sel, uint32_t bias2) {
    const uint32_t m = __byte_perm(codes, 0x43434343u, sel);   // 128 + code, exact
    __nv_bfloat162 v = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&m),
                               *reinterpret_cast<const __nv_bfloat162 *>(&bias2));
    return *reinterpret_cast<uint32_t *>(&v);
}
constexpr uint32_t SEL_LO = 0x5140u, SEL_HI = 0x7362u;
__host__ __device__ constexpr uint32_t bias_bf16x2(int bias) {
    // bf16 of 128 + bias for bias in [0, 32]: exponent 2^7, mantissa bias
    return (uint32_t)(0x4300u | (uint32_t)bias) * 0x10001u;
}

// Signed int8 codes (Q8_0) -> two bf16x2 via binary32 (exact: |q| <= 128).
__device__ __forceinline__ void codes_i8(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const float f0 = (float)(int8_t)(w & 255u), f1 = (float)(int8_t)((w >> 8) & 255u);
    const float f2 = (float)(int8_t)((w >> 16) & 255u), f3 = (float)(int8_t)(w >> 24);
    __nv_bfloat162 a = __floats2bfloat162_rn(f0, f1), b = __floats2bfloat162_rn(f2, f3);
    lo = *reinterpret_cast<uint32_t *>(&a);
    hi = *reinterpret_cast<uint32_t *>(&b);
}

// Spread 4 bits into bit `pos` of each byte.
__device__ __forceinline__ uint32_t spread4(uint32_t b, int pos) {
    return (((b & 1u)) | ((b & 2u) << 7) | ((b & 4u) << 14) | ((b & 8u) << 21)) << pos;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                               const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// ------------------------------------------------------------------------------------------ per-type fragments
// A macro block is 256 consecutive weights of a row (one K-quant super-block, 8 legacy blocks, 4 A4G64
// blocks), 16 groups of 16 weights. For group u, lane t supplies 4 weights of each of its two rows;
// Frag<QT> fixes which:
//   load(r, mb, t, nblk)  reads what lane t needs of one macro block of one row (nblk valid blocks, for
//                         the legacy types at a K tail);
//   codes(r, u)           the lane's 4 stored codes of group u, one per byte;
//   xoff(u, t)            offset, within the macro block, of the 4 consecutive weights those codes are
//                         (the activations are read from the same place);
//   UNIT                  weights per scale unit; the groups of unit s are u = s*UNIT/16 .. consecutive;
//   scale(r, s, ds, off)  the unit's scale and additive term (w = ds*(q - BIAS) + off).
// Types whose scales take several operations to unpack (the K-quants) set SPLIT: each lane then unpacks
// only a quarter of the units and the others fetch them with a warp shuffle.
template <int QT> struct Frag;

__device__ __forceinline__ float small_u2f(uint32_t v) {   // exact for v < 2^23
    return __int_as_float(0x4B000000 | v) - 8388608.0f;
}
__device__ __forceinline__ float small_i2f(int v) {         // exact for |v| < 2^22
    return __int_as_float(0x4B400000 + v) - 12582912.0f;
}

template <> struct Frag<T_Q4_0> {
    static constexpr int UNIT = 32, BIAS = 8;
    static constexpr bool SPLIT = false;
    struct Raw { uint32_t q[8]; float d[8]; };
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int nblk) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (b < nblk) {
                r.q[b] = ldw_a2(mb + 18 * b + 2 + 4 * t);
                r.d[b] = h2f(ld_u16(mb + 18 * b));
            } else { r.q[b] = 0; r.d[b] = 0.0f; }
        }
    }
    __device__ static uint32_t codes(const Raw &r, int u) { return (r.q[u >> 1] >> (4 * (u & 1))) & 0x0F0F0F0Fu; }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    __device__ static void scale(const Raw &r, int s, float &ds, float &off) { ds = r.d[s]; off = 0.0f; }
};

template <> struct Frag<T_Q4_1> {
    static constexpr int UNIT = 32, BIAS = 0;
    static constexpr bool SPLIT = false;
    struct Raw { uint32_t q[8]; uint32_t dm[8]; };
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int nblk) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (b < nblk) {
                r.q[b] = ld_u32(mb + 20 * b + 4 + 4 * t);
                r.dm[b] = ld_u32(mb + 20 * b);
            } else { r.q[b] = 0; r.dm[b] = 0; }
        }
    }
    __device__ static uint32_t codes(const Raw &r, int u) { return (r.q[u >> 1] >> (4 * (u & 1))) & 0x0F0F0F0Fu; }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    __device__ static void scale(const Raw &r, int s, float &ds, float &off) {
        ds = h2f(r.dm[s] & 0xffffu); off = h2f(r.dm[s] >> 16);
    }
};

// Q5_0 / Q5_1: element 16h + 4t + j of a block is the low (h = 0) or high (h = 1) nibble of qs[4t + j]
// plus bit 16h + 4t + j of qh as the fifth bit.
template <int QT> struct FragQ5 {
    static constexpr bool ONE = QT == T_Q5_1;
    static constexpr int UNIT = 32, BIAS = ONE ? 0 : 16, BYTES = ONE ? 24 : 22, QS = ONE ? 8 : 6, QH = ONE ? 4 : 2;
    static constexpr bool SPLIT = false;
    struct Raw { uint32_t q[8]; uint32_t qh[8]; uint32_t dm[8]; };
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int nblk) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (b < nblk) {
                r.q[b] = ONE ? ld_u32(mb + BYTES * b + QS + 4 * t) : ldw_a2(mb + BYTES * b + QS + 4 * t);
                r.qh[b] = ((ONE ? ld_u32(mb + BYTES * b + QH) : ldw_a2(mb + BYTES * b + QH)) >> (4 * t)) & 0x000F000Fu;
                r.dm[b] = ONE ? ld_u32(mb + BYTES * b) : ld_u16(mb + BYTES * b);
            } else { r.q[b] = 0; r.qh[b] = 0; r.dm[b] = 0; }
        }
    }
    __device__ static uint32_t codes(const Raw &r, int u) {
        const int b = u >> 1, h = u & 1;
        return ((r.q[b] >> (4 * h)) & 0x0F0F0F0Fu) | spread4((r.qh[b] >> (16 * h)) & 15u, 4);
    }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    __device__ static void scale(const Raw &r, int s, float &ds, float &off) {
        ds = h2f(r.dm[s] & 0xffffu);
        off = ONE ? h2f(r.dm[s] >> 16) : 0.0f;
    }
};
template <> struct Frag<T_Q5_0> : FragQ5<T_Q5_0> {};
template <> struct Frag<T_Q5_1> : FragQ5<T_Q5_1> {};

template <> struct Frag<T_Q8_0> {
    static constexpr int UNIT = 32, BIAS = 0;
    static constexpr bool SPLIT = false;
    struct Raw { uint32_t q[16]; float d[8]; };
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int nblk) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (b < nblk) {
                r.q[2 * b] = ldw_a2(mb + 34 * b + 2 + 4 * t);
                r.q[2 * b + 1] = ldw_a2(mb + 34 * b + 18 + 4 * t);
                r.d[b] = h2f(ld_u16(mb + 34 * b));
            } else { r.q[2 * b] = 0; r.q[2 * b + 1] = 0; r.d[b] = 0.0f; }
        }
    }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    __device__ static void scale(const Raw &r, int s, float &ds, float &off) { ds = r.d[s]; off = 0.0f; }
};

template <> struct Frag<T_Q2_K> {
    static constexpr int UNIT = 16, BIAS = 0;
    static constexpr bool SPLIT = true;
    struct Raw { uint32_t q[4]; uint32_t sc; uint32_t dd; };
    // lane t keeps the sub-block scale bytes of units 4t .. 4t+3 (scales[4t .. 4t+3])
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int) {
#pragma unroll
        for (int i = 0; i < 4; ++i) r.q[i] = ld_u32(mb + 16 + 32 * (i >> 1) + 16 * (i & 1) + 4 * t);
        r.sc = ld_u32(mb + 4 * t);
        r.dd = ld_u32(mb + 80);
    }
    __device__ static uint32_t codes(const Raw &r, int u) {
        return (r.q[2 * (u >> 3) + (u & 1)] >> (2 * ((u & 7) >> 1))) & 0x03030303u;
    }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    // unit 4t + i of this lane
    __device__ static void scale_own(const Raw &r, int i, float &ds, float &off) {
        const uint32_t b = (r.sc >> (8 * i)) & 255u;
        ds = __fmul_rn(h2f(r.dd & 0xffffu), small_u2f(b & 15u));
        off = -__fmul_rn(h2f(r.dd >> 16), small_u2f(b >> 4));
    }
};

template <> struct Frag<T_Q3_K> {
    static constexpr int UNIT = 16, BIAS = 4;
    static constexpr bool SPLIT = true;
    struct Raw { uint32_t q[4]; uint32_t hm[2]; uint32_t s[3]; float d; };
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int) {
#pragma unroll
        for (int i = 0; i < 4; ++i) r.q[i] = ldw_a2(mb + 32 + 32 * (i >> 1) + 16 * (i & 1) + 4 * t);
        r.hm[0] = ldw_a2(mb + 4 * t);
        r.hm[1] = ldw_a2(mb + 16 + 4 * t);
#pragma unroll
        for (int i = 0; i < 3; ++i) r.s[i] = ldw_a2(mb + 96 + 4 * i);
        r.d = h2f(ld_u16(mb + 108));
    }
    __device__ static uint32_t codes(const Raw &r, int u) {
        const uint32_t lo = (r.q[2 * (u >> 3) + (u & 1)] >> (2 * ((u & 7) >> 1))) & 0x03030303u;
        const uint32_t hb = (r.hm[u & 1] >> (u >> 1)) & 0x01010101u;
        return lo | (hb << 2);
    }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    __device__ static void scale_own_t(const Raw &r, int s, float &ds, float &off) {
        ds = __fmul_rn(r.d, small_i2f((int)six_bits(r.s[0], r.s[1], r.s[2], s) - 32));
        off = 0.0f;
    }
};

// Q4_K / Q5_K: lane t reads 8 consecutive code bytes of each 32-byte chunk c of qs, which hold weights
// 8t .. 8t+7 of sub-blocks 2c (low nibbles) and 2c+1 (high nibbles). Group u = 4c + 2*nib + hb takes the
// low (hb = 0) or high (hb = 1) four of them, nib selecting the sub-block.
template <int QT> struct FragQ45K {
    static constexpr int UNIT = 32, BIAS = 0;
    static constexpr bool SPLIT = true;
    struct Raw { uint2 q[4]; uint2 qh; uint32_t s0, s1, s2; uint32_t dd; };
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int) {
        const uint4 hd = ld_u128(mb);
        r.dd = hd.x; r.s0 = hd.y; r.s1 = hd.z; r.s2 = hd.w;
        constexpr int QOFF = QT == T_Q4_K ? 16 : 48;
#pragma unroll
        for (int c = 0; c < 4; ++c) r.q[c] = *reinterpret_cast<const uint2 *>(mb + QOFF + 32 * c + 8 * t);
        if (QT == T_Q5_K) r.qh = *reinterpret_cast<const uint2 *>(mb + 16 + 8 * t);
    }
    __device__ static uint32_t codes(const Raw &r, int u) {
        const int c = u >> 2, nib = (u >> 1) & 1, hb = u & 1;
        const uint32_t w = hb ? r.q[c].y : r.q[c].x;
        uint32_t v = (w >> (4 * nib)) & 0x0F0F0F0Fu;
        if (QT == T_Q5_K) v |= (((hb ? r.qh.y : r.qh.x) >> (u >> 1)) & 0x01010101u) << 4;
        return v;
    }
    __device__ static int xoff(int u, int t) { return 32 * (u >> 1) + 8 * t + 4 * (u & 1); }
    __device__ static void scale_own_t(const Raw &r, int s, float &ds, float &off) {
        ds = __fmul_rn(h2f(r.dd & 0xffffu), small_u2f(six_bits(r.s0, r.s1, r.s2, s)));
        off = -__fmul_rn(h2f(r.dd >> 16), small_u2f(six_bits(r.s0, r.s1, r.s2, 8 + s)));
    }
};
template <> struct Frag<T_Q4_K> : FragQ45K<T_Q4_K> {};
template <> struct Frag<T_Q5_K> : FragQ45K<T_Q5_K> {};

template <> struct Frag<T_Q6_K> {
    static constexpr int UNIT = 16, BIAS = 32;
    static constexpr bool SPLIT = true;
    struct Raw { uint32_t ql[8]; uint32_t qh[4]; uint32_t sc; float d; };
    // lane t keeps the int8 scales of units 4t .. 4t+3. The block starts 4-byte aligned or 2 past it.
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int) {
        if ((reinterpret_cast<uintptr_t>(mb) & 3u) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) r.ql[i] = ld_u32(mb + 64 * (i >> 2) + 16 * (i & 3) + 4 * t);
#pragma unroll
            for (int i = 0; i < 4; ++i) r.qh[i] = ld_u32(mb + 128 + 32 * (i >> 1) + 16 * (i & 1) + 4 * t);
            r.sc = ld_u32(mb + 192 + 4 * t);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) r.ql[i] = ldw_a2(mb + 64 * (i >> 2) + 16 * (i & 3) + 4 * t);
#pragma unroll
            for (int i = 0; i < 4; ++i) r.qh[i] = ldw_a2(mb + 128 + 32 * (i >> 1) + 16 * (i & 1) + 4 * t);
            r.sc = ldw_a2(mb + 192 + 4 * t);
        }
        r.d = h2f(ld_u16(mb + 208));
    }
    __device__ static uint32_t codes(const Raw &r, int u) {
        const int h = u >> 3;
        const uint32_t lo = (r.ql[4 * h + (u & 3)] >> (4 * ((u & 7) >> 2))) & 0x0F0F0F0Fu;
        const uint32_t hb = (r.qh[2 * h + (u & 1)] >> (2 * ((u & 7) >> 1))) & 0x03030303u;
        return lo | (hb << 4);
    }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    __device__ static void scale_own(const Raw &r, int i, float &ds, float &off) {
        ds = __fmul_rn(r.d, small_i2f((int)(int8_t)((r.sc >> (8 * i)) & 255u)));
        off = 0.0f;
    }
};

template <> struct Frag<T_A4G64> {
    static constexpr int UNIT = 64, BIAS = 0;
    static constexpr bool SPLIT = false;
    struct Raw { uint32_t q[8]; uint32_t sb[4]; };
    __device__ static void load(Raw &r, const uint8_t *mb, int t, int nblk) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            if (b < nblk) {
                r.q[2 * b] = ld_u32(mb + 36 * b + 4 + 4 * t);
                r.q[2 * b + 1] = ld_u32(mb + 36 * b + 20 + 4 * t);
                r.sb[b] = ld_u32(mb + 36 * b);
            } else { r.q[2 * b] = 0; r.q[2 * b + 1] = 0; r.sb[b] = 0; }
        }
    }
    __device__ static uint32_t codes(const Raw &r, int u) {
        return (r.q[2 * (u >> 2) + (u & 1)] >> (4 * ((u & 3) >> 1))) & 0x0F0F0F0Fu;
    }
    __device__ static int xoff(int u, int t) { return 16 * u + 4 * t; }
    __device__ static void scale(const Raw &r, int s, float &ds, float &off) {
        ds = bf2f(r.sb[s] & 0xffffu); off = bf2f(r.sb[s] >> 16);
    }
};

// The scale units a lane unpacks itself when SPLIT: units [t*UPL, (t+1)*UPL), UPL = units per lane.
template <int QT> struct OwnScales {
    static constexpr int UPL = (256 / Frag<QT>::UNIT) / 4;
    float ds[UPL], off[UPL];
};
template <int QT>
__device__ __forceinline__ void own_scales(const typename Frag<QT>::Raw &r, int t, OwnScales<QT> &o) {
    constexpr int UPL = OwnScales<QT>::UPL;
#pragma unroll
    for (int i = 0; i < UPL; ++i) {
        if constexpr (QT == T_Q2_K || QT == T_Q6_K) Frag<QT>::scale_own(r, i, o.ds[i], o.off[i]);
        else Frag<QT>::scale_own_t(r, UPL * t + i, o.ds[i], o.off[i]);
    }
}
// (ds, off) of unit s (compile-time) for the row this lane's group g decodes: from lane (g, s / UPL).
template <int QT>
__device__ __forceinline__ void unit_scale(const typename Frag<QT>::Raw &r, const OwnScales<QT> &o, int s, int g,
                                           float &ds, float &off) {
    if constexpr (Frag<QT>::SPLIT) {
        constexpr int UPL = OwnScales<QT>::UPL;
        const int src = 4 * g + s / UPL;
        ds = __shfl_sync(0xffffffffu, o.ds[s % UPL], src);
        off = (QT == T_Q6_K || QT == T_Q3_K) ? 0.0f : __shfl_sync(0xffffffffu, o.off[s % UPL], src);
    } else {
        Frag<QT>::scale(r, s, ds, off);
    }
}

// A operand halves (lo pair, hi pair) of one row for 16-weight group u.
template <int QT>
__device__ __forceinline__ void frag_codes(const typename Frag<QT>::Raw &r, int u, uint32_t &lo, uint32_t &hi) {
    if constexpr (QT == T_Q8_0) {
        codes_i8(r.q[u], lo, hi);
    } else {
        const uint32_t c = Frag<QT>::codes(r, u);
        constexpr uint32_t B2 = bias_bf16x2(Frag<QT>::BIAS);
        lo = codes_pair(c, SEL_LO, B2);
        hi = codes_pair(c, SEL_HI, B2);
    }
}

// ------------------------------------------------------------------------------------------ the kernel
// Shared memory, in order: the warps' mbarriers (NSMAX per warp), the weight ring (per warp NS stages of
// 16 rows x one macro block, one row per SLOT bytes), the activations of the CTA's K segment as bf16
// columns (xs), per-unit activation sums (sx), and the partial results that the warps of a CTA, then the
// CTAs of a cluster, add up (part).
constexpr int NSMAX = 8;
// Bytes of one row's macro block in a ring stage. A bulk copy must start and end on 16-byte boundaries, so
// a stage row holds the 16-byte-aligned range around the macro block: at most 15 bytes more on each side.
// An odd number of 16-byte units spreads the 8 rows a warp load touches over distinct banks.
template <int QT> __host__ __device__ constexpr int slot_bytes() {
    constexpr int B = (256 / TypeInfo<QT>::QK) * TypeInfo<QT>::BYTES;
    constexpr int S = (B + 15 + 15) / 16 * 16;
    return (S / 16) % 2 ? S : S + 16;
}
// Row stride of the resident tile for a segment of `seg` bytes per row: room for the 16-byte-aligned range
// around it, an odd number of 16-byte units.
__host__ __device__ inline int resident_stride(int seg) {
    const int s = (seg + 15 + 15) / 16 * 16;
    return (s / 16) % 2 ? s : s + 16;
}
template <int NT, bool XBF16> struct Layout {
    static constexpr int COLS = 8 * NT;              // MMA columns
    static constexpr int TOK = XBF16 ? 8 * NT : 4 * NT;   // tokens served
    static constexpr int WARPS = 8;
    // the warps' stage barriers, then one barrier that is initialised but never signalled (a test hook
    // waits on it to make a bounded wait run out)
    static constexpr int BARS = WARPS * NSMAX * 8 + 16;
    __host__ __device__ static int xs_stride(int kpad) { return kpad + 16; }   // elements; +32 B breaks bank aliasing
    // Columns actually staged: with one column group only those the tokens use (a power of two; the MMA
    // reads the others from a used column and their results are never read).
    __host__ __device__ static int staged_cols(int M) {
        if (NT > 1) return COLS;
        const int need = XBF16 ? M : 2 * M;
        int c = 2;
        while (c < need) c *= 2;
        return c < COLS ? c : COLS;
    }
    // activations, unit sums and partials
    __host__ __device__ static size_t xbytes(int kpad, int unit, int M) {
        return (size_t)staged_cols(M) * xs_stride(kpad) * 2 + (size_t)TOK * (kpad / unit) * 4 +
               (size_t)WARPS * 16 * TOK * 4;
    }
    __host__ __device__ static size_t ring_bytes(int slot, int ns) { return (size_t)WARPS * ns * 16 * slot; }
    // cluster reduction slots in rank 0: S slots of RG x 16 rows x TOK tokens
    __host__ __device__ static size_t red_bytes(int S, int rg) { return S > 1 ? (size_t)S * rg * 16 * TOK * 4 : 0; }
    // resident mode: RG row groups of 16 rows, `seg` bytes each
    __host__ __device__ static size_t tile_bytes(int rg, int seg) { return (size_t)rg * 16 * resident_stride(seg); }
    __host__ __device__ static size_t bytes(int kpad, int unit, int M, int slot, int ns) {
        return BARS + ring_bytes(slot, ns) + xbytes(kpad, unit, M);
    }
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split cluster barrier: arrive (relaxed) early, wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// Address of `local` (a shared memory location of this CTA) in the CTA of the cluster with rank `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    return ra;
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// One macro block of two rows into the accumulators. FULL: all 16 groups lie inside K.
template <int QT, int NT, bool XBF16, bool FULL>
__device__ __forceinline__ void macro_step(const typename Frag<QT>::Raw &cur0, const typename Frag<QT>::Raw &cur1,
                                           const __nv_bfloat16 *xs, int xst, const float *sx, int sxs, int kloc,
                                           int nvalid, int g, int t, int colmask, float (&acc)[NT][4]) {
    using F = Frag<QT>;
    constexpr int UNIT = F::UNIT, GPU = UNIT / 16;
    // types without an additive term (w = ds * (q - bias))
    constexpr bool SYM = QT == T_Q4_0 || QT == T_Q5_0 || QT == T_Q8_0 || QT == T_Q3_K || QT == T_Q6_K;
    OwnScales<QT> own0, own1;
    if constexpr (F::SPLIT) {
        own_scales<QT>(cur0, t, own0);
        own_scales<QT>(cur1, t, own1);
    }
    float d[NT][4];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        if (!FULL && u >= nvalid) break;
        uint32_t a[4];
        frag_codes<QT>(cur0, u, a[0], a[2]);
        frag_codes<QT>(cur1, u, a[1], a[3]);
        const int xo = kloc + F::xoff(u, t);
#pragma unroll
        for (int mt = 0; mt < NT; ++mt) {
            const int col = NT == 1 ? (g & colmask) : 8 * mt + g;
            const uint2 b = *reinterpret_cast<const uint2 *>(xs + (size_t)col * xst + xo);
            if ((u % GPU) == 0) {
                const float z[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16_16816(d[mt], a, b.x, b.y, z);
            } else {
                mma_bf16_16816(d[mt], a, b.x, b.y, d[mt]);
            }
        }
        if ((u % GPU) == GPU - 1) {
            const int su = u / GPU;                      // scale unit within the macro block
            const int sul = (kloc + 16 * u) / UNIT;      // scale unit within the segment
            float ds0, of0, ds1, of1;
            unit_scale<QT>(cur0, own0, su, g, ds0, of0);
            unit_scale<QT>(cur1, own1, su, g, ds1, of1);
#pragma unroll
            for (int mt = 0; mt < NT; ++mt) {
                if constexpr (XBF16 && SYM) {
                    acc[mt][0] = fmaf(ds0, d[mt][0], acc[mt][0]);
                    acc[mt][1] = fmaf(ds0, d[mt][1], acc[mt][1]);
                    acc[mt][2] = fmaf(ds1, d[mt][2], acc[mt][2]);
                    acc[mt][3] = fmaf(ds1, d[mt][3], acc[mt][3]);
                } else if constexpr (XBF16) {
                    const int tk = 8 * mt + 2 * t;
                    const float sx0 = sx[tk * sxs + sul], sx1 = sx[(tk + 1) * sxs + sul];
                    acc[mt][0] = fmaf(ds0, d[mt][0], fmaf(of0, sx0, acc[mt][0]));
                    acc[mt][1] = fmaf(ds0, d[mt][1], fmaf(of0, sx1, acc[mt][1]));
                    acc[mt][2] = fmaf(ds1, d[mt][2], fmaf(of1, sx0, acc[mt][2]));
                    acc[mt][3] = fmaf(ds1, d[mt][3], fmaf(of1, sx1, acc[mt][3]));
                } else if constexpr (SYM) {
                    acc[mt][0] = fmaf(ds0, d[mt][0] + d[mt][1], acc[mt][0]);
                    acc[mt][2] = fmaf(ds1, d[mt][2] + d[mt][3], acc[mt][2]);
                } else {
                    const float sxt = sx[(4 * mt + t) * sxs + sul];
                    acc[mt][0] = fmaf(ds0, d[mt][0] + d[mt][1], fmaf(of0, sxt, acc[mt][0]));
                    acc[mt][2] = fmaf(ds1, d[mt][2] + d[mt][3], fmaf(of1, sxt, acc[mt][2]));
                }
            }
        }
    }
}

// CTA: 8 warps = RG row groups of 16 rows x KW slices of the CTA's K segment; the cluster's S CTAs take
// consecutive K segments of the same rows.
//
// Weight stream, in one of two modes; in both the weights go to shared memory by bulk copies
// (cp.async.bulk) that lanes 0-15 of a warp issue, one per row, each arriving on an mbarrier with its byte
// count, and the copies are issued before the kernel waits for its predecessor in the stream, so that
// the weight stream of this launch overlaps the end of the previous one.
//   resident (ns == 0): the CTA's whole tile (its rows x its K segment) fits in shared memory. Warp
//     (rg, 0) copies each of its row group's 16 rows in one piece, all at once; the KW warps of the row
//     group wait on the group's mbarrier and decode their macro blocks from the tile.
//   ring (ns > 0): each warp streams its 16 rows through its own ring of `ns` stages of one macro block:
//     it waits on a stage's mbarrier, decodes the stage and refills it with the macro block `ns` steps
//     ahead. Used when the tile does not fit.
// Few large copies stream faster than many small ones, which is why the resident mode is preferred.
// Several weight matrices of one type and one K that take the same activations, served by one launch: the
// CTAs cover the row blocks of matrix 0, then of matrix 1, ...; rb0[i] is the first CTA (x index) of matrix i.
constexpr int kMaxMulti = 8;
struct Multi {
    int count;                      // 0: a single matrix (the kernel's own wq, N, y)
    int rb0[kMaxMulti + 1];
    const uint8_t *wq[kMaxMulti];
    int N[kMaxMulti];
    float *y[kMaxMulti];
};

template <int QT, int NT, bool XBF16, int KW>
__global__ void __launch_bounds__(256, 2)
    gemv_tc_kernel(const uint8_t *__restrict__ wq_, int N_, int64_t K, int64_t rowbytes, const void *__restrict__ x,
                   int M, float *__restrict__ y_, int kseg, int ns, unsigned int *__restrict__ status, int stall,
                   int early, const __grid_constant__ Multi multi) {
    using F = Frag<QT>;
    using LY = Layout<NT, XBF16>;
    constexpr int WARPS = LY::WARPS, RG = WARPS / KW;
    constexpr int UNIT = F::UNIT;
    constexpr int TOK = LY::TOK;
    constexpr int QK = TypeInfo<QT>::QK, BYTES = TypeInfo<QT>::BYTES;
    constexpr int BPM = 256 / QK;                     // blocks per macro block
    constexpr int SLOT = slot_bytes<QT>();
    extern __shared__ __align__(16) uint8_t smem[];

    const int S = gridDim.y;
    const int64_t kb = (int64_t)blockIdx.y * kseg;
    const int64_t ke = (kb + kseg < K) ? kb + kseg : K;
    const int kpad = kseg;                            // multiple of 256
    const int xst = LY::xs_stride(kpad), sxs = kpad / UNIT;
    const int scols = LY::staged_cols(M);
    const int colmask = scols - 1;                    // NT == 1: staged columns are a power of two
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *ring = smem + LY::BARS;
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(
        ring + (ns == 0 ? LY::tile_bytes(RG, kseg / 256 * BPM * BYTES) : LY::ring_bytes(SLOT, ns)));
    float *sx = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(xs) + (size_t)scols * xst * 2);
    float *part = sx + (size_t)TOK * sxs;             // [WARPS][16][TOK]

    // this CTA's matrix and its row block within it
    const uint8_t *wq = wq_;
    int N = N_;
    float *y = y_;
    int bx = blockIdx.x;
    if (multi.count > 0) {
        int i = 0;
        while (i + 1 < multi.count && bx >= multi.rb0[i + 1]) ++i;
        bx -= multi.rb0[i];
        wq = multi.wq[i];
        N = multi.N[i];
        y = multi.y[i];
    }

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int rg = warp / KW, ks = warp % KW;
    const int nrow0 = bx * (16 * RG) + 16 * rg;
    // this warp's macro blocks: a balanced share of the segment's
    const int64_t smb = kb / 256, nmb = (ke - kb + 255) / 256;
    const int64_t mb_beg = smb + (nmb * ks) / KW, mb_end = smb + (nmb * (ks + 1)) / KW;
    const int nsteps = (int)(mb_end - mb_beg);
    const int64_t nblocks_row = K / QK;
    const int64_t full_end = K / 256;                 // macro blocks lying entirely inside K
    auto nblk_of = [&](int64_t mb) {
        const int64_t r = nblocks_row - mb * BPM;
        return (int)(r < BPM ? r : BPM);
    };

    uint64_t *wbar = bars + warp * NSMAX;             // this warp's stage barriers (ring mode)
    uint64_t *gbar = bars + rg * NSMAX;                // the row group's tile barrier (resident mode)
    uint8_t *wring = ring + (size_t)warp * ns * 16 * SLOT;
    const bool resident = ns == 0;
    const int rstride = resident_stride(kseg / 256 * BPM * BYTES);
    uint8_t *gtile = ring + (size_t)rg * 16 * rstride;  // resident mode: row group rg's 16 rows
    // Lane l < 16 copies row nrow0 + l (clamped to the last row; the rows past N are never stored).
    const int crow = nrow0 + (lane & 15) < N ? nrow0 + (lane & 15) : N - 1;
    const uintptr_t wend = reinterpret_cast<uintptr_t>(wq) + (uintptr_t)N * (uintptr_t)rowbytes;
    auto issue = [&](int step) {
        const int slot = step % ns;
        if (lane < 16) {
            const int64_t mb = mb_beg + step;
            const uintptr_t a = reinterpret_cast<uintptr_t>(wq + (int64_t)crow * rowbytes + mb * BPM * BYTES);
            const uintptr_t e = a + (uintptr_t)nblk_of(mb) * BYTES;
            const uintptr_t a0 = a & ~(uintptr_t)15;
            uintptr_t e1 = (e + 15) & ~(uintptr_t)15;
            if (e1 > wend) e1 = wend & ~(uintptr_t)15;  // the buffer's last bytes, past its last 16-byte boundary
            uint8_t *dst = wring + (size_t)(slot * 16 + (lane & 15)) * SLOT;
            for (uintptr_t q = e1 > a0 ? e1 : a0; q < e; ++q) dst[q - a0] = *reinterpret_cast<const uint8_t *>(q);
            ptx::fence_proxy_async_smem();           // earlier generic reads of the stage before the async write
            ptx::mbar_arrive_expect_tx(&wbar[slot], e1 > a0 ? (uint32_t)(e1 - a0) : 0u);
            if (e1 > a0) ptx::bulk_load(dst, reinterpret_cast<const void *>(a0), (uint32_t)(e1 - a0), &wbar[slot]);
        }
    };
    // Rows g and g + 8 of a stage start where the copy put them: at the data's offset within 16 bytes.
    const uintptr_t radr0 = reinterpret_cast<uintptr_t>(wq + (int64_t)(nrow0 + g < N ? nrow0 + g : N - 1) * rowbytes);
    const uintptr_t radr1 =
        reinterpret_cast<uintptr_t>(wq + (int64_t)(nrow0 + g + 8 < N ? nrow0 + g + 8 : N - 1) * rowbytes);

    // Test hook (stall != 0): every warp of the first CTA that has weights to decode waits for its first
    // weight stage on `never`, a barrier nobody arrives on, so that the bounded wait runs out; the copies
    // themselves are issued and waited for (drained) as usual.
    uint64_t *never = bars + WARPS * NSMAX;
    const bool stall_here = stall != 0 && blockIdx.x == 0 && blockIdx.y == 0;
    if (stall_here && warp == 0 && lane == 0) ptx::mbar_init(never, 1);   // visible after the staging barrier

    // Before waiting for the preceding kernel in the stream, the weights this warp will copy are only
    // prefetched into L2 (coherent, so never stale even if that kernel wrote them); they are copied into
    // shared memory, and activations and outputs touched, only after the wait. With `early` (the caller
    // states that the preceding kernel does not write the weights) the copies themselves are issued before
    // the wait, so that they overlap the end of the preceding kernel.
    if (lane == 0)
        for (int i = 0; i < ns; ++i) ptx::mbar_init(&wbar[i], 16);
    if (resident && ks == 0 && lane == 0) ptx::mbar_init(gbar, 16);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (!early && lane < 16 && (!resident || ks == 0) && nsteps + (resident ? 1 : 0) > 0) {
        // resident: the row's whole segment; ring: this warp's macro blocks of the row
        const int64_t pb = resident ? smb : mb_beg;
        const int64_t pe_blocks = resident ? ((nblocks_row - smb * BPM) < (int64_t)(kseg / QK) ? nblocks_row - smb * BPM
                                                                                              : (int64_t)(kseg / QK))
                                           : (mb_end - mb_beg) * BPM;
        const uintptr_t a = reinterpret_cast<uintptr_t>(wq + (int64_t)crow * rowbytes + pb * BPM * BYTES);
        uintptr_t e = a + (uintptr_t)pe_blocks * BYTES;
        const uintptr_t rend = reinterpret_cast<uintptr_t>(wq + (int64_t)(crow + 1) * rowbytes);
        if (e > rend) e = rend;
        const uintptr_t a0 = a & ~(uintptr_t)15;
        uintptr_t e1 = (e + 15) & ~(uintptr_t)15;
        if (e1 > wend) e1 = wend & ~(uintptr_t)15;
        if (e1 > a0) ptx::prefetch_l2(reinterpret_cast<const void *>(a0), (uint32_t)(e1 - a0));
    }
    auto copy_weights = [&]() {
        if (resident) {
            // one copy per row: the segment's blocks of that row (warps with ks > 0 only wait for them)
            if (ks == 0 && lane < 16) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(wq + (int64_t)crow * rowbytes + smb * BPM * BYTES);
                const int64_t sblocks = (nblocks_row - smb * BPM) < (int64_t)(kseg / QK) ? nblocks_row - smb * BPM
                                                                                         : (int64_t)(kseg / QK);
                const uintptr_t e = a + (uintptr_t)sblocks * BYTES;
                const uintptr_t a0 = a & ~(uintptr_t)15;
                uintptr_t e1 = (e + 15) & ~(uintptr_t)15;
                if (e1 > wend) e1 = wend & ~(uintptr_t)15;
                uint8_t *dst = gtile + (size_t)lane * rstride;
                for (uintptr_t q = e1 > a0 ? e1 : a0; q < e; ++q) dst[q - a0] = *reinterpret_cast<const uint8_t *>(q);
                ptx::mbar_arrive_expect_tx(gbar, e1 > a0 ? (uint32_t)(e1 - a0) : 0u);
                if (e1 > a0) ptx::bulk_load(dst, reinterpret_cast<const void *>(a0), (uint32_t)(e1 - a0), gbar);
            }
        } else {
            const int npre = nsteps < ns ? nsteps : ns;
            for (int i = 0; i < npre; ++i) issue(i);
        }
    };
    if (early) copy_weights();
    if (gridDim.y > 1) cluster_arrive_relaxed();      // matched by the wait before the partials move
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!early) copy_weights();

    // ---- stage this segment's activations (tokens < M): bf16 columns and per-unit sums. The loads of XU
    //      iterations are issued together so that their latencies overlap.
    {
        constexpr int XU = 4, STEP = WARPS * 32;
        const int k4n = kpad / 4;
        const int mtok = M < TOK ? M : TOK;
        const int total = mtok * k4n;                 // a multiple of 64: the loop below is warp-uniform
        for (int base = tid; base < total; base += XU * STEP) {
            float v[XU][4];
#pragma unroll
            for (int j = 0; j < XU; ++j) {
                const int idx = base + j * STEP;
                const int tok = idx / k4n, k4 = idx - tok * k4n;
                const int64_t k = kb + 4 * k4;
                v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.0f;
                if (idx < total && k < ke) {
                    if constexpr (XBF16) {
                        const uint2 p = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(x) +
                                                                              (int64_t)tok * K + k));
                        v[j][0] = __uint_as_float(p.x << 16); v[j][1] = __uint_as_float(p.x & 0xffff0000u);
                        v[j][2] = __uint_as_float(p.y << 16); v[j][3] = __uint_as_float(p.y & 0xffff0000u);
                    } else {
                        const float4 p = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(x) +
                                                                               (int64_t)tok * K + k));
                        v[j][0] = p.x; v[j][1] = p.y; v[j][2] = p.z; v[j][3] = p.w;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < XU; ++j) {
                const int idx = base + j * STEP;
                if (idx >= total) break;
                const int tok = idx / k4n, k4 = idx - tok * k4n;
                if constexpr (XBF16) {
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[j][0], v[j][1]),
                                   h1 = __floats2bfloat162_rn(v[j][2], v[j][3]);
                    *reinterpret_cast<uint2 *>(xs + (size_t)tok * xst + 4 * k4) =
                        make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
                } else {
                    float hi[4], lo[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        hi[i] = __bfloat162float(__float2bfloat16_rn(v[j][i]));
                        lo[i] = __fsub_rn(v[j][i], hi[i]);
                    }
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(hi[0], hi[1]), h1 = __floats2bfloat162_rn(hi[2], hi[3]);
                    __nv_bfloat162 l0 = __floats2bfloat162_rn(lo[0], lo[1]), l1 = __floats2bfloat162_rn(lo[2], lo[3]);
                    const int col = 8 * (tok >> 2) + 2 * (tok & 3);
                    *reinterpret_cast<uint2 *>(xs + (size_t)col * xst + 4 * k4) =
                        make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
                    *reinterpret_cast<uint2 *>(xs + (size_t)(col + 1) * xst + 4 * k4) =
                        make_uint2(*reinterpret_cast<uint32_t *>(&l0), *reinterpret_cast<uint32_t *>(&l1));
                }
                // per-unit sums of x (binary32, original values), reduced over the UNIT/4 lanes of a unit
                float sum = (v[j][0] + v[j][1]) + (v[j][2] + v[j][3]);
#pragma unroll
                for (int off = 1; off < UNIT / 4; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                if ((k4 & (UNIT / 4 - 1)) == 0) sx[tok * sxs + (4 * k4) / UNIT] = sum;
            }
        }
    }
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int mt = 0; mt < NT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[mt][j] = 0.0f;

    typename F::Raw cur0, cur1;
    int done = 0;                                     // stages consumed (a timed-out wait stops the stream)
    for (; done < nsteps; ++done) {
        const int64_t mb = mb_beg + done;
        const uint8_t *p0, *p1;
        uint64_t *first = stall_here && done == 0 ? never : nullptr;
        if (resident) {
            if (done == 0 && !__all_sync(0xffffffffu, ptx::mbar_wait(first ? first : gbar, 0u, status))) break;
            const uintptr_t so = (uintptr_t)(smb * BPM * BYTES);          // the segment's first byte in a row
            const size_t jo = (size_t)(mb - smb) * BPM * BYTES;           // this macro block within the segment
            p0 = gtile + (size_t)g * rstride + ((radr0 + so) & 15) + jo;
            p1 = gtile + (size_t)(g + 8) * rstride + ((radr1 + so) & 15) + jo;
        } else {
            const int slot = done % ns;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(first ? first : &wbar[slot], (uint32_t)((done / ns) & 1),
                                                         status)))
                break;
            const uintptr_t mo = (uintptr_t)(mb * BPM * BYTES);
            p0 = wring + (size_t)(slot * 16 + g) * SLOT + ((radr0 + mo) & 15);
            p1 = wring + (size_t)(slot * 16 + g + 8) * SLOT + ((radr1 + mo) & 15);
        }
        F::load(cur0, p0, t, nblk_of(mb));
        F::load(cur1, p1, t, nblk_of(mb));
        const int kloc = (int)(mb * 256 - kb);    // position of this macro block in the segment
        if (mb < full_end) {
            macro_step<QT, NT, XBF16, true>(cur0, cur1, xs, xst, sx, sxs, kloc, 16, g, t, colmask, acc);
        } else {
            macro_step<QT, NT, XBF16, false>(cur0, cur1, xs, xst, sx, sxs, kloc, (int)((K - mb * 256) / 16), g, t,
                                             colmask, acc);
        }
        if (!resident) {
            __syncwarp();
            if (done + ns < nsteps) issue(done + ns);
        }
    }
    // After a timeout: wait (bounded) for this warp's copies still in flight before the shared memory is
    // released: in the ring, the stage that was being waited for and those issued after it; in resident
    // mode, the tile (its copies were issued by this row group's first warp).
    if (done < nsteps) {
        if (resident) {
            if (done == 0) ptx::mbar_wait(gbar, 0u, status);
        } else {
            for (int i = done; i < nsteps && i < done + ns; ++i)
                ptx::mbar_wait(&wbar[i % ns], (uint32_t)((i / ns) & 1), status);
        }
    }

    // ---- results. binary32 x: acc[mt][0] = (row g, token 4mt+t), acc[mt][2] = (row g+8, token 4mt+t);
    //      bf16 x: acc[mt][0/1] = (row g, tokens 8mt+2t, +1), acc[mt][2/3] = (row g+8, same tokens).
    float *pw = part + (size_t)warp * 16 * TOK;
#pragma unroll
    for (int mt = 0; mt < NT; ++mt) {
        if constexpr (XBF16) {
            const int tk = 8 * mt + 2 * t;
            pw[g * TOK + tk] = acc[mt][0]; pw[g * TOK + tk + 1] = acc[mt][1];
            pw[(g + 8) * TOK + tk] = acc[mt][2]; pw[(g + 8) * TOK + tk + 1] = acc[mt][3];
        } else {
            const int tk = 4 * mt + t;
            pw[g * TOK + tk] = acc[mt][0];
            pw[(g + 8) * TOK + tk] = acc[mt][2];
        }
    }
    __syncthreads();
    // Add the KW slices (fixed order). With a cluster, every CTA then stores its sums into rank 0's
    // shared memory (slot = its rank), one cluster barrier makes them visible, and rank 0 adds the S slots
    // in rank order.
    const int mtok = M < TOK ? M : TOK;
    const int nres = RG * 16 * mtok;
    float *red = part + (size_t)WARPS * 16 * TOK;     // [S][nres], used in rank 0 (cluster launches only)
    uint32_t rank = 0, red0 = 0;
    if (S > 1) {
        cluster_wait();                               // every CTA of the cluster has started
        rank = cluster_rank();
        red0 = dsmem_addr(red, 0);
    }
    for (int idx = tid; idx < nres; idx += WARPS * 32) {
        const int r = idx / mtok, tk = idx - r * mtok;     // r: row within the CTA
        const int rgi = r >> 4, rr = r & 15;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < KW; ++q) sum += part[((size_t)(rgi * KW + q) * 16 + rr) * TOK + tk];
        if (S == 1) {
            const int n = bx * (16 * RG) + r;
            if (n < N) y[(int64_t)tk * N + n] = sum;
        } else {
            st_dsmem_f32(red0 + 4u * (rank * (uint32_t)nres + (uint32_t)idx), sum);
        }
    }
    if (S > 1) {
        cluster_sync();
        if (rank == 0) {
            for (int idx = tid; idx < nres; idx += WARPS * 32) {
                const int r = idx / mtok, tk = idx - r * mtok;
                float sum = 0.0f;
                for (int q = 0; q < S; ++q) sum += red[q * nres + idx];
                const int n = bx * (16 * RG) + r;
                if (n < N) y[(int64_t)tk * N + n] = sum;
            }
        }
    }
}


// ------------------------------------------------------------------------------------------ expert-indexed
// Expert-indexed mat-vec (the pages' MUL_MAT_ID; llama.cpp PR 28086, "metal : fix idle threads in
// mul_mv_iq3_xxs for ne00 < 1024", "Overview"): y[(t*topk + j)*N + n] = sum_k dequant(W_e)[n, k] x[t, k]
// with e = ids[t*topk + j]. CTA (row block, K segment, rank u) serves the u-th distinct expert in
// ascending id order: it reads the routing table after waiting for its predecessor (the table usually
// comes from the router kernel), copies that expert's rows of its row block into shared memory once (one
// bulk copy per row, as the resident mode of the mat-vec kernel), and multiplies them by the activations
// of every (token, slot) routed to the expert, TOK of them per pass, the activations gathered into MMA
// columns. So each expert's weights are read once per call however many tokens chose it. CTAs whose rank
// exceeds the number of distinct experts leave at once (the whole cluster, which shares the rank).
struct IdExperts {
    const uint8_t *p[QMM_MAX_EXPERTS];
};

template <int QT, int NT, bool XBF16, int KW>
__global__ void __launch_bounds__(256, 2)
    gemv_tc_id_kernel(const __grid_constant__ IdExperts ex, int E, int N, int64_t K, int64_t rowbytes,
                      const void *__restrict__ x, int xdiv, const int32_t *__restrict__ ids, int M, int topk,
                      float *__restrict__ y, int kseg, unsigned int *__restrict__ status) {
    using F = Frag<QT>;
    using LY = Layout<NT, XBF16>;
    constexpr int WARPS = LY::WARPS, RG = WARPS / KW;
    constexpr int UNIT = F::UNIT;
    constexpr int TOK = LY::TOK;
    constexpr int QK = TypeInfo<QT>::QK, BYTES = TypeInfo<QT>::BYTES;
    constexpr int BPM = 256 / QK;
    extern __shared__ __align__(16) uint8_t smem[];

    const int S = gridDim.y;
    const int u = blockIdx.z;
    const int64_t kb = (int64_t)blockIdx.y * kseg;
    const int64_t ke = (kb + kseg < K) ? kb + kseg : K;
    const int kpad = kseg;
    const int xst = LY::xs_stride(kpad), sxs = kpad / UNIT;
    const int scols = LY::COLS;                        // all columns staged (the token count varies per pass)
    const int nslot = M * topk;
    const int rstride = resident_stride(kseg / 256 * BPM * BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *tile = smem + LY::BARS;
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(tile + LY::tile_bytes(RG, kseg / 256 * BPM * BYTES));
    float *sx = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(xs) + (size_t)scols * xst * 2);
    float *part = sx + (size_t)TOK * sxs;              // [WARPS][16][TOK]
    float *red = part + (size_t)WARPS * 16 * TOK;      // [S][RG*16*TOK] in rank 0
    int *s_slot = reinterpret_cast<int *>(red + (S > 1 ? (size_t)S * RG * 16 * TOK : 0));   // [nslot]
    unsigned char *s_used = reinterpret_cast<unsigned char *>(s_slot + nslot);              // [QMM_MAX_EXPERTS]
    __shared__ int s_nexp, s_expert, s_ns;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int rg = warp / KW, ks = warp % KW;
    const int nrow0 = blockIdx.x * (16 * RG) + 16 * rg;

    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (S > 1) cluster_arrive_relaxed();              // matched by the wait before the partials move

    // ---- routing: distinct experts in ascending id order, and the slots routed to this CTA's expert.
    //      The table is read once, into s_slot; the slot list of the expert later replaces it in place.
    for (int i = tid; i < QMM_MAX_EXPERTS; i += WARPS * 32) s_used[i] = 0;
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < nslot; i += WARPS * 32) {
        const int e = ids[i];
        s_slot[i] = e;
        if (e >= 0 && e < E) s_used[e] = 1;
        else bad = true;
    }
    bad = __syncthreads_or(bad);
    if (warp == 0) {
        int base = 0, mine = -1;
        for (int w0 = 0; w0 < QMM_MAX_EXPERTS; w0 += 32) {
            const bool used = s_used[w0 + lane] != 0;
            const unsigned b = __ballot_sync(0xffffffffu, used);
            if (used && base + __popc(b & ((1u << lane) - 1u)) == u) mine = w0 + lane;
            base += __popc(b);
        }
        mine = __reduce_max_sync(0xffffffffu, mine);
        if (lane == 0) { s_nexp = base; s_expert = mine; }
    }
    __syncthreads();
    if (bad && u == 0 && blockIdx.y == 0) {
        // slots with an id outside [0, E): NaN rows (this CTA's rows) and a status bit
        for (int p = 0; p < nslot; ++p) {
            const int e = s_slot[p];
            if (e < 0 || e >= E)
                for (int r = tid; r < 16 * RG; r += WARPS * 32) {
                    const int n = blockIdx.x * (16 * RG) + r;
                    if (n < N) y[(int64_t)p * N + n] = __int_as_float(0x7fc00000);
                }
        }
        if (tid == 0 && blockIdx.x == 0) atomicOr(status, kStatusBadId);
    }
    if (u >= s_nexp) {
        if (S > 1) cluster_wait();                    // (the whole cluster leaves: it shares u)
        return;
    }
    const int e = s_expert;
    __syncthreads();                                  // the table in s_slot is read before it is compacted

    // ---- this expert's rows of the row block, one bulk copy per row of the K segment (issued first)
    const uint8_t *wq = ex.p[e];
    const int64_t smb = kb / 256, nmb = (ke - kb + 255) / 256;
    const int64_t mb_beg = smb + (nmb * ks) / KW, mb_end = smb + (nmb * (ks + 1)) / KW;
    const int nsteps = (int)(mb_end - mb_beg);
    const int64_t nblocks_row = K / QK;
    const int64_t full_end = K / 256;
    auto nblk_of = [&](int64_t mb) {
        const int64_t r = nblocks_row - mb * BPM;
        return (int)(r < BPM ? r : BPM);
    };
    uint64_t *gbar = bars + rg * NSMAX;
    uint8_t *gtile = tile + (size_t)rg * 16 * rstride;
    const uintptr_t wend = reinterpret_cast<uintptr_t>(wq) + (uintptr_t)N * (uintptr_t)rowbytes;
    if (ks == 0) {
        if (lane == 0) ptx::mbar_init(gbar, 16);
        ptx::fence_mbar_init();
        __syncwarp();
        if (lane < 16) {
            const int crow = nrow0 + lane < N ? nrow0 + lane : N - 1;
            const uintptr_t a = reinterpret_cast<uintptr_t>(wq + (int64_t)crow * rowbytes + smb * BPM * BYTES);
            const int64_t sblocks = (nblocks_row - smb * BPM) < (int64_t)(kseg / QK) ? nblocks_row - smb * BPM
                                                                                     : (int64_t)(kseg / QK);
            const uintptr_t en = a + (uintptr_t)sblocks * BYTES;
            const uintptr_t a0 = a & ~(uintptr_t)15;
            uintptr_t e1 = (en + 15) & ~(uintptr_t)15;
            if (e1 > wend) e1 = wend & ~(uintptr_t)15;
            uint8_t *dst = gtile + (size_t)lane * rstride;
            for (uintptr_t q = e1 > a0 ? e1 : a0; q < en; ++q) dst[q - a0] = *reinterpret_cast<const uint8_t *>(q);
            ptx::mbar_arrive_expect_tx(gbar, e1 > a0 ? (uint32_t)(e1 - a0) : 0u);
            if (e1 > a0) ptx::bulk_load(dst, reinterpret_cast<const void *>(a0), (uint32_t)(e1 - a0), gbar);
        }
    }
    if (warp == 0) {
        // ordered compaction of the slots of expert e, in place: a chunk of 32 is read before any lane
        // writes, and writes land at or before the chunk
        int c = 0;
        for (int p0 = 0; p0 < nslot; p0 += 32) {
            const bool hit = p0 + lane < nslot && s_slot[p0 + lane] == e;
            const unsigned b = __ballot_sync(0xffffffffu, hit);
            if (hit) s_slot[c + __popc(b & ((1u << lane) - 1u))] = p0 + lane;
            c += __popc(b);
        }
        if (lane == 0) s_ns = c;
    }
    __syncthreads();                                  // slot list and tile barrier initialised
    const int ns = s_ns;
    const uintptr_t radr0 = reinterpret_cast<uintptr_t>(wq + (int64_t)(nrow0 + g < N ? nrow0 + g : N - 1) * rowbytes);
    const uintptr_t radr1 =
        reinterpret_cast<uintptr_t>(wq + (int64_t)(nrow0 + g + 8 < N ? nrow0 + g + 8 : N - 1) * rowbytes);
    const uintptr_t so = (uintptr_t)(smb * BPM * BYTES);
    bool tile_ok = true;
    if (S > 1) cluster_wait();                        // every CTA of the cluster has started

    for (int p0 = 0; p0 < ns; p0 += TOK) {
        const int mtok = ns - p0 < TOK ? ns - p0 : TOK;
        // ---- gathered activations of this pass's tokens: bf16 columns and per-unit sums
        {
            const int k4n = kpad / 4;
            const int total = mtok * k4n;             // a multiple of 64: warp-uniform loop
            for (int idx = tid; idx < total; idx += WARPS * 32) {
                const int tk = idx / k4n, k4 = idx - tk * k4n;
                const int64_t k = kb + 4 * k4;
                const int tok = s_slot[p0 + tk] / xdiv;     // x row: the token's (xdiv = topk) or the slot's
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (k < ke) {
                    if constexpr (XBF16) {
                        const uint2 pv = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(x) +
                                                                               (int64_t)tok * K + k));
                        v[0] = __uint_as_float(pv.x << 16); v[1] = __uint_as_float(pv.x & 0xffff0000u);
                        v[2] = __uint_as_float(pv.y << 16); v[3] = __uint_as_float(pv.y & 0xffff0000u);
                    } else {
                        const float4 pv = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(x) +
                                                                                (int64_t)tok * K + k));
                        v[0] = pv.x; v[1] = pv.y; v[2] = pv.z; v[3] = pv.w;
                    }
                }
                if constexpr (XBF16) {
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
                    *reinterpret_cast<uint2 *>(xs + (size_t)tk * xst + 4 * k4) =
                        make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
                } else {
                    float hi[4], lo[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        hi[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
                        lo[i] = __fsub_rn(v[i], hi[i]);
                    }
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(hi[0], hi[1]), h1 = __floats2bfloat162_rn(hi[2], hi[3]);
                    __nv_bfloat162 l0 = __floats2bfloat162_rn(lo[0], lo[1]), l1 = __floats2bfloat162_rn(lo[2], lo[3]);
                    const int col = 8 * (tk >> 2) + 2 * (tk & 3);
                    *reinterpret_cast<uint2 *>(xs + (size_t)col * xst + 4 * k4) =
                        make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
                    *reinterpret_cast<uint2 *>(xs + (size_t)(col + 1) * xst + 4 * k4) =
                        make_uint2(*reinterpret_cast<uint32_t *>(&l0), *reinterpret_cast<uint32_t *>(&l1));
                }
                float sum = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
                for (int off = 1; off < UNIT / 4; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                if ((k4 & (UNIT / 4 - 1)) == 0) sx[tk * sxs + (4 * k4) / UNIT] = sum;
            }
        }
        __syncthreads();

        float acc[NT][4];
#pragma unroll
        for (int mt = 0; mt < NT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[mt][j] = 0.0f;
        if (p0 == 0 && nsteps > 0)
            tile_ok = __all_sync(0xffffffffu, ptx::mbar_wait(gbar, 0u, status));
        if (tile_ok) {
            typename F::Raw cur0, cur1;
            for (int i = 0; i < nsteps; ++i) {
                const int64_t mb = mb_beg + i;
                const size_t jo = (size_t)(mb - smb) * BPM * BYTES;
                F::load(cur0, gtile + (size_t)g * rstride + ((radr0 + so) & 15) + jo, t, nblk_of(mb));
                F::load(cur1, gtile + (size_t)(g + 8) * rstride + ((radr1 + so) & 15) + jo, t, nblk_of(mb));
                const int kloc = (int)(mb * 256 - kb);
                if (mb < full_end)
                    macro_step<QT, NT, XBF16, true>(cur0, cur1, xs, xst, sx, sxs, kloc, 16, g, t, scols - 1, acc);
                else
                    macro_step<QT, NT, XBF16, false>(cur0, cur1, xs, xst, sx, sxs, kloc, (int)((K - mb * 256) / 16), g,
                                                     t, scols - 1, acc);
            }
        }
        float *pw = part + (size_t)warp * 16 * TOK;
#pragma unroll
        for (int mt = 0; mt < NT; ++mt) {
            if constexpr (XBF16) {
                const int tk = 8 * mt + 2 * t;
                pw[g * TOK + tk] = acc[mt][0]; pw[g * TOK + tk + 1] = acc[mt][1];
                pw[(g + 8) * TOK + tk] = acc[mt][2]; pw[(g + 8) * TOK + tk + 1] = acc[mt][3];
            } else {
                const int tk = 4 * mt + t;
                pw[g * TOK + tk] = acc[mt][0];
                pw[(g + 8) * TOK + tk] = acc[mt][2];
            }
        }
        __syncthreads();
        // K slices (fixed order), then the K segments of the cluster in rank order (as the mat-vec kernel)
        const int nres = RG * 16 * mtok;
        const uint32_t rank = S > 1 ? cluster_rank() : 0;
        const uint32_t red0 = S > 1 ? dsmem_addr(red, 0) : 0;
        for (int idx = tid; idx < nres; idx += WARPS * 32) {
            const int r = idx / mtok, tk = idx - r * mtok;
            const int rgi = r >> 4, rr = r & 15;
            float sum = 0.0f;
#pragma unroll
            for (int q = 0; q < KW; ++q) sum += part[((size_t)(rgi * KW + q) * 16 + rr) * TOK + tk];
            if (S == 1) {
                const int n = blockIdx.x * (16 * RG) + r;
                if (n < N) y[(int64_t)s_slot[p0 + tk] * N + n] = sum;
            } else {
                st_dsmem_f32(red0 + 4u * (rank * (uint32_t)nres + (uint32_t)idx), sum);
            }
        }
        if (S > 1) {
            cluster_sync();
            if (rank == 0) {
                for (int idx = tid; idx < nres; idx += WARPS * 32) {
                    const int r = idx / mtok, tk = idx - r * mtok;
                    float sum = 0.0f;
                    for (int q = 0; q < S; ++q) sum += red[q * nres + idx];
                    const int n = blockIdx.x * (16 * RG) + r;
                    if (n < N) y[(int64_t)s_slot[p0 + tk] * N + n] = sum;
                }
            }
            cluster_sync();                           // rank 0 has read its slots before the next pass
        }
        __syncthreads();                              // activations and partials are reused by the next pass
    }
    // After a timeout nothing more is read from the tile, but the copies must land before the CTA exits.
    if (!tile_ok) ptx::mbar_wait(gbar, 0u, status);
    if (ns == 0 && nsteps > 0) ptx::mbar_wait(gbar, 0u, status);
}

}  // namespace gtc

// ------------------------------------------------------------------------------------------ host side
namespace {

// Shared memory a CTA may take: two CTAs fit on an SM (228 KB), so one CTA of the next launch in the
// stream can start streaming its weights while one of this launch still runs.
constexpr size_t kSmemCap = 110 * 1024;
// A resident tile may also take up to this much when the split then fits one wave at one CTA per SM (the
// next launch cannot start its copies early on such an SM, which the work-split cost charges).
constexpr size_t kSmemBig = 200 * 1024;

// CTAs of this kernel instance that can be resident at once when launched in clusters of S (S = 1: no
// cluster), for a given dynamic shared memory size; queried once per (S, 4 KB size class) and cached.
template <int QT, int NT, bool XBF16, int KW>
int64_t gtc_capacity(int64_t S, size_t smem) {
    using LY = gtc::Layout<NT, XBF16>;
    auto kern = gtc::gemv_tc_kernel<QT, NT, XBF16, KW>;
    constexpr int NCLS = (int)(kSmemBig / 4096) + 1;
    static int64_t cache[kMaxDevices][9][NCLS] = {};
    static bool attr_set[kMaxDevices] = {};
    const int dev = current_device_index();
    const int cls = (int)((smem + 4095) / 4096);
    if (S < 1 || S > 8 || cls >= NCLS) return 0;
    if (cache[dev][S][cls]) return cache[dev][S][cls];
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBig) != cudaSuccess)
            return 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess) return 0;
        attr_set[dev] = true;
    }
    const size_t smem_q = (size_t)cls * 4096;
    int64_t cap = 0;
    if (S == 1) {
        int per_sm = 0;
        const int sms = device_sm_count();
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, LY::WARPS * 32, smem_q) == cudaSuccess)
            cap = (int64_t)per_sm * sms;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)S, 1);
        cfg.blockDim = dim3(LY::WARPS * 32, 1, 1);
        cfg.dynamicSmemBytes = smem_q;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)S;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) == cudaSuccess) cap = (int64_t)nclusters * S;
    }
    if (cap <= 0) cap = S;          // unknown: assume one cluster at a time rather than fail
    cache[dev][S][cls] = cap;
    return cap;
}

template <int QT, int NT, bool XBF16, int KW>
int launch_gtc_kw(const MatSet &ms, int64_t K, const void *x, int M, int64_t S, int64_t kseg, int ns,
                  unsigned int *status, cudaStream_t st, int stall, int early) {
    using LY = gtc::Layout<NT, XBF16>;
    constexpr int UNIT = gtc::Frag<QT>::UNIT, RG = LY::WARPS / KW;
    auto kern = gtc::gemv_tc_kernel<QT, NT, XBF16, KW>;
    if (gtc_capacity<QT, NT, XBF16, KW>(1, 0) <= 0) return -6;   // also sets the kernel's attributes
    gtc::Multi multi = {};
    int64_t nrb = 0;
    for (int i = 0; i < ms.count; ++i) {
        multi.rb0[i] = (int)nrb;
        multi.wq[i] = static_cast<const uint8_t *>(ms.wq[i]);
        multi.N[i] = (int)ms.N[i];
        multi.y[i] = ms.y[i];
        nrb += (ms.N[i] + 16 * RG - 1) / (16 * RG);
    }
    multi.rb0[ms.count] = (int)nrb;
    multi.count = ms.count > 1 ? ms.count : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nrb, (unsigned)S, 1);
    cfg.blockDim = dim3(LY::WARPS * 32, 1, 1);
    constexpr int MB_BYTES = 256 / TypeInfo<QT>::QK * TypeInfo<QT>::BYTES;
    cfg.dynamicSmemBytes = (ns == 0 ? LY::BARS + LY::tile_bytes(RG, (int)(kseg / 256 * MB_BYTES)) +
                                          LY::xbytes((int)kseg, UNIT, M)
                                    : LY::bytes((int)kseg, UNIT, M, gtc::slot_bytes<QT>(), ns)) +
                           LY::red_bytes((int)S, RG);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, multi.count ? multi.wq[0] : static_cast<const uint8_t *>(ms.wq[0]),
                                       (int)ms.N[0], K, row_bytes(QT, K), x, M, ms.y[0], (int)kseg, ns, status, stall,
                                       early, multi);
    return e == cudaSuccess ? 0 : -6;
}

// Work split. The CTAs of one launch should fit in one wave (resident CTAs as the occupancy calculator
// reports them, clusters included: a cluster must fit on one GPC, which strands slots): a second, partial
// wave doubles the time of these short kernels. Among the (K slices per CTA, K segments per cluster)
// choices that fit, take the one that leaves each warp the fewest macro blocks to stream (counting a
// cluster and a ring as one macro block more each, as measured on the layer shapes); larger M keeps
// more row groups per CTA so that the activations each CTA stages stay small next to its weights. Each
// warp's ring takes as many stages as the shared memory left over allows (at most its macro blocks).
template <int QT, int NT, bool XBF16>
int launch_gtc_t(const MatSet &ms, int64_t K, const void *x, int M, unsigned int *status, cudaStream_t st, bool dry,
                 int stall, int early) {
    using LY = gtc::Layout<NT, XBF16>;
    constexpr int UNIT = gtc::Frag<QT>::UNIT, SLOT = gtc::slot_bytes<QT>();
    constexpr int MB_BYTES = 256 / TypeInfo<QT>::QK * TypeInfo<QT>::BYTES;   // bytes of a macro block
    int64_t total_rows = 0;
    for (int i = 0; i < ms.count; ++i) total_rows += ms.N[i];
    // CTAs in x for `rg` row groups per CTA: every matrix's row blocks separately
    auto row_blocks = [&](int64_t rg) {
        int64_t n = 0;
        for (int i = 0; i < ms.count; ++i) n += ((ms.N[i] + 15) / 16 + rg - 1) / rg;
        return n;
    };
    const int64_t nmacro = (K + 255) / 256;
    // K slices per CTA: more for fewer tokens (the staged activations are then small); only the counts
    // that some M of this column-group count can use are compiled.
    constexpr int KWMAX = NT == 1 ? 8 : ((NT == 2 && !XBF16) ? 2 : 1);
    int kw_cap = M <= 2 ? 8 : (M <= 4 ? 4 : (M <= 8 ? 2 : 1));
    if (kw_cap > KWMAX) kw_cap = KWMAX;
    int best_kw = 1, best_s = 1, best_ns = 1;
    int64_t best_cost = -1, best_ctas = 0;
    for (int kw = 1; kw <= kw_cap; kw *= 2) {
        const int64_t nrb = row_blocks(8 / kw);
        for (int64_t S = 1; S <= 8 && S <= nmacro; ++S) {
            const int64_t kseg = ((nmacro + S - 1) / S) * 256;
            if ((K + kseg - 1) / kseg != S) continue;                 // S segments must all be non-empty
            const int64_t per_warp = (kseg / 256 + kw - 1) / kw;      // macro blocks per warp (at most)
            const size_t fixed = LY::BARS + LY::xbytes((int)kseg, UNIT, M) + LY::red_bytes((int)S, 8 / kw);
            const size_t tile = LY::tile_bytes(8 / kw, (int)(kseg / 256 * MB_BYTES));
            const int64_t ctas = nrb * S;
            // candidates: resident tile (two CTAs per SM, or one with a large tile), or a ring
            auto consider = [&](int64_t ns, size_t smem, int64_t extra) {
                int64_t resident = 0;
                if (kw == 1) resident = gtc_capacity<QT, NT, XBF16, 1>(S, smem);
                if constexpr (KWMAX >= 2) if (kw == 2) resident = gtc_capacity<QT, NT, XBF16, 2>(S, smem);
                if constexpr (KWMAX >= 4) if (kw == 4) resident = gtc_capacity<QT, NT, XBF16, 4>(S, smem);
                if constexpr (KWMAX >= 8) if (kw == 8) resident = gtc_capacity<QT, NT, XBF16, 8>(S, smem);
                if (resident <= 0) return;
                const int64_t waves = (ctas + resident - 1) / resident;
                // In macro blocks per warp: +2 per wave for its start, the activation staging and the
                // reduction, +1 more per 4096 activations a CTA stages, +1 for a cluster (its barriers and
                // the exchange of partial sums cost about as much as a macro block), plus `extra`.
                const int64_t cost = waves * (per_warp + 2) + ((int64_t)M * kseg) / 4096 + (S > 1 ? 1 : 0) + extra;
                if (best_cost < 0 || cost < best_cost || (cost == best_cost && ctas > best_ctas)) {
                    best_cost = cost; best_kw = kw; best_s = (int)S; best_ctas = ctas; best_ns = (int)ns;
                }
            };
            const size_t smem_res = fixed + tile;
            if (smem_res <= kSmemCap) {
                consider(0, smem_res, 0);
                continue;
            }
            if (smem_res <= kSmemBig) consider(0, smem_res, 1);    // no overlap with the next launch
            if (fixed + LY::ring_bytes(SLOT, 1) > kSmemCap) continue;
            int64_t ns = (int64_t)((kSmemCap - fixed) / LY::ring_bytes(SLOT, 1));
            if (ns > per_warp) ns = per_warp;
            if (ns > gtc::NSMAX) ns = gtc::NSMAX;
            if (ns < 2 && per_warp >= 2) continue;                    // no overlap of copies and decoding
            // small copies stream slower than one copy per row (measured: about one macro block at one
            // token, three with more)
            consider(ns, LY::bytes((int)kseg, UNIT, M, SLOT, (int)ns) + LY::red_bytes((int)S, 8 / kw), M > 1 ? 3 : 1);
        }
    }
    if (best_cost < 0) return -3;                                     // caller splits the tokens
    // A ring with several column groups streams slower than two launches on halves of the tokens with
    // resident tiles (measured: ffn_down 2560x9728 Q6_K at 7 tokens 25.6 us as a ring); for matrices
    // up to 64 MB the caller halves the tokens instead.
    if (NT > 1 && best_ns > 0 && total_rows * row_bytes(QT, K) < ((int64_t)64 << 20)) return -3;
    // 9-16 binary32 tokens (hi + lo: 32 MMA columns) stage as many activation bytes per K as the tile holds
    // weight bytes, so no split of a large matrix fits two CTAs per SM; for the 2-5-bit types two launches
    // of up to 8 tokens, the second finding the weights in L2, measured faster there (9728 x 2560 at 16
    // tokens: Q4_K 31.3 -> 23.2 us, Q4_0 28.6 -> 20.6, Q2_K 29.8 -> 23.8, Q5_0 32.2 -> 27.7), and slower for
    // Q3_K, Q6_K and Q8_0, which stay one launch, as do small matrices.
    constexpr bool kHalve16 = QT == T_Q4_0 || QT == T_Q4_1 || QT == T_Q5_0 || QT == T_Q5_1 || QT == T_Q2_K ||
                              QT == T_Q4_K || QT == T_Q5_K;
    if (kHalve16 && NT == 4 && !XBF16 && total_rows * K >= ((int64_t)16 << 20)) return -3;
    if (dry) return 0;                                                // planning only (launch counting)
    const int64_t kseg = ((nmacro + best_s - 1) / best_s) * 256;
    if constexpr (KWMAX >= 8) if (best_kw == 8) return launch_gtc_kw<QT, NT, XBF16, 8>(ms, K, x, M, best_s, kseg, best_ns, status, st, stall, early);
    if constexpr (KWMAX >= 4) if (best_kw == 4) return launch_gtc_kw<QT, NT, XBF16, 4>(ms, K, x, M, best_s, kseg, best_ns, status, st, stall, early);
    if constexpr (KWMAX >= 2) if (best_kw == 2) return launch_gtc_kw<QT, NT, XBF16, 2>(ms, K, x, M, best_s, kseg, best_ns, status, st, stall, early);
    return launch_gtc_kw<QT, NT, XBF16, 1>(ms, K, x, M, best_s, kseg, best_ns, status, st, stall, early);
}

struct GtcLaunch {
    bool xbf16;
    const MatSet *ms;
    int64_t K;
    const void *x;
    int M;
    unsigned int *status;
    cudaStream_t st;
    bool dry;
    int stall, early;
    template <int QT> int operator()() {
        if constexpr (QT <= T_BF16) {
            return -1;
        } else {
            if (xbf16) return M <= 8 ? launch_gtc_t<QT, 1, true>(*ms, K, x, M, status, st, dry, stall, early)
                                     : launch_gtc_t<QT, 2, true>(*ms, K, x, M, status, st, dry, stall, early);
            if (M <= 4) return launch_gtc_t<QT, 1, false>(*ms, K, x, M, status, st, dry, stall, early);
            if (M <= 8) return launch_gtc_t<QT, 2, false>(*ms, K, x, M, status, st, dry, stall, early);
            return launch_gtc_t<QT, 4, false>(*ms, K, x, M, status, st, dry, stall, early);
        }
    }
};

// ---- expert-indexed launches
template <int QT, int NT, bool XBF16, int KW>
int launch_gtc_id_kw(const gtc::IdExperts &ex, int E, int64_t N, int64_t K, const void *x, int xdiv, const int32_t *ids,
                     int M, int topk, float *y, int S, int64_t kseg, size_t smem, unsigned int *status, cudaStream_t st) {
    using LY = gtc::Layout<NT, XBF16>;
    constexpr int RG = LY::WARPS / KW;
    auto kern = gtc::gemv_tc_id_kernel<QT, NT, XBF16, KW>;
    static bool attr_set[kMaxDevices] = {};
    const int devi = current_device_index();
    if (!attr_set[devi]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemCap) != cudaSuccess)
            return -6;
        attr_set[devi] = true;
    }
    const int64_t dmax = (int64_t)M * topk < E ? (int64_t)M * topk : E;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + 16 * RG - 1) / (16 * RG)), (unsigned)S, (unsigned)dmax);
    cfg.blockDim = dim3(LY::WARPS * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ex, E, (int)N, K, row_bytes(QT, K), x, xdiv, ids, M, topk, y,
                                       (int)kseg, status);
    return e == cudaSuccess ? 0 : -6;
}

// Work split of the expert-indexed kernel: the per-expert matrices are narrow (K of a few macro blocks), so
// the split takes the K slices per CTA and K segments per cluster (at most 4) that minimise waves x (macro
// blocks per warp + a per-CTA prologue), over CTAs of every possible expert (those of absent experts leave
// at once), with the whole row-block tile resident in shared memory. Returns -3 when no split fits.
template <int QT, int NT, bool XBF16>
int launch_gtc_id_t(const gtc::IdExperts &ex, int E, int64_t N, int64_t K, const void *x, int xdiv, const int32_t *ids,
                    int M, int topk, float *y, unsigned int *status, cudaStream_t st) {
    using LY = gtc::Layout<NT, XBF16>;
    constexpr int UNIT = gtc::Frag<QT>::UNIT, TOK = LY::TOK;
    constexpr int MB_BYTES = 256 / TypeInfo<QT>::QK * TypeInfo<QT>::BYTES;
    constexpr int KWMAX = NT == 1 ? 8 : ((NT == 2 && !XBF16) ? 2 : 1);
    const int64_t ngroups = (N + 15) / 16, nmacro = (K + 255) / 256;
    const int nslot = M * topk;
    const int64_t dmax = nslot < E ? nslot : E;
    const int nsm = device_sm_count();
    int best_kw = 0, best_s = 1;
    int64_t best_cost = -1;
    size_t best_smem = 0;
    for (int kw = 1; kw <= KWMAX; kw *= 2) {
        if (kw > nmacro) break;
        const int rg = 8 / kw;
        const int64_t nrb = (ngroups + rg - 1) / rg;
        for (int S = 1; S <= 4 && S <= nmacro; ++S) {
            const int64_t kseg = ((nmacro + S - 1) / S) * 256;
            if ((K + kseg - 1) / kseg != S) continue;
            const size_t smem = LY::BARS + LY::tile_bytes(rg, (int)(kseg / 256 * MB_BYTES)) +
                                LY::xbytes((int)kseg, UNIT, TOK) + LY::red_bytes(S, rg) +
                                (((size_t)nslot * 4 + QMM_MAX_EXPERTS + 15) & ~(size_t)15);
            if (smem > kSmemCap) continue;
            const int64_t per_warp = (kseg / 256 + kw - 1) / kw;
            // CTAs of every possible expert, two per SM; each wave also pays the routing prologue
            const int64_t ctas = nrb * S * dmax;
            const int64_t waves = (ctas + 2 * nsm - 1) / (2 * nsm);
            const int64_t cost = 4 * waves * (per_warp + 3) + (S > 1 ? 4 : 0);
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost; best_kw = kw; best_s = S; best_smem = smem;
            }
        }
    }
    if (best_cost < 0) return -3;
    const int64_t kseg = ((nmacro + best_s - 1) / best_s) * 256;
    if constexpr (KWMAX >= 8) if (best_kw == 8) return launch_gtc_id_kw<QT, NT, XBF16, 8>(ex, E, N, K, x, xdiv, ids, M, topk, y, best_s, kseg, best_smem, status, st);
    if constexpr (KWMAX >= 4) if (best_kw == 4) return launch_gtc_id_kw<QT, NT, XBF16, 4>(ex, E, N, K, x, xdiv, ids, M, topk, y, best_s, kseg, best_smem, status, st);
    if constexpr (KWMAX >= 2) if (best_kw == 2) return launch_gtc_id_kw<QT, NT, XBF16, 2>(ex, E, N, K, x, xdiv, ids, M, topk, y, best_s, kseg, best_smem, status, st);
    return launch_gtc_id_kw<QT, NT, XBF16, 1>(ex, E, N, K, x, xdiv, ids, M, topk, y, best_s, kseg, best_smem, status, st);
}

struct GtcIdLaunch {
    bool xbf16;
    const gtc::IdExperts *ex;
    int E;
    int64_t N, K;
    const void *x;
    int xdiv;
    const int32_t *ids;
    int M, topk;
    float *y;
    unsigned int *status;
    cudaStream_t st;
    template <int QT> int operator()() {
        if constexpr (QT <= T_BF16) {
            return -3;
        } else {
            // one 4-token (8 for bf16 activations) column group per pass: an expert rarely gets more
            if (xbf16) return launch_gtc_id_t<QT, 1, true>(*ex, E, N, K, x, xdiv, ids, M, topk, y, status, st);
            return launch_gtc_id_t<QT, 1, false>(*ex, E, N, K, x, xdiv, ids, M, topk, y, status, st);
        }
    }
};

}  // namespace

// M <= 16 tokens (bigger M is split into groups of 16 by the caller). Returns -3 when the K segments a
// cluster allows cannot hold the activations of this many tokens (the caller then halves the group).
// dry: plan only, launch nothing (0 or -3), for counting launches.
int launch_gemv_tc(int qt, bool xbf16, const void *wq, int64_t N, int64_t K, const void *x, int M, float *y,
                   unsigned int *status, cudaStream_t st, bool dry, int stall, bool early) {
    MatSet ms = {};
    ms.count = 1;
    ms.wq[0] = wq;
    ms.N[0] = N;
    ms.y[0] = y;
    GtcLaunch f{xbf16, &ms, K, x, M, status, st, dry, stall, early ? 1 : 0};
    return dispatch_type(qt, f);
}

// Several matrices of one type and K sharing x in one launch (M <= 16; the matrices' outputs y[i] are
// M x N[i]). Returns -3 when no work split fits on chip for this many tokens.
int launch_gemv_tc_multi(int qt, bool xbf16, const MatSet &ms, int64_t K, const void *x, int M,
                         unsigned int *status, cudaStream_t st, bool dry, bool early) {
    GtcLaunch f{xbf16, &ms, K, x, M, status, st, dry, 0, early ? 1 : 0};
    return dispatch_type(qt, f);
}

// Expert-indexed product on the tensor-core mat-vec machinery (quantized types). Returns -3 when it does
// not apply (plain types, or no work split fits on chip); the caller then uses the CUDA-core kernel.
int launch_gemv_tc_id(int qt, bool xbf16, const void *const *wq, int64_t E, int64_t N, int64_t K, const void *x,
                      bool x_per_slot, const int32_t *ids, int64_t M, int topk, float *y, unsigned int *status,
                      cudaStream_t st) {
    gtc::IdExperts ex;
    for (int e = 0; e < QMM_MAX_EXPERTS; ++e) ex.p[e] = e < E ? static_cast<const uint8_t *>(wq[e]) : nullptr;
    GtcIdLaunch f{xbf16, &ex, (int)E, N, K, x, x_per_slot ? 1 : topk, ids, (int)M, topk, y, status, st};
    return dispatch_type(qt, f);
}

}  // namespace wqk


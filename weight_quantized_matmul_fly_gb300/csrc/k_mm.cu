// Tensor-core path for larger token counts: y = x * dequant(W)^T on tcgen05 with a TMEM accumulator.
//
// The method (candle PR 4056, "Metal: 64-token tile for the quantized matrix-matrix kernel", section "Why
// the tile sets the weight reuse"): a thread block owns a slab of weight rows; at every step along K it
// reads those rows' quantized blocks, dequantizes them into shared memory and multiplies them by every
// token it holds, so each weight is fetched and dequantized once per token tile. Here:
//   - a CTA owns BM = 128 weight rows (the MMA's M) and J token tiles of T = 32, 64 or 128 tokens (the
//     MMA's N), J*T <= 256, or 512 for large M (the whole tensor memory); the J tiles share every decoded
//     slab, so a larger J*T divides the decoding work per multiply-add (J = 1..6 or 8, only as many tiles
//     as the tokens need);
//   - warp 0 loads the J*T x 64 activation tile of each K step by TMA (rows past M read as zero): bf16
//     straight into the operand stage, or binary32 into a staging slot from which the decoder group of
//     that step rounds it to bf16 into the operand stage (no separate conversion pass);
//   - warps 2..17 decode the 128 x 64 weight slab of each step to bf16 (round to nearest even of the
//     binary32 value) straight into the 128-byte-swizzled K-major layout tcgen05 reads; they form two
//     groups of 8 that take alternate K steps, so each keeps the raw bytes of its next two steps (four K
//     steps ahead) in flight and twice as many warps hide the load latency;
//   - warp 1 issues, per step, 4 (K = 16) tcgen05.mma of N = min(J*T, 256) tokens (two at 512) into TMEM
//     and commits them to the stage's "empty" barrier, which hands the stage back to the producer and the
//     decoders;
//   - the decoder warps then read TMEM with tcgen05.ld and write y; when K is split over S CTAs they form
//     a thread block cluster and add their partial tiles in split order through distributed shared
//     memory, so a call is one kernel and needs no scratch.
// Bit-identity across T: every output element sees the same K steps, the same K=16 MMAs in the same
// order and the same K split whatever T is (candle PR 4056, section "Same results, bit for bit").
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "mm_slab.cuh"

namespace wqk {
namespace mm {

struct Smem {
    uint64_t full_b[MAX_STAGES], full_a[MAX_STAGES], empty[MAX_STAGES], done;
    uint64_t xfull[MAX_XSLOTS], xempty[MAX_XSLOTS];
    uint32_t tmem;
    int abort;
};

// y = x * dequant(W)^T for a 128-row block, TN = T*J token columns and one K split of the work plan.
//   XF32 = false: x is bfloat16 (the caller's, or the bf16 copy of binary32 activations); warp 0 loads the
//                 activation tile of each K step straight into the operand stage by TMA (128-byte swizzle).
//   XF32 = true:  x is binary32; warp 0 loads its tile by TMA into a ring of staging slots, and the decoder
//                 group that decodes the K step's weights also rounds the step's activations to bfloat16
//                 (nearest even) into the operand stage, so no separate conversion pass is needed.
// When K is split over S CTAs (gridDim.z = S > 1), the partial tiles are added in split order in one of two
// ways, with the same result bit for bit:
//   part == nullptr: the S CTAs of an output tile form a thread block cluster; each stores its binary32
//     partial tile into its own shared memory and, after a cluster barrier, rank r adds the S partials of
//     its share of the tile's columns in rank (= split) order and writes y: no scratch, no second kernel;
//   part != nullptr: each CTA writes its partial tile to part + split * split_stride (M x N binary32), and a
//     second kernel adds them in split order. Measured faster when the kernel follows the separate bf16
//     conversion pass of x (a cluster launch starts later behind a kernel that is not one).
template <int QT, int T, int J, bool XF32>
__global__ void __launch_bounds__(THREADS, 1)
    mm_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint8_t *__restrict__ wq, int N, int64_t K,
              int64_t rowbytes, int M, float *__restrict__ y, int ksteps_per_split, float *__restrict__ part,
              int64_t split_stride, int early, unsigned int *status) {
    constexpr int TN = T * J;
    constexpr int STAGES = stages_of(TN, XF32);
    constexpr int XSLOTS = xslots_of(TN, XF32);
    constexpr uint32_t TMEM_COLS = TN <= 32 ? 32 : (TN <= 64 ? 64 : (TN <= 128 ? 128 : (TN <= 256 ? 256 : 512)));
    // One MMA covers up to 256 token columns (all J tiles of T at once; the tiles are contiguous in
    // shared memory and in TMEM): N = MN per instruction, NMMA instructions per K = 16.
    constexpr int MN = TN > 256 ? 256 : TN, NMMA = TN / MN;
    static_assert(MN % 16 == 0 && TN % MN == 0, "MMA N");
    static_assert(!XF32 || TN <= 128, "binary32 activations are converted in-kernel up to 128 token columns");
    static_assert(smem_bytes(TN, XF32) <= 227 * 1024, "shared memory of one CTA");
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, MN);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    uint8_t *sX = sB + STAGES * b_stage_bytes(TN);              // binary32 staging slots (XF32)
    Smem *sm = reinterpret_cast<Smem *>(sX + XSLOTS * x_slot_bytes(TN));
    float *red = reinterpret_cast<float *>(smem);              // after the main loop: this CTA's partial tile

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * TN;
    const int S = (int)gridDim.z, split = blockIdx.z;
    const int ktotal = (int)((K + BK - 1) / BK);
    const int kbeg = split * ksteps_per_split;
    const int kend = (kbeg + ksteps_per_split < ktotal) ? kbeg + ksteps_per_split : ktotal;
    const int nsteps = kend > kbeg ? kend - kbeg : 0;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&sm->full_b[s], 1);
            ptx::mbar_init(&sm->full_a[s], 8);   // the 8 warps of the group that decodes this step
            ptx::mbar_init(&sm->empty[s], 1);
        }
        for (int j = 0; j < XSLOTS; ++j) {
            ptx::mbar_init(&sm->xfull[j], 1);
            ptx::mbar_init(&sm->xempty[j], 8);   // the 8 warps of the group that converted the slot
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

    // Programmatic dependent launch: the next kernel in the stream may start its prologue now; it waits
    // for this grid's completion before touching memory this grid writes.
    asm volatile("griddepcontrol.launch_dependents;");
    if (warp == 0) {
        // ---------------- activation producer: the activations may come from the preceding kernel, so
        // they are loaded only after it has completed
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (lane == 0) {
            constexpr int NB = XF32 ? XSLOTS : STAGES;     // ring the loads go to
            int issued = 0;
            for (int i = 0; i < nsteps; ++i) {
                const int s = i % NB;
                uint64_t *freed = XF32 ? &sm->xempty[s] : &sm->empty[s];
                if (i >= NB && !ptx::mbar_wait(freed, ((i / NB) - 1) & 1, status)) {
                    sm->abort = 1;
                    break;
                }
                if (*(volatile int *)&sm->abort) break;
                if constexpr (XF32) {
                    ptx::mbar_arrive_expect_tx(&sm->xfull[s], (uint32_t)x_slot_bytes(TN));
                    ptx::tma_load_2d(sX + s * x_slot_bytes(TN), &tmap_x, (kbeg + i) * BK, m0, &sm->xfull[s]);
                } else {
                    ptx::mbar_arrive_expect_tx(&sm->full_b[s], (uint32_t)b_stage_bytes(TN));
                    // a tensor-map box has at most 256 rows: 512 tokens take two boxes
#pragma unroll
                    for (int q = 0; q < (TN > 256 ? TN / 256 : 1); ++q)
                        ptx::tma_load_2d(sB + s * b_stage_bytes(TN) + q * 256 * 128, &tmap_x, (kbeg + i) * BK,
                                         m0 + 256 * q, &sm->full_b[s]);
                }
                issued = i + 1;
            }
            // every requested tile lands before the CTA may go on (its shared memory is reused below)
            for (int i = (issued > NB ? issued - NB : 0); i < issued; ++i)
                ptx::mbar_wait(XF32 ? &sm->xfull[i % NB] : &sm->full_b[i % NB], (i / NB) & 1, status);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t sA_u32 = ptx::smem_u32(sA), sB_u32 = ptx::smem_u32(sB);
            for (int i = 0; i < nsteps; ++i) {
                const int s = i % STAGES;
                const uint32_t par = (i / STAGES) & 1;
                if (!ptx::mbar_wait(&sm->full_a[s], par, status) ||
                    (!XF32 && !ptx::mbar_wait(&sm->full_b[s], par, status))) {
                    sm->abort = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t adesc = ptx::sw128_desc(sA_u32 + s * A_STAGE);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
                    for (int jj = 0; jj < NMMA; ++jj) {
                        const uint64_t bdesc = ptx::sw128_desc(sB_u32 + s * b_stage_bytes(TN) + jj * MN * 128);
                        // advancing 16 bf16 = 32 bytes inside the swizzle row moves the start address by 2 units
                        ptx::mma_bf16(tmem + jj * MN, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (i | kk) != 0);
                    }
                }
                ptx::mma_commit(&sm->empty[s]);
            }
            ptx::mma_commit(&sm->done);   // tracks every MMA issued above
        }
    } else {
        // ---------------- decoders: group grp decodes the K steps i = grp (mod NGRP); within a group warp
        // dw handles rows 16dw .. 16dw+15 of the slab; lane -> (row, chunk)
        const int d = warp - 2;
        const int grp = d >> 3, dw = d & 7;
        const int r_local = 16 * dw + (lane >> 1), h = lane & 1;
        const int row = n0 + r_local;
        const bool row_ok = row < N;
        const uint8_t *wrow = wq + (int64_t)(row_ok ? row : N - 1) * rowbytes;
        const int nchunks = (int)((K + 31) / 32);
        const uint32_t sA_u32 = ptx::smem_u32(sA), sB_u32 = ptx::smem_u32(sB);
        using SL = Slab<QT>;
        // Before waiting for the preceding kernel, this row's weights of the split are only prefetched into
        // L2 (coherent, so never stale even if that kernel wrote them); they are read after the wait. With
        // `early` (the caller states that the preceding kernel does not write the weights) the decoders
        // start reading them at once, overlapping the end of that kernel.
        if (!early && h == 0 && grp == 0 && row_ok && nsteps > 0) {
            const int64_t cb = (int64_t)kbeg * BK / TypeInfo<QT>::QK, ce = (int64_t)kend * BK / TypeInfo<QT>::QK;
            const int64_t nb = K / TypeInfo<QT>::QK;
            const uintptr_t a = reinterpret_cast<uintptr_t>(wrow + cb * TypeInfo<QT>::BYTES);
            const uintptr_t e = reinterpret_cast<uintptr_t>(wrow + (ce < nb ? ce : nb) * TypeInfo<QT>::BYTES);
            const uintptr_t wend = reinterpret_cast<uintptr_t>(wq + (int64_t)N * rowbytes);
            const uintptr_t a0 = a & ~(uintptr_t)15;
            uintptr_t e1 = (e + 15) & ~(uintptr_t)15;
            if (e1 > wend) e1 = wend & ~(uintptr_t)15;
            if (e1 > a0) ptx::prefetch_l2(reinterpret_cast<const void *>(a0), (uint32_t)(e1 - a0));
        }
        if (!early) asm volatile("griddepcontrol.wait;" ::: "memory");
        // raw bytes of the group's next PFT K steps are in flight while a step is decoded (rw[0] is the
        // step being decoded, rw[PFT] the one requested during it)
        constexpr int PFT = pf_of<QT>();
        typename SL::Raw rw[PFT + 1];
        if constexpr (SL::FAST) {
            const int c0 = 2 * (kbeg + grp) + h;
#pragma unroll
            for (int j = 0; j < PFT; ++j)
                if (grp + j * NGRP < nsteps && c0 + 2 * j * NGRP < nchunks) SL::load(rw[j], wrow, c0 + 2 * j * NGRP);
        }
        for (int i = grp; i < nsteps; i += NGRP) {
            const int s = i % STAGES;
            const int c = 2 * (kbeg + i) + h;
            if constexpr (SL::FAST) {
                if (i + PFT * NGRP < nsteps && c + 2 * PFT * NGRP < nchunks)
                    SL::load(rw[PFT], wrow, c + 2 * PFT * NGRP);
            }
            if (i >= STAGES && !ptx::mbar_wait(&sm->empty[s], ((i / STAGES) - 1) & 1, status)) {
                sm->abort = 1;
                break;
            }
            if (*(volatile int *)&sm->abort) break;
            uint32_t o[16];
            if (row_ok && c < nchunks) {
                if constexpr (SL::FAST) {
                    SL::decode(rw[0], c, o);
                } else {
                    float w[32];
                    decode_chunk<QT>(wrow, c, K, w);
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = pack_bf16x2(w[2 * j], w[2 * j + 1]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) o[j] = 0u;
            }
            const uint32_t a_base = sA_u32 + s * A_STAGE;
#pragma unroll
            for (int p = 0; p < 4; ++p)
                ptx::st_shared_v4(a_base + sw128_off(r_local, 4 * h + p), o[4 * p], o[4 * p + 1], o[4 * p + 2],
                                  o[4 * p + 3]);
            if constexpr (XF32) {
                // this step's activations: binary32 staging slot -> bf16 operand stage, 8 columns (one 16-byte
                // piece of the swizzled row) per thread and pass; rows past M were read as zero by the TMA
                const int xs = i % XSLOTS;
                if (!ptx::mbar_wait(&sm->xfull[xs], (i / XSLOTS) & 1, status)) {
                    sm->abort = 1;
                    break;
                }
                const float *xsrc = reinterpret_cast<const float *>(sX + xs * x_slot_bytes(TN));
                const uint32_t b_base = sB_u32 + s * b_stage_bytes(TN);
                const int gt = 32 * dw + lane;              // thread index within the group
#pragma unroll
                for (int pc = gt; pc < TN * 8; pc += 256) {
                    const int rr = pc >> 3, pp = pc & 7;
                    const float4 a = *reinterpret_cast<const float4 *>(xsrc + rr * BK + 8 * pp);
                    const float4 b = *reinterpret_cast<const float4 *>(xsrc + rr * BK + 8 * pp + 4);
                    ptx::st_shared_v4(b_base + sw128_off(rr, pp), pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                      pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm->xempty[xs]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm->full_a[s]);
            if constexpr (SL::FAST) {
#pragma unroll
                for (int j = 0; j < PFT; ++j) rw[j] = rw[j + 1];
            }
        }
    }

    // ---------------- epilogue: TMEM lanes = weight rows, columns = tokens. Every MMA has completed once
    // `done` has; the operand stages are then free (the producer waited for all its loads above).
    constexpr int PARTS = NDEC / 4;             // warps per TMEM lane quarter; they split the columns
    const bool dec = warp >= 2;
    const int q = warp & 3;                     // TMEM lane quarter this warp may access
    const int pw = part_of(warp);               // (q, pw) runs over all quarters x parts once
    const int r = 32 * q + lane;                // row within the block
    // y (and the scratch partials) are written only once the preceding kernel has completed; with the split
    // added inside the cluster every thread writes y
    if (dec || (S > 1 && !part)) asm volatile("griddepcontrol.wait;" ::: "memory");
    bool ok = true;
    if (dec && nsteps > 0) {
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&sm->done, 0, status) && !*(volatile int *)&sm->abort);
        ptx::tc_fence_after();
    }
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    if (S == 1) {
        if (dec && ok) {
            for (int c0 = 16 * pw; c0 < TN; c0 += 16 * PARTS) {
                uint32_t v[16];
                if (nsteps > 0) {
                    ptx::tmem_ld_32x32b_x16(lane_base + c0, v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0u;       // an empty K range contributes zeros
                }
                if (n0 + r < N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = m0 + c0 + j;
                        if (tok < M) y[(int64_t)tok * N + n0 + r] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    } else if (part) {
        float *py = part + (int64_t)split * split_stride;
        if (dec) {
            for (int c0 = 16 * pw; c0 < TN; c0 += 16 * PARTS) {
                uint32_t v[16];
                if (nsteps > 0 && ok) {
                    ptx::tmem_ld_32x32b_x16(lane_base + c0, v);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0u;
                }
                if (n0 + r < N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = m0 + c0 + j;
                        if (tok < M) py[(int64_t)tok * N + n0 + r] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    } else {
        // every load the producer issued has landed before the operand stages are reused
        __syncthreads();
        // K split over the cluster: rounds of RC columns. Each CTA stores its partial [RC columns][128 rows]
        // into its own (now idle) operand stages; after a cluster barrier, rank `split` adds up, for columns
        // [split*cw, split*cw + cw) of the round, the S partials in rank order and writes y; a second barrier
        // keeps every CTA's shared memory alive until all ranks have read it.
        constexpr int RC = TN > 256 ? 256 : TN;
        const int cw = (RC + S - 1) / S;
        for (int rc0 = 0; rc0 < TN; rc0 += RC) {
            if (dec) {
                for (int c0 = 16 * pw; c0 < RC; c0 += 16 * PARTS) {
                    uint32_t v[16];
                    if (nsteps > 0 && ok) {
                        ptx::tmem_ld_32x32b_x16(lane_base + rc0 + c0, v);
                        ptx::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = 0u;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) red[(c0 + j) * BM + r] = __uint_as_float(v[j]);
                }
            }
            ptx::cluster_sync();
            const int cb = split * cw, ce = cb + cw < RC ? cb + cw : RC;
            for (int e = tid + cb * BM; e < ce * BM; e += THREADS) {
                const int col = e / BM, row = e - col * BM;
                const int tok = m0 + rc0 + col;
                if (tok >= M || n0 + row >= N) continue;
                // the S loads are issued back to back, then added in rank order
                float v[MAX_SPLIT];
#pragma unroll
                for (int qq = 0; qq < MAX_SPLIT; ++qq)
                    if (qq < S) v[qq] = ptx::ld_dsmem_f32(ptx::mapa(red + e, (uint32_t)qq));
                float a = v[0];
#pragma unroll
                for (int qq = 1; qq < MAX_SPLIT; ++qq)
                    if (qq < S) a += v[qq];
                y[(int64_t)tok * N + n0 + row] = a;
            }
            ptx::cluster_sync();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA this CTA issued has completed before its accumulator is freed, also when a bounded
        // wait gave up above (the issuer committed `done` after its last MMA whatever happened)
        if (nsteps > 0) {
            if (lane == 0) ptx::mbar_wait(&sm->done, 0, status);
            __syncwarp();
            ptx::tc_fence_after();
        }
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// y[i] = sum over s of part[s][i], s ascending (the K splits' partial tiles added in split order).
// This kernel and the conversion below let the next kernel in the stream launch at once (it waits for them
// before it touches what they write), so the next tensor-core kernel's prologue and first weight loads
// overlap them; they read their inputs only after the kernel before them has completed.
__global__ void splitk_reduce_kernel(const float4 *__restrict__ part, int64_t stride4, int S, float4 *__restrict__ y,
                                     int64_t n4) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int64_t i = beg + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float a = part[i];
        for (int s = 1; s < S; ++s) a += part[i + s * stride];
        y[i] = a;
    }
}

// binary32 -> bfloat16 (round to nearest even), 8 elements per thread; n is a multiple of 8.
__global__ void x_to_bf16_kernel(const float4 *__restrict__ x, uint4 *__restrict__ out, int64_t n8) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

// Tensor map of the activations: bf16 rows read as 128-byte-swizzled K-major tiles straight into an operand
// stage, or binary32 rows read unswizzled into a staging slot (64 columns = 256 bytes per row). Rows past M
// and columns past K read as zero.
static bool make_x_tmap(CUtensorMap *map, const void *x, bool f32, int64_t M, int64_t K, int rows) {
    auto enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * (f32 ? 4 : 2)};
    const cuuint32_t box[2] = {(cuuint32_t)mm::BK, (cuuint32_t)rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct MmPlan {
    int S;      // K split (CTAs of one cluster)
    int cols;   // token columns per CTA
};

namespace {

// Launch with programmatic stream serialization (the kernel may start while its predecessor in the stream
// finishes; it orders its own memory accesses with griddepcontrol.wait) and, for S > 1, clusters of the S
// CTAs that split one output tile's K range. Returns 0 or -6.
template <typename... Args>
int launch_pdl(const void *kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_z, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (cluster_z > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = (unsigned)cluster_z;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    void *argv[] = {reinterpret_cast<void *>(&args)...};
    return cudaLaunchKernelExC(&cfg, kern, argv) == cudaSuccess ? 0 : -6;
}

// Token tiles per CTA for a plan of `cols` token columns per CTA (128, 256 or 512): cols / T tiles, at most
// 256 columns with 32-token tiles, and not more tiles than the tokens need (a power of two).
inline int tiles_per_cta(int T, int64_t M, int cols) {
    int j = cols / T;
    if (T == 32 && j > 8) j = 8;
    if (j < 1) j = 1;
    const int64_t need = (M + T - 1) / T;
    while (j > 1 && j / 2 >= need) j /= 2;
    // 3, 5 and 6 tiles too, so that a CTA does not multiply up to twice the tokens it holds
    if (j == 4 && need == 3 && T <= 64) j = 3;
    if (j == 8 && need <= 6 && need >= 5 && T == 32) j = (int)need;
    return j;
}

// Sets the kernel's shared-memory attribute once per device. Returns false on failure.
template <int QT, int T, int J, bool XF32>
bool mm_attrs() {
    static bool attr_set[kMaxDevices] = {};
    const int devi = current_device_index();
    if (!attr_set[devi]) {
        auto kern = mm::mm_kernel<QT, T, J, XF32>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mm::smem_bytes(T * J, XF32)) !=
            cudaSuccess)
            return false;
        attr_set[devi] = true;
    }
    return true;
}

template <int QT, int T, int J, bool XF32>
int launch_mm_t(const void *wq, int64_t N, int64_t K, const void *x, int64_t M, float *y, int S, int kps, float *part,
                int64_t split_stride, int early, unsigned int *status, cudaStream_t st) {
    constexpr int TN = T * J;
    CUtensorMap map;
    if (!make_x_tmap(&map, x, XF32, M, K, TN > 256 ? 256 : TN)) return -6;
    if (!mm_attrs<QT, T, J, XF32>()) return -6;
    auto kern = mm::mm_kernel<QT, T, J, XF32>;
    dim3 grid((unsigned)((N + mm::BM - 1) / mm::BM), (unsigned)((M + TN - 1) / TN), (unsigned)S);
    const int64_t rb = row_bytes(QT, K);
    const uint8_t *w8 = static_cast<const uint8_t *>(wq);
    const int Ni = (int)N, Mi = (int)M;
    return launch_pdl(reinterpret_cast<const void *>(kern), grid, dim3(mm::THREADS),
                      (size_t)mm::smem_bytes(TN, XF32), st, part ? 1 : S, map, w8, Ni, K, rb, Mi, y, kps, part,
                      split_stride, early, status);
}

struct MmLaunch {
    int tile, J;
    bool xf32;
    const void *wq;
    int64_t N, K;
    const void *x;
    int64_t M;
    float *y;
    int S, kps;
    float *part;
    int64_t split_stride;
    int early;
    unsigned int *status;
    cudaStream_t st;
    template <int QT, int T, int JJ> int go_j() {
        constexpr int TN = T * JJ;
        constexpr bool shape_ok = (TN <= 256 && ((JJ & (JJ - 1)) == 0 || T == 32 || (T == 64 && JJ == 3))) ||
                                  (T >= 64 && TN <= 512 && (JJ & (JJ - 1)) == 0);
        if constexpr (!shape_ok) {
            return -7;
        } else {
            if (!xf32)
                return launch_mm_t<QT, T, JJ, false>(wq, N, K, x, M, y, S, kps, part, split_stride, early, status, st);
            if constexpr (TN <= 128)
                return launch_mm_t<QT, T, JJ, true>(wq, N, K, x, M, y, S, kps, part, split_stride, early, status, st);
            return -7;
        }
    }
    template <int QT, int T> int go() {
        switch (J) {
        case 1: return go_j<QT, T, 1>();
        case 2: return go_j<QT, T, 2>();
        case 3: return go_j<QT, T, 3>();
        case 4: return go_j<QT, T, 4>();
        case 5: return go_j<QT, T, 5>();
        case 6: return go_j<QT, T, 6>();
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

// CTAs of the tensor-core kernel resident at once when launched in clusters of S (every instance runs one
// CTA per SM; a cluster must fit in one GPC, which can strand SMs), queried once per device and S.
int64_t mm_capacity(int S) {
    static int64_t cache[kMaxDevices][mm::MAX_SPLIT + 1] = {};
    const int dev = current_device_index();
    if (S < 1 || S > mm::MAX_SPLIT) return 0;
    if (cache[dev][S]) return cache[dev][S];
    int64_t cap = device_sm_count();
    if (S > 1) {
        auto kern = mm::mm_kernel<T_Q4_0, 32, 4, false>;
        int nclusters = 0;
        if (mm_attrs<T_Q4_0, 32, 4, false>()) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, 1, (unsigned)S);
            cfg.blockDim = dim3(mm::THREADS);
            cfg.dynamicSmemBytes = (size_t)mm::smem_bytes(128, false);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = (unsigned)S;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess) nclusters = 0;
        }
        // unknown (no device): assume a cluster packs as well as single CTAs
        cap = nclusters > 0 ? (int64_t)nclusters * S : (device_sm_count() / S) * S;
    }
    cache[dev][S] = cap;
    return cap;
}

}  // namespace

// Work plan of the tensor-core path: the K split S and the token columns per CTA (128, 256 or 512), a
// function of (type, N, K, M) and of how a split is added (inside a cluster or by a second kernel) only,
// never of the token tile, so that every tile variant adds the same partial sums in the same order. CTAs of
// 128 rows run one per SM. With `cluster` the S CTAs of a split form a cluster (S <= 8), and a wave holds as
// many of them as the clusters that fit at once; otherwise S <= 32 and a wave is one CTA per SM. The plan
// minimises the modelled time
//     waves * (t_wave + ksteps_per_split * t_step(cols, type))  +  2 S M N * 4 bytes / 6 TB/s  (S > 1)
// A K step (64 weights) of a CTA costs 0.45 / 0.49 / 0.71 us at 128 / 256 / 512 columns for 4-bit K-quants
// (fitted to a GB300 sweep of every split and column count over the seven Qwen3-Embedding-4B projections at
// 128, 512 and 2048 tokens; the weight decoding, not the tensor core, sets the pace below 512 columns), 1.7
// times that for Q6_K; a wave costs about 1.4 us to start and drain; the last term charges the partial
// tiles (moved through shared memory and read across the cluster), which measured as costly as writing
// and reading them through HBM: without it, plans with several splits at 512 columns ran 1.2-1.6 times
// slower than the unsplit ones. Splits keep at least 4 K steps each and leave no split empty.
MmPlan mm_plan(int qt, int64_t N, int64_t K, int64_t M, bool cluster) {
    const int64_t ksteps = (K + mm::BK - 1) / mm::BK;
    const int64_t rowblocks = (N + mm::BM - 1) / mm::BM;
    const double t_wave = 1.4, hbm_bytes_per_us = 6.0e6;
    const double type_factor = qt == T_Q6_K ? 1.7 : 1.0;
    MmPlan best{1, 128};
    double best_t = -1.0;
    for (int cols : {128, 256, 512}) {
        if (cols > 128 && cols / 2 >= M) break;      // more columns than the tokens need
        const double t_step = type_factor * (cols == 128 ? 0.45 : (cols == 256 ? 0.49 : 0.71));
        const int64_t ctas1 = rowblocks * ((M + cols - 1) / cols);
        for (int S = 1; S <= (cluster ? mm::MAX_SPLIT : 32); ++S) {
            const int64_t kps = (ksteps + S - 1) / S;
            if (S > 1 && (ksteps / S < 4 || (S - 1) * kps >= ksteps)) continue;
            const int64_t cap = cluster ? mm_capacity(S) : device_sm_count();
            if (cap <= 0) continue;
            const int64_t waves = (ctas1 * S + cap - 1) / cap;
            double t = (double)waves * (t_wave + (double)kps * t_step);
            if (S > 1) t += 2.0 * S * (double)M * (double)N * 4.0 / hbm_bytes_per_us;
            if (best_t < 0 || t < best_t * 0.98) { best_t = t; best = MmPlan{S, cols}; }
        }
    }
    return best;
}

int mm_ksplit(int qt, int64_t N, int64_t K, int64_t M, bool cluster) { return mm_plan(qt, N, K, M, cluster).S; }

// Token columns per CTA of the plan (128, 256 or 512).
int mm_plan_cols(int qt, int64_t N, int64_t K, int64_t M, bool cluster) { return mm_plan(qt, N, K, M, cluster).cols; }

// Partial tiles of the K splits in scratch are M*N binary32 each, padded to a multiple of 4 elements so that
// every split starts 16-byte aligned.
static inline int64_t split_stride_of(int64_t M, int64_t N) { return (M * N + 3) & ~(int64_t)3; }

// Bytes of scratch for the K splits' partial tiles (0 when the plan does not split K).
size_t mm_partial_bytes(int qt, int64_t N, int64_t K, int64_t M) {
    const int S = mm_ksplit(qt, N, K, M, false);
    return S > 1 ? (size_t)S * (size_t)split_stride_of(M, N) * 4 : 0;
}

// x: M x K, bfloat16 (x_f32 false) or binary32 (x_f32 true, converted inside the kernel: the plan's columns
// are then capped at 128), row stride a multiple of 16 bytes, 16-byte aligned. y: M x N binary32. `part`:
// scratch of mm_partial_bytes() for the K splits' partial tiles (then the plan is the unclustered one), or
// nullptr to add them inside a cluster (the clustered plan).
int launch_mm(int qt, int tile, const void *wq, int64_t N, int64_t K, const void *x, bool x_f32, int64_t M,
              float *y, float *part, bool early, unsigned int *status, cudaStream_t st) {
    const MmPlan plan = mm_plan(qt, N, K, M, part == nullptr);
    const int S = plan.S;
    const int cols = x_f32 && plan.cols > 128 ? 128 : plan.cols;
    const int64_t ksteps = (K + mm::BK - 1) / mm::BK;
    const int kps = (int)((ksteps + S - 1) / S);
    if (S == 1) part = nullptr;
    const int64_t sstride = split_stride_of(M, N);
    MmLaunch f{tile, tiles_per_cta(tile, M, cols), x_f32, wq, N, K, x, M, y, S, kps, part, sstride, early ? 1 : 0,
               status, st};
    int rc = dispatch_type(qt, f);
    if (rc || !part) return rc;
    const int64_t n = M * N, n4 = n / 4;
    if (n4 > 0) {
        int64_t blocks = (n4 + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        const float4 *p4 = reinterpret_cast<const float4 *>(part);
        float4 *y4 = reinterpret_cast<float4 *>(y);
        const int64_t s4 = sstride / 4;
        if (launch_pdl(reinterpret_cast<const void *>(mm::splitk_reduce_kernel), dim3((unsigned)blocks), dim3(256), 0,
                       st, 1, p4, s4, S, y4, n4))
            return -6;
    }
    if (n % 4) {
        const float *pc = part;
        const int64_t beg = n4 * 4;
        if (launch_pdl(reinterpret_cast<const void *>(mm::splitk_reduce_tail_kernel), dim3(1), dim3(32), 0, st, 1, pc,
                       sstride, S, y, beg, n))
            return -6;
    }
    return 0;
}

int launch_x_to_bf16(const float *x, void *out, int64_t n, cudaStream_t st) {
    const int64_t n8 = n / 8;
    const int threads = 256;
    int64_t blocks = (n8 + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    uint4 *o4 = static_cast<uint4 *>(out);
    return launch_pdl(reinterpret_cast<const void *>(mm::x_to_bf16_kernel), dim3((unsigned)blocks), dim3(threads), 0,
                      st, 1, x4, o4, n8);
}

}  // namespace wqk

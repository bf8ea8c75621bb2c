// Expert-indexed product on the tensor cores, for many routed tokens per expert (MUL_MAT_ID at prefill
// sizes; llama.cpp PR 28086, "metal : fix idle threads in mul_mv_iq3_xxs for ne00 < 1024", sections
// "Overview" and "Test methodology": one product per (token, routed expert)):
//     y[(t*topk + j)*N + n] = sum_k dequant(W_e)[n, k] * x[r*K + k],  e = ids[t*topk + j],
// r = t (one activation row per token) or r = t*topk + j (one row per routed pair).
//
// The grouping of the expert-indexed mat-vec kernel, carried onto the tensor-core pipeline of the dense
// path (candle PR 4056, "Metal: 64-token tile for the quantized matrix-matrix kernel", "Why the tile sets
// the weight reuse"): CTA (row block, rank u) reads the routing table, finds the u-th distinct expert in
// ascending id order and lists, in ascending slot order, the (token, slot) pairs routed to it. It then runs
// the K loop over that expert's 128 rows once per pass of up to TN listed pairs: the weights of each K step
// are decoded once for all the pass's pairs, as the dense kernel does for a token tile. The pairs'
// activation rows are gathered by one bulk copy each into a staging slot, and the decoder group of the K
// step rounds them to bf16 into the swizzled operand stage (columns past K, and pairs past the list, read
// as zero). Outputs are scattered to the pairs' rows of y. CTAs of ranks beyond the number of distinct
// experts leave at once; an id outside [0, E) gives NaN rows and a status bit, as on the mat-vec path.
// Every output element sees the same K steps and MMAs in the same order whatever the pass it falls in.
#include "../../include/qmm.h"
#include "mm_slab.cuh"

namespace wqk {
namespace mmid {

using mm::A_STAGE;
using mm::BK;
using mm::BM;
using mm::NDEC;
using mm::NGRP;
using mm::pf_of;
using mm::THREADS;

struct Experts {
    const uint8_t *p[QMM_MAX_EXPERTS];
};

struct Smem {
    uint64_t full_a[mm::MAX_STAGES], empty[mm::MAX_STAGES], xfull[mm::MAX_XSLOTS], xempty[mm::MAX_XSLOTS];
    uint64_t done, tfree;
    uint32_t tmem;
    int abort, nexp, expert, ns;
};

// Dynamic shared memory: operand stages and staging slots (as the dense kernel with binary32 activations),
// the Smem block, then the routing table / slot list and the expert flags.
__host__ __device__ constexpr int smem_bytes(int TN) {
    return mm::smem_bytes(TN, true) + (int)sizeof(Smem) + QMM_MAX_ID_SLOTS * 4 + QMM_MAX_EXPERTS;
}

template <int QT, int TN, bool XBF16>
__global__ void __launch_bounds__(THREADS, 1)
    mm_id_kernel(const __grid_constant__ Experts ex, int E, int N, int64_t K, int64_t rowbytes,
                 const void *__restrict__ x, int xdiv, const int32_t *__restrict__ ids, int M, int topk,
                 float *__restrict__ y, unsigned int *status) {
    constexpr int STAGES = mm::stages_of(TN, true), XSLOTS = mm::xslots_of(TN, true);
    constexpr int ESZ = XBF16 ? 2 : 4;
    constexpr int XROW = BK * ESZ;                        // staging bytes of one pair per K step
    constexpr uint32_t TMEM_COLS = TN <= 32 ? 32 : (TN <= 64 ? 64 : 128);
    static_assert(TN == 32 || TN == 64 || TN == 128, "token columns per pass");
    static_assert(smem_bytes(TN) <= 227 * 1024, "shared memory of one CTA");
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, TN);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    uint8_t *sX = sB + STAGES * mm::b_stage_bytes(TN);
    Smem *sm = reinterpret_cast<Smem *>(sX + XSLOTS * mm::x_slot_bytes(TN));
    int *s_slot = reinterpret_cast<int *>(sm + 1);                               // [QMM_MAX_ID_SLOTS]
    unsigned char *s_used = reinterpret_cast<unsigned char *>(s_slot + QMM_MAX_ID_SLOTS);   // [QMM_MAX_EXPERTS]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BM, u = blockIdx.y;
    const int nslot = M * topk;

    // The routing table usually comes from the preceding kernel (the router), and y may be read by it:
    // wait for it before anything else.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- routing: distinct experts in ascending id order; this CTA's expert and its slots
    for (int i = tid; i < QMM_MAX_EXPERTS; i += THREADS) s_used[i] = 0;
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < nslot; i += THREADS) {
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
        if (lane == 0) { sm->nexp = base; sm->expert = mine; }
    }
    __syncthreads();
    if (bad && u == 0) {
        // pairs routed to an id outside [0, E): NaN rows (this row block's part) and a status bit
        for (int p = 0; p < nslot; ++p) {
            const int e = s_slot[p];
            if (e < 0 || e >= E)
                for (int r = tid; r < BM; r += THREADS)
                    if (n0 + r < N) y[(int64_t)p * N + n0 + r] = __int_as_float(0x7fc00000);
        }
        if (tid == 0 && blockIdx.x == 0) atomicOr(status, kStatusBadId);
    }
    if (u >= sm->nexp) return;                            // no expert of this rank: the whole CTA leaves
    const int e = sm->expert;
    __syncthreads();                                      // every thread has read the table before compaction
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
        if (lane == 0) sm->ns = c;
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&sm->full_a[s], 8);            // the 8 warps of the group that fills this stage
            ptx::mbar_init(&sm->empty[s], 1);
        }
        for (int j = 0; j < XSLOTS; ++j) {
            ptx::mbar_init(&sm->xfull[j], 1);
            ptx::mbar_init(&sm->xempty[j], 8);
        }
        ptx::mbar_init(&sm->done, 1);
        ptx::mbar_init(&sm->tfree, NDEC);
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
    const int ns = sm->ns;
    const int npass = (ns + TN - 1) / TN;
    const int nsteps = (int)((K + BK - 1) / BK);
    const int G = npass * nsteps;                         // K steps over all passes
    const uint8_t *wq = ex.p[e];

    if (warp == 0) {
        // ---------------- gather: the pairs' activation rows of each K step into a staging slot
        for (int g = 0; g < G; ++g) {
            const int p = g / nsteps, i = g - p * nsteps, s = g % XSLOTS;
            int go = 1;
            if (lane == 0) {
                if (g >= XSLOTS) go = ptx::mbar_wait(&sm->xempty[s], ((g / XSLOTS) - 1) & 1, status);
                if (*(volatile int *)&sm->abort) go = 0;
                if (!go) sm->abort = 1;
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;     // the warp decides together
            const int cnt = ns - p * TN < TN ? ns - p * TN : TN;
            const int64_t k0 = (int64_t)i * BK;
            const uint32_t rowb = (uint32_t)((K - k0 < BK ? K - k0 : BK) * ESZ);   // a multiple of 16
            if (lane == 0) ptx::mbar_arrive_expect_tx(&sm->xfull[s], (uint32_t)cnt * rowb);
            __syncwarp();
            for (int c = lane; c < cnt; c += 32) {
                const int row = s_slot[p * TN + c] / xdiv;
                const uint8_t *src = static_cast<const uint8_t *>(x) + ((int64_t)row * K + k0) * ESZ;
                ptx::bulk_load(sX + s * mm::x_slot_bytes(TN) + c * XROW, src, rowb, &sm->xfull[s]);
            }
        }
        // every copy lands before the CTA may exit
        if (lane == 0)
            for (int g = (G > XSLOTS ? G - XSLOTS : 0); g < G; ++g)
                ptx::mbar_wait(&sm->xfull[g % XSLOTS], (g / XSLOTS) & 1, status);
    } else if (warp == 1) {
        // ---------------- MMA issuer: one pass after the other into the same accumulator
        if (lane == 0) {
            const uint32_t sA_u32 = ptx::smem_u32(sA), sB_u32 = ptx::smem_u32(sB);
            for (int p = 0; p < npass && !sm->abort; ++p) {
                if (p > 0 && !ptx::mbar_wait(&sm->tfree, (p - 1) & 1, status)) { sm->abort = 1; break; }
                bool stop = false;
                for (int i = 0; i < nsteps; ++i) {
                    const int g = p * nsteps + i, s = g % STAGES;
                    if (!ptx::mbar_wait(&sm->full_a[s], (g / STAGES) & 1, status)) {
                        sm->abort = 1;
                        stop = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t adesc = ptx::sw128_desc(sA_u32 + s * A_STAGE);
                    const uint64_t bdesc = ptx::sw128_desc(sB_u32 + s * mm::b_stage_bytes(TN));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        ptx::mma_bf16(tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (i | kk) != 0);
                    ptx::mma_commit(&sm->empty[s]);
                }
                ptx::mma_commit(&sm->done);               // the pass's MMAs (and all before them)
                if (stop) break;
            }
        }
    } else {
        // ---------------- decoders (as in the dense kernel) and, per pass, the epilogue
        const int d = warp - 2;
        const int grp = d >> 3, dw = d & 7;
        const int r_local = 16 * dw + (lane >> 1), h = lane & 1;
        const int row = n0 + r_local;
        const bool row_ok = row < N;
        const uint8_t *wrow = wq + (int64_t)(row_ok ? row : N - 1) * rowbytes;
        const int nchunks = (int)((K + 31) / 32);
        const uint32_t sA_u32 = ptx::smem_u32(sA), sB_u32 = ptx::smem_u32(sB);
        const int q = warp & 3, pw = mm::part_of(warp);
        const int r = 32 * q + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        using SL = mm::Slab<QT>;
        bool stop = false;
        for (int p = 0; p < npass && !stop; ++p) {
            const int cnt = ns - p * TN < TN ? ns - p * TN : TN;
            constexpr int PFT = pf_of<QT>();
            typename SL::Raw rw[PFT + 1];
            if constexpr (SL::FAST) {
                const int c0 = 2 * grp + h;
#pragma unroll
                for (int j = 0; j < PFT; ++j)
                    if (grp + j * NGRP < nsteps && c0 + 2 * j * NGRP < nchunks) SL::load(rw[j], wrow, c0 + 2 * j * NGRP);
            }
            for (int i = grp; i < nsteps; i += NGRP) {
                const int g = p * nsteps + i, s = g % STAGES, xs = g % XSLOTS;
                const int c = 2 * i + h;
                if constexpr (SL::FAST) {
                    if (i + PFT * NGRP < nsteps && c + 2 * PFT * NGRP < nchunks)
                        SL::load(rw[PFT], wrow, c + 2 * PFT * NGRP);
                }
                if (g >= STAGES && !ptx::mbar_wait(&sm->empty[s], ((g / STAGES) - 1) & 1, status)) {
                    sm->abort = 1;
                    stop = true;
                    break;
                }
                uint32_t o[16];
                if (row_ok && c < nchunks) {
                    if constexpr (SL::FAST) {
                        SL::decode(rw[0], c, o);
                    } else {
                        float w[32];
                        decode_chunk<QT>(wrow, c, K, w);
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = mm::pack_bf16x2(w[2 * j], w[2 * j + 1]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = 0u;
                }
                const uint32_t a_base = sA_u32 + s * A_STAGE;
#pragma unroll
                for (int pp = 0; pp < 4; ++pp)
                    ptx::st_shared_v4(a_base + mm::sw128_off(r_local, 4 * h + pp), o[4 * pp], o[4 * pp + 1],
                                      o[4 * pp + 2], o[4 * pp + 3]);
                // this step's gathered activations -> bf16 operand stage (pairs past the list and columns
                // past K as zero)
                if (!ptx::mbar_wait(&sm->xfull[xs], (g / XSLOTS) & 1, status)) {
                    sm->abort = 1;
                    stop = true;
                    break;
                }
                const uint8_t *xsrc = sX + xs * mm::x_slot_bytes(TN);
                const uint32_t b_base = sB_u32 + s * mm::b_stage_bytes(TN);
                const int gt = 32 * dw + lane;
                const int64_t k0 = (int64_t)i * BK;
#pragma unroll
                for (int pc = gt; pc < TN * 8; pc += 256) {
                    const int rr = pc >> 3, q8 = pc & 7;
                    uint32_t v0 = 0u, v1 = 0u, v2 = 0u, v3 = 0u;
                    if (rr < cnt && k0 + 8 * q8 < K) {
                        if constexpr (XBF16) {
                            const uint4 a = *reinterpret_cast<const uint4 *>(xsrc + rr * XROW + 16 * q8);
                            v0 = a.x; v1 = a.y; v2 = a.z; v3 = a.w;
                        } else {
                            const float4 a = *reinterpret_cast<const float4 *>(xsrc + rr * XROW + 32 * q8);
                            const float4 b = *reinterpret_cast<const float4 *>(xsrc + rr * XROW + 32 * q8 + 16);
                            v0 = mm::pack_bf16x2(a.x, a.y); v1 = mm::pack_bf16x2(a.z, a.w);
                            v2 = mm::pack_bf16x2(b.x, b.y); v3 = mm::pack_bf16x2(b.z, b.w);
                        }
                    }
                    ptx::st_shared_v4(b_base + mm::sw128_off(rr, q8), v0, v1, v2, v3);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm->xempty[xs]);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm->full_a[s]);
                if constexpr (SL::FAST) {
#pragma unroll
                    for (int j = 0; j < PFT; ++j) rw[j] = rw[j + 1];
                }
            }
            stop = !__all_sync(0xffffffffu, !stop);
            // ---- epilogue of the pass: TMEM lanes = weight rows, columns = the pass's pairs
            const bool ok = !stop && __all_sync(0xffffffffu, ptx::mbar_wait(&sm->done, p & 1, status) &&
                                                                  !*(volatile int *)&sm->abort);
            ptx::tc_fence_after();
            if (ok) {
                for (int c0 = 16 * pw; c0 < TN; c0 += 16 * (NDEC / 4)) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(lane_base + c0, v);
                    ptx::tmem_ld_wait();
                    if (n0 + r < N) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < cnt) y[(int64_t)s_slot[p * TN + c0 + j] * N + n0 + r] = __uint_as_float(v[j]);
                    }
                }
            } else {
                stop = true;
            }
            // the accumulator is free for the next pass
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm->tfree);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA this CTA issued has completed before the accumulator is freed (the issuer committed
        // `done` after the last pass it started)
        if (G > 0) {
            if (lane == 0) {
                const int last = npass - 1;
                ptx::mbar_wait(&sm->done, last & 1, status);
            }
            __syncwarp();
            ptx::tc_fence_after();
        }
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace mmid

// ------------------------------------------------------------------------------------------ host side
namespace {

struct MmIdLaunch {
    bool xbf16;
    const mmid::Experts *ex;
    int E;
    int64_t N, K;
    const void *x;
    int xdiv;
    const int32_t *ids;
    int M, topk;
    float *y;
    int tn;
    unsigned int *status;
    cudaStream_t st;
    template <int QT, int TN, bool XB> int go() {
        auto kern = mmid::mm_id_kernel<QT, TN, XB>;
        constexpr int smem = mmid::smem_bytes(TN);
        static bool attr_set[kMaxDevices] = {};
        const int devi = current_device_index();
        if (!attr_set[devi]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -6;
            attr_set[devi] = true;
        }
        const int64_t nslot = (int64_t)M * topk;
        const int64_t dmax = nslot < E ? nslot : E;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((N + mm::BM - 1) / mm::BM), (unsigned)dmax, 1);
        cfg.blockDim = dim3(mm::THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, *ex, E, (int)N, K, row_bytes(QT, K), x, xdiv, ids, M, topk,
                                                 y, status);
        return e == cudaSuccess ? 0 : -6;
    }
    template <int QT, int TN> int go_x() { return xbf16 ? go<QT, TN, true>() : go<QT, TN, false>(); }
    template <int QT> int operator()() {
        switch (tn) {
        case 32: return go_x<QT, 32>();
        case 64: return go_x<QT, 64>();
        case 128: return go_x<QT, 128>();
        default: return -7;
        }
    }
};

}  // namespace

// Token columns per pass of the tensor-core expert path: enough for the pairs an expert gets on average
// when the routing spreads M*topk pairs over min(E, M*topk) experts (an expert with more takes several
// passes, each decoding its weights again), at least 32.
int mm_id_columns(int64_t E, int64_t M, int topk) {
    const int64_t nslot = M * topk, used = nslot < E ? nslot : E;
    const int64_t avg = (nslot + used - 1) / used;
    return avg <= 32 ? 32 : (avg <= 64 ? 64 : 128);
}

// Expert-indexed product on the tensor cores. x rows: the token's (x_per_slot false) or the pair's.
int launch_mm_id(int qt, bool xbf16, const void *const *wq, int64_t E, int64_t N, int64_t K, const void *x,
                 bool x_per_slot, const int32_t *ids, int64_t M, int topk, float *y, unsigned int *status,
                 cudaStream_t st) {
    mmid::Experts ex;
    for (int e = 0; e < QMM_MAX_EXPERTS; ++e) ex.p[e] = e < E ? static_cast<const uint8_t *>(wq[e]) : nullptr;
    MmIdLaunch f{xbf16, &ex, (int)E, N, K, x, x_per_slot ? 1 : topk, ids, (int)M, topk, y, mm_id_columns(E, M, topk),
                 status, st};
    return dispatch_type(qt, f);
}

}  // namespace wqk

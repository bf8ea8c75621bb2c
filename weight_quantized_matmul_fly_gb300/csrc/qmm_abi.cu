// The C-ABI of libqmm: argument checks, path and tile choice, launches. No device memory is touched on
// the host; every call is asynchronous on the caller's stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/qmm.h"
#include "qmm_common.cuh"

namespace wqk {
// The device status word (QMM_STATUS_* bits). Host code reaches it through status_ptr().
__device__ unsigned int g_status = 0;

int launch_gemv(int qt, bool xbf16, const void *wq, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                cudaStream_t st);
int launch_gemv_tc(int qt, bool xbf16, const void *wq, int64_t N, int64_t K, const void *x, int M, float *y,
                   unsigned int *status, cudaStream_t st, bool dry = false, int stall = 0, bool early = false);
int launch_gemv_tc_multi(int qt, bool xbf16, const MatSet &ms, int64_t K, const void *x, int M,
                         unsigned int *status, cudaStream_t st, bool dry, bool early);
int launch_gemv_tc_id(int qt, bool xbf16, const void *const *wq, int64_t E, int64_t N, int64_t K, const void *x,
                      bool x_per_slot, const int32_t *ids, int64_t M, int topk, float *y, unsigned int *status,
                      cudaStream_t st);
int launch_mm(int qt, int tile, const void *wq, int64_t N, int64_t K, const void *x, bool x_f32, int64_t M,
              float *y, float *part, bool early, unsigned int *status, cudaStream_t st);
size_t mm_partial_bytes(int qt, int64_t N, int64_t K, int64_t M);
int mm_ksplit(int qt, int64_t N, int64_t K, int64_t M, bool cluster);
int mm_plan_cols(int qt, int64_t N, int64_t K, int64_t M, bool cluster);
int launch_x_to_bf16(const float *x, void *out, int64_t n, cudaStream_t st);
int launch_mm_id(int qt, bool xbf16, const void *const *wq, int64_t E, int64_t N, int64_t K, const void *x,
                 bool x_per_slot, const int32_t *ids, int64_t M, int topk, float *y, unsigned int *status,
                 cudaStream_t st);
int launch_mvid(int qt, bool xbf16, const void *const *wq, int64_t E, int64_t N, int64_t K, const void *x,
                bool x_per_slot, const int32_t *ids, int64_t M, int topk, float *y, unsigned int *status,
                cudaStream_t st);
int launch_dequant(int qt, const void *wq, int64_t N, int64_t K, float *out, cudaStream_t st);
int launch_quantize(int qt, const float *w, int64_t N, int64_t K, void *out, cudaStream_t st);
}  // namespace wqk

using namespace wqk;

namespace {

constexpr int64_t kMaxDim = (int64_t)1 << 31;   // rows, columns and tokens each below 2^31
constexpr int kGemvMaxM = 16;                   // mat-vec path up to here, tensor-core path above

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Common checks of qmm-family arguments. Returns 0 or a QMM_E* code.
int check_qmm(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, const float *y) {
    if ((qtype & ~(0xff | QMM_X_BF16 | QMM_W_STATIC)) != 0) return QMM_EQTYPE;
    const int qt = qtype & 0xff;
    if (qt < 0 || qt >= T_COUNT) return QMM_EQTYPE;
    if (N <= 0 || K <= 0 || M <= 0 || N >= kMaxDim || K >= kMaxDim || M >= kMaxDim) return QMM_EDIM;
    if (K % kQK[qt] != 0) return QMM_EBLOCK;
    if (!wq || !x || !y) return QMM_ENULL;
    if (!aligned16(wq) || !aligned16(x) || !aligned16(y)) return QMM_EALIGN;
    return 0;
}

// The tensor-core path reads bf16 activation rows by TMA: their stride (K * 2 bytes) must be a multiple of
// 16 bytes, and the decoders walk 32-weight chunks.
inline bool mm_eligible(int qt, int64_t K) { return (K % 8) == 0 && (kQK[qt] >= 32 || K % 32 == 0); }

// Device address of the status word on the current device (looked up once per device; host threads that
// race on the first lookup all store the same address).
unsigned int *status_ptr() {
    static std::atomic<void *> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    void *p = cache[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        cache[dev].store(p, std::memory_order_relaxed);
    }
    return static_cast<unsigned int *>(p);
}

// The mat-vec path: quantized types on the tensor-core mat-vec kernel (16 tokens per launch at most,
// halved when the activations of a K segment would not fit on chip); the plain types on the binary32 one.
// With `launches` non-null nothing is launched: the launches the call would make are counted instead.
int run_matvec(int qt, bool xbf16, const void *wq, int64_t N, int64_t K, const void *x, int64_t M, float *y,
               cudaStream_t st, int *launches = nullptr, int stall = 0, bool early = false) {
    if (is_plain(qt)) {
        if (launches) { *launches = (int)((M + 15) / 16); return 0; }
        return launch_gemv(qt, xbf16, wq, N, K, x, M, y, st);
    }
    const int esz = xbf16 ? 2 : 4;
    unsigned int *status = launches ? nullptr : status_ptr();
    if (!launches && !status) return QMM_ECUDA;
    int count = 0;
    for (int64_t m0 = 0; m0 < M;) {
        int mg = (int)((M - m0) < 16 ? (M - m0) : 16);
        int rc;
        for (;;) {
            rc = launch_gemv_tc(qt, xbf16, wq, N, K, static_cast<const uint8_t *>(x) + m0 * K * esz, mg,
                                y + m0 * N, status, st, launches != nullptr, m0 == 0 ? stall : 0, early);
            if (rc != -3 || mg <= 4) break;
            mg = (mg + 1) / 2;
        }
        if (rc) return rc == -3 ? QMM_EDIM : rc;
        ++count;
        m0 += mg;
    }
    if (launches) *launches = count;
    return 0;
}

// The mat-vec path for several matrices of one type and K that share x: one launch per token group, its
// CTAs covering the row blocks of every matrix (the groups halved as run_matvec halves them).
int run_matvec_multi(int qt, bool xbf16, const MatSet &ms, int64_t K, const void *x, int64_t M, cudaStream_t st,
                     bool early) {
    const int esz = xbf16 ? 2 : 4;
    unsigned int *status = status_ptr();
    if (!status) return QMM_ECUDA;
    for (int64_t m0 = 0; m0 < M;) {
        int mg = (int)((M - m0) < 16 ? (M - m0) : 16);
        MatSet g = ms;
        for (int i = 0; i < ms.count; ++i) g.y[i] = ms.y[i] + m0 * ms.N[i];
        int rc;
        for (;;) {
            rc = launch_gemv_tc_multi(qt, xbf16, g, K, static_cast<const uint8_t *>(x) + m0 * K * esz, mg, status, st,
                                      false, early);
            if (rc != -3 || mg <= 4) break;
            mg = (mg + 1) / 2;
        }
        if (rc) return rc == -3 ? QMM_EDIM : rc;
        m0 += mg;
    }
    return 0;
}

inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Binary32 activations on the tensor-core path. With scratch from the caller (qmm_ws) and more than 32
// tokens, a separate pass writes a bf16 copy of x that the kernel loads by TMA at the plan's full width, and
// a K split writes its partial tiles to the scratch for a second kernel to add. Otherwise (qmm and
// qmm_with_tile, which take no scratch, and up to 32 tokens) the kernel converts x itself, with at most 128
// columns per CTA, and adds a K split inside a thread block cluster. Measured on the Qwen3-Embedding-4B
// projections: the conversion pass, chained to the kernel by programmatic dependent launch, costs 0.3-0.5 us
// a call, converting inside the kernel 3-11 us at 64-128 columns but nothing at 32; behind the pass, a
// cluster launch starts later than the second kernel costs; with bf16 activations the cluster is faster.
// The two ways plan their K split separately (up to 32 CTAs, or up to 8 in a cluster), so qmm_ws and qmm
// may differ in the last bits; each is the same for every token tile.
bool f32_copy(int qtype, int64_t M, int path) { return path != 0 && !(qtype & QMM_X_BF16) && M > 32; }
size_t ws_x_bytes(int qtype, int64_t K, int64_t M, int path) {
    return f32_copy(qtype, M, path) ? align256((size_t)M * (size_t)K * 2) : 0;
}
size_t ws_bytes(int qtype, int64_t N, int64_t K, int64_t M, int path) {
    if (!f32_copy(qtype, M, path)) return 0;
    return ws_x_bytes(qtype, K, M, path) + align256(mm_partial_bytes(qtype & 0xff, N, K, M));
}

int run_mm(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y, int tile,
           void *ws, size_t wsb, cudaStream_t st) {
    const int qt = qtype & 0xff;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return QMM_EALIGN;
    unsigned int *status = status_ptr();
    if (!status) return QMM_ECUDA;
    const bool xf32 = !(qtype & QMM_X_BF16), early = (qtype & QMM_W_STATIC) != 0;
    const size_t need = ws_bytes(qtype, N, K, M, tile);
    if (need && ws && wsb >= need) {
        int rc = launch_x_to_bf16(static_cast<const float *>(x), ws, M * K, st);
        if (rc) return rc;
        float *part = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + ws_x_bytes(qtype, K, M, tile));
        return launch_mm(qt, tile, wq, N, K, ws, false, M, y, part, early, status, st);
    }
    return launch_mm(qt, tile, wq, N, K, x, xf32, M, y, nullptr, early, status, st);
}

// Expert-indexed path for the routing a call carries on average: the tensor-core kernel once an expert
// gets enough routed pairs that decoding its weights once per pass of up to 32-128 pairs beats the mat-vec
// machinery's passes of 4 (8 with bf16 activations) pairs. Measured on GB300 (experts of 4096 x K Q4_0,
// K = 512-1024, top-8): the mat-vec kernel is faster up to 16 pairs per expert (128 experts, 256 tokens) and
// at 32; the two break even at 128 pairs per expert, and the tensor-core kernel is ahead (5 %) at 256.
constexpr int64_t kIdTensorMinPairs = 128;
int pick_id_path(int qt, int64_t E, int64_t K, int64_t M, int topk) {
    const int64_t nslot = M * topk, used = nslot < E ? nslot : E;
    return (mm_eligible(qt, K) && nslot >= kIdTensorMinPairs * used) ? 2 : 1;
}

int run_qmm_id(const void *const *wq, int64_t E, int qtype, int64_t N, int64_t K, const void *x, const int32_t *ids,
               int64_t M, int topk, float *y, void *stream, int path) {
    if ((qtype & ~(0xff | QMM_X_BF16 | QMM_X_PER_SLOT | QMM_W_STATIC)) != 0) return QMM_EQTYPE;
    const int qt = qtype & 0xff;
    if (qt < 0 || qt >= T_COUNT) return QMM_EQTYPE;
    if (N <= 0 || K <= 0 || M <= 0 || N >= kMaxDim || K >= kMaxDim) return QMM_EDIM;
    if (K % kQK[qt] != 0 || K % 32 != 0) return QMM_EBLOCK;
    if (E < 1 || E > QMM_MAX_EXPERTS || topk < 1 || M * (int64_t)topk > QMM_MAX_ID_SLOTS) return QMM_ERANGE;
    if (path < 0 || path > 2) return QMM_ERANGE;
    if (!wq || !x || !ids || !y) return QMM_ENULL;
    for (int64_t e = 0; e < E; ++e) {
        if (!wq[e]) return QMM_ENULL;
        if (!aligned16(wq[e])) return QMM_EALIGN;
    }
    if (!aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return QMM_EALIGN;
    unsigned int *status = status_ptr();
    if (!status) return QMM_ECUDA;
    const bool xbf16 = (qtype & QMM_X_BF16) != 0, per_slot = (qtype & QMM_X_PER_SLOT) != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (path == 0) path = pick_id_path(qt, E, K, M, topk);
    if (path == 2) {
        if (!mm_eligible(qt, K)) return QMM_EBLOCK;
        return launch_mm_id(qt, xbf16, wq, E, N, K, x, per_slot, ids, M, topk, y, status, st);
    }
    const int rc = launch_gemv_tc_id(qt, xbf16, wq, E, N, K, x, per_slot, ids, M, topk, y, status, st);
    if (rc != -3) return rc;
    return launch_mvid(qt, xbf16, wq, E, N, K, x, per_slot, ids, M, topk, y, status, st);
}

}  // namespace

namespace wqk {
// The argument checks of qmm / qmm_ws, for the other entry points of the qmm family.
int check_qmm_args(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, const float *y) {
    return check_qmm(wq, qtype, N, K, x, M, y);
}
}  // namespace wqk

extern "C" {

int qmm_pick_tile(int64_t M) {
    if (M <= 0) return 0;
    const int64_t pad32 = (M + 31) / 32 * 32 - M;
    int best = 32;
    for (int T : {64, 128})
        if ((M + T - 1) / T * T - M == pad32) best = T;
    return best;
}

int qmm_pick_path(int qtype, int64_t N, int64_t K, int64_t M) {
    (void)N;
    const int qt = qtype & 0xff;
    if (qt < 0 || qt >= T_COUNT) return QMM_EQTYPE;
    if (M <= kGemvMaxM || !mm_eligible(qt, K)) return 0;
    return qmm_pick_tile(M);
}

size_t qmm_workspace_size(int qtype, int64_t N, int64_t K, int64_t M) {
    const int path = qmm_pick_path(qtype, N, K, M);
    if (path <= 0) return 0;
    return ws_bytes(qtype, N, K, M, path);
}

int qmm_ws(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y, void *workspace,
           size_t workspace_bytes, void *stream) {
    int rc = check_qmm(wq, qtype, N, K, x, M, y);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int path = qmm_pick_path(qtype, N, K, M);
    if (path == 0)
        return run_matvec(qtype & 0xff, (qtype & QMM_X_BF16) != 0, wq, N, K, x, M, y, st, nullptr, 0,
                          (qtype & QMM_W_STATIC) != 0);
    const size_t need = ws_bytes(qtype, N, K, M, path);
    if (need && (!workspace || workspace_bytes < need)) return QMM_EWORKSPACE;
    return run_mm(wq, qtype, N, K, x, M, y, path, workspace, workspace_bytes, st);
}

int qmm(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y, void *stream) {
    int rc = check_qmm(wq, qtype, N, K, x, M, y);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int path = qmm_pick_path(qtype, N, K, M);
    if (path == 0)
        return run_matvec(qtype & 0xff, (qtype & QMM_X_BF16) != 0, wq, N, K, x, M, y, st, nullptr, 0,
                          (qtype & QMM_W_STATIC) != 0);
    return run_mm(wq, qtype, N, K, x, M, y, path, nullptr, 0, st);
}

int qmm_batch(int count, const void *const *wq, const int64_t *N, float *const *y, int qtype, int64_t K,
              const void *x, int64_t M, void *stream) {
    if (count < 1 || count > kMaxBatch) return QMM_ERANGE;
    if (!wq || !N || !y) return QMM_ENULL;
    for (int i = 0; i < count; ++i) {
        const int rc = check_qmm(wq[i], qtype, N[i], K, x, M, y[i]);
        if (rc) return rc;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int qt = qtype & 0xff;
    if (M <= kGemvMaxM && !is_plain(qt) && count > 1) {
        MatSet ms = {};
        ms.count = count;
        for (int i = 0; i < count; ++i) {
            ms.wq[i] = wq[i];
            ms.N[i] = N[i];
            ms.y[i] = y[i];
        }
        return run_matvec_multi(qt, (qtype & QMM_X_BF16) != 0, ms, K, x, M, st, (qtype & QMM_W_STATIC) != 0);
    }
    for (int i = 0; i < count; ++i) {
        const int rc = qmm(wq[i], qtype, N[i], K, x, M, y[i], stream);
        if (rc) return rc;
    }
    return 0;
}

int qmm_with_tile(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y, int tile,
                  void *stream) {
    int rc = check_qmm(wq, qtype, N, K, x, M, y);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (tile == 0)
        return run_matvec(qtype & 0xff, (qtype & QMM_X_BF16) != 0, wq, N, K, x, M, y, st, nullptr, 0,
                          (qtype & QMM_W_STATIC) != 0);
    if (tile != 32 && tile != 64 && tile != 128) return QMM_ERANGE;
    if (!mm_eligible(qtype & 0xff, K)) return QMM_EBLOCK;
    return run_mm(wq, qtype, N, K, x, M, y, tile, nullptr, 0, st);
}

int qmm_id(const void *const *wq, int64_t E, int qtype, int64_t N, int64_t K, const void *x, const int32_t *ids,
           int64_t M, int topk, float *y, void *stream) {
    return run_qmm_id(wq, E, qtype, N, K, x, ids, M, topk, y, stream, 0);
}

int qmm_id_with_path(const void *const *wq, int64_t E, int qtype, int64_t N, int64_t K, const void *x,
                     const int32_t *ids, int64_t M, int topk, float *y, int path, void *stream) {
    return run_qmm_id(wq, E, qtype, N, K, x, ids, M, topk, y, stream, path);
}

int qmm_id_pick_path(int qtype, int64_t E, int64_t K, int64_t M, int topk) {
    const int qt = qtype & 0xff;
    if (qt < 0 || qt >= T_COUNT) return QMM_EQTYPE;
    if (E < 1 || M < 1 || topk < 1) return QMM_ERANGE;
    return pick_id_path(qt, E, K, M, topk);
}

int qmm_dequant(const void *wq, int qtype, int64_t N, int64_t K, float *w_out, void *stream) {
    if (qtype < 0 || qtype >= T_COUNT) return QMM_EQTYPE;
    if (N <= 0 || K <= 0 || N >= kMaxDim || K >= kMaxDim) return QMM_EDIM;
    if (K % kQK[qtype] != 0) return QMM_EBLOCK;
    if (!wq || !w_out) return QMM_ENULL;
    if (!aligned16(wq) || !aligned16(w_out)) return QMM_EALIGN;
    return launch_dequant(qtype, wq, N, K, w_out, static_cast<cudaStream_t>(stream));
}

int qmm_quantize(const float *w_in, int qtype, int64_t N, int64_t K, void *wq_out, void *stream) {
    if (qtype < 0 || qtype >= T_COUNT) return QMM_EQTYPE;
    if (N <= 0 || K <= 0 || N >= kMaxDim || K >= kMaxDim) return QMM_EDIM;
    if (K % kQK[qtype] != 0) return QMM_EBLOCK;
    if (!w_in || !wq_out) return QMM_ENULL;
    if (!aligned16(w_in) || !aligned16(wq_out)) return QMM_EALIGN;
    return launch_quantize(qtype, w_in, N, K, wq_out, static_cast<cudaStream_t>(stream));
}

int qmm_type_info(int qtype, int *block_weights, int *block_bytes) {
    if (qtype < 0 || qtype >= T_COUNT) return QMM_EQTYPE;
    if (!block_weights || !block_bytes) return QMM_ENULL;
    *block_weights = kQK[qtype];
    *block_bytes = kBytes[qtype];
    return 0;
}

int qmm_get_status(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int zero = 0, v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return QMM_ECUDA;
    if (cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return QMM_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return QMM_ECUDA;
    return (int)(v & 0x7fffffffu);
}

int qmm_debug_stall(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                    void *stream) {
    int rc = check_qmm(wq, qtype, N, K, x, M, y);
    if (rc) return rc;
    const int qt = qtype & 0xff;
    if (is_plain(qt) || M > kGemvMaxM) return QMM_ERANGE;
    return run_matvec(qt, (qtype & QMM_X_BF16) != 0, wq, N, K, x, M, y, static_cast<cudaStream_t>(stream),
                      nullptr, 1);
}

int qmm_plan_info(int qtype, int64_t N, int64_t K, int64_t M, int *ksplit, int *cols) {
    if (!ksplit || !cols) return QMM_ENULL;
    const int path = qmm_pick_path(qtype, N, K, M);
    if (path < 0) return path;
    if (path == 0) { *ksplit = 0; *cols = 0; return 0; }
    if (N <= 0 || K <= 0 || M <= 0 || N >= kMaxDim || K >= kMaxDim || M >= kMaxDim) return QMM_EDIM;
    const bool cluster = !f32_copy(qtype, M, path);
    *ksplit = mm_ksplit(qtype & 0xff, N, K, M, cluster);
    *cols = mm_plan_cols(qtype & 0xff, N, K, M, cluster);
    return path;
}

int qmm_launch_count(int qtype, int64_t N, int64_t K, int64_t M) {
    const int path = qmm_pick_path(qtype, N, K, M);
    if (path < 0) return path;
    if (path == 0) {
        // the mat-vec path's own plan (token groups of 16, halved where the activations would not fit)
        // (one launch per 16 tokens when there is no device to plan on)
        int n = 0;
        const int rc = run_matvec(qtype & 0xff, (qtype & QMM_X_BF16) != 0, nullptr, N, K, nullptr, M, nullptr,
                                  nullptr, &n);
        return rc ? (int)((M + 15) / 16) : n;
    }
    if (!f32_copy(qtype, M, path)) return 1;
    const int S = mm_ksplit(qtype & 0xff, N, K, M, false);
    return 2 + (S > 1 ? 1 + ((M * N) % 4 ? 1 : 0) : 0);
}

const char *qmm_strerror(int code) {
    switch (code) {
    case QMM_OK: return "ok";
    case QMM_EQTYPE: return "unknown weight type or flag";
    case QMM_EBLOCK: return "K is not a multiple of the block size";
    case QMM_EDIM: return "dimension out of range";
    case QMM_ENULL: return "null pointer";
    case QMM_EALIGN: return "pointer not 16-byte aligned";
    case QMM_ECUDA: return "CUDA launch or runtime error";
    case QMM_ERANGE: return "E, topk or tile out of range";
    case QMM_EWORKSPACE: return "workspace missing or too small";
    default: return "unknown error";
    }
}

}  // extern "C"

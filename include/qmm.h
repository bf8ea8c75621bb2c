/*
 * libqmm: block-quantized weight matmul for one GB300 GPU (sm_103a).
 *
 *     y[m, n] = sum_k dequant(W)[n, k] * x[m, k]
 *
 * The weights stay quantized in device memory and are dequantized on the fly inside the kernels: each
 * weight block is read, dequantized and multiplied by the activation rows of a token tile (candle PR 4056,
 * "Metal: 64-token tile for the quantized matrix-matrix kernel", section "Why the tile sets the weight
 * reuse"). The expert-indexed form computes one mat-vec per routed (token, expert) pair (llama.cpp PR
 * 28086, "metal : fix idle threads in mul_mv_iq3_xxs for ne00 < 1024", MUL_MAT_ID).
 *
 * Weight types and block layouts: QMM_F32 ... QMM_A4G64 below. The layouts are this library's own block
 * format specification (the pages name the types but do not define them); each block stores a scale (and
 * for some types a minimum or bias) plus packed integer codes, and row n of an N x K matrix is K/QK blocks
 * stored back to back, rows following each other without padding.
 *
 * Conventions shared by every entry point:
 *   - Pointers named wq, x, y, ids, w_out, w_in are DEVICE pointers owned by the caller. The library
 *     keeps no reference to them after the call returns and frees nothing it did not allocate.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call is asynchronous on it:
 *     a return value of 0 means the work was launched, not that it finished.
 *   - Return values: 0 on success, a negative QMM_E* code otherwise (qmm_strerror() names it). On any
 *     error nothing is launched. Arguments are checked on the host without dereferencing device memory.
 *   - wq, x and y must be 16-byte aligned.
 *   - Nothing here is thread-safe against concurrent calls that share an output buffer.
 *   - The matmul kernels are launched with programmatic dependent launch: each may start while the
 *     previous kernel in the stream finishes. Before that kernel has completed they only prefetch their
 *     weights into L2 (which is coherent); wq, x, ids and y are read or written only after it has. So
 *     any kernel, including one that writes wq or x, may immediately precede a call. With QMM_W_STATIC
 *     in qtype the caller states that the kernel launched immediately before the call on the same stream
 *     does not write wq (true of model weights): the kernels then read the weights at once, overlapping
 *     the end of that kernel (measured 2-8 % faster per call).
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight types (block size QK in weights / bytes per block). */
enum qmm_type {
    QMM_F32 = 0,   /*   1 /   4  plain binary32 */
    QMM_F16 = 1,   /*   1 /   2  plain binary16 */
    QMM_BF16 = 2,  /*   1 /   2  plain bfloat16 */
    QMM_Q4_0 = 3,  /*  32 /  18  w = d*(q-8) */
    QMM_Q4_1 = 4,  /*  32 /  20  w = d*q + m */
    QMM_Q5_0 = 5,  /*  32 /  22  w = d*(q-16) */
    QMM_Q5_1 = 6,  /*  32 /  24  w = d*q + m */
    QMM_Q8_0 = 7,  /*  32 /  34  w = d*q */
    QMM_Q2_K = 8,  /* 256 /  84  w = d*sc*q - dmin*mn, 16 sub-blocks of 16 */
    QMM_Q3_K = 9,  /* 256 / 110  w = d*(sc-32)*(q-4), 16 sub-blocks of 16 */
    QMM_Q4_K = 10, /* 256 / 144  w = d*sc*q - dmin*mn, 8 sub-blocks of 32 */
    QMM_Q5_K = 11, /* 256 / 176  w = d*sc*q - dmin*mn, 8 sub-blocks of 32 */
    QMM_Q6_K = 12, /* 256 / 210  w = d*sc*(q-32), 16 sub-blocks of 16 */
    QMM_A4G64 = 13,/*  64 /  36  w = s*q + b, bf16 s and b (MLX-style group-64 affine 4-bit) */
    QMM_NTYPES = 14
};

/* OR into `qtype` to pass bfloat16 activations instead of binary32. */
#define QMM_X_BF16 0x100
/* qmm_id only: OR into `qtype` when x holds one activation row per (token, slot), M x topk x K, instead
 * of one row per token shared by its topk slots (the experts' down projection, whose input differs per
 * routed expert: llama.cpp PR 28086, "Test methodology", ffn_down_exps). */
#define QMM_X_PER_SLOT 0x200
/* OR into `qtype` when the kernel launched immediately before the call on the same stream does not write
 * wq (see the conventions above); accepted by every matmul entry point. */
#define QMM_W_STATIC 0x400

/* Error codes. */
#define QMM_OK 0
#define QMM_EQTYPE (-1)   /* unknown weight type or flag */
#define QMM_EBLOCK (-2)   /* K is not a multiple of the type's block size */
#define QMM_EDIM (-3)     /* a dimension is <= 0 or too large */
#define QMM_ENULL (-4)    /* a required pointer is NULL */
#define QMM_EALIGN (-5)   /* wq, x or y is not 16-byte aligned */
#define QMM_ECUDA (-6)    /* a CUDA runtime call or launch failed */
#define QMM_ERANGE (-7)   /* E, topk or a tile argument out of range */
#define QMM_EWORKSPACE (-8) /* workspace missing or too small */

/* Limits. */
#define QMM_MAX_EXPERTS 256
#define QMM_MAX_ID_SLOTS 4096 /* M * topk for qmm_id */

/*
 * qmm: y = x * dequant(W)^T.
 *   wq    N x K weight matrix of type (qtype & 0xff), N * (K/QK) * bytes_per_block bytes.
 *   x     M x K row-major activations, binary32, or bfloat16 when qtype has QMM_X_BF16.
 *   y     M x N row-major binary32, overwritten.
 * M <= 16 runs the memory-bound mat-vec path (all lanes on weights, narrow-K row split); larger M runs
 * the tcgen05 tensor-core path with a 32/64/128-token tile picked by qmm_pick_tile(M). The tensor-core
 * path rounds x and the dequantized weights to bfloat16 (round to nearest even) and accumulates in
 * binary32 (for Q4_K, Q5_K and A4G64 the weight rounded is the binary32 weight up to 2^-17 times its
 * sub-block scale); the mat-vec path multiplies the binary32 dequantized weights by x in binary32.
 * qmm() allocates nothing. It launches one kernel on the tensor-core path, and on the mat-vec path one per
 * group of tokens (all of them, or two halves where a group's activations do not fit on chip next to its
 * weights, and for 9-16 binary32 tokens of large 2-5-bit matrices; see qmm_launch_count). On the
 * tensor-core path the work plan (a function of the type, N, K and M) may split the K dimension over
 * S <= 8 thread blocks; they form a cluster and add their partial sums in split order in shared memory.
 * Binary32 activations are rounded to bfloat16 inside the tensor-core kernel, with at most 128 token
 * columns per thread block. qmm_ws() is faster on that path with binary32 activations and M > 32: with
 * scratch (qmm_workspace_size()), a separate pass writes a bfloat16 copy of x that the kernel reads at the
 * plan's full width, and a K split (up to 32 thread blocks) sends its partial sums through the scratch to
 * a second kernel that adds them in split order. The two plan their K split separately, so their results
 * can differ in the last bits (both within the stated tolerance); each is bit-identical across token tiles.
 */
int qmm(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y, void *stream);

/* Bytes of scratch qmm_ws() needs for these arguments (0 when none): on the tensor-core path with binary32
 * x and M > 32, M*K*2 bytes (rounded up to 256) for its bfloat16 copy plus S*M*N*4 bytes for the partial sums
 * when the plan splits K over S thread blocks; nothing on the mat-vec path, up to 32 tokens, or with
 * bfloat16 activations (qmm_ws then runs as qmm). */
size_t qmm_workspace_size(int qtype, int64_t N, int64_t K, int64_t M);

/* qmm() with caller-provided scratch: `workspace` is a device buffer of at least
 * qmm_workspace_size(...) bytes, 256-byte aligned; may be NULL when that size is 0 (QMM_EWORKSPACE when
 * the size is not 0 and the buffer is missing or smaller). */
int qmm_ws(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y,
           void *workspace, size_t workspace_bytes, void *stream);

/*
 * qmm_noalloc: qmm() for callers that cannot allocate device memory. (The source pages have no
 * counterpart; this entry point exists for users of the library.)
 *
 * Who needs it: code whose execution step must not call cudaMalloc / cudaMallocAsync, for example a
 * plugin inside a framework that plans all device memory up front and forbids allocation while it runs,
 * code with hard latency limits (an allocation can synchronize the device or wait on the driver), or a
 * stream capture under a mode that rejects allocation calls. qmm() would allocate its tensor-core
 * scratch there; qmm_ws() needs a buffer the caller may have no way to obtain.
 *
 * What it does: the same computation and kernels as qmm_ws(), with the scratch taken from one device
 * array of QMM_NOALLOC_SCRATCH_BYTES that the library defines statically. The caller still passes wq, x
 * and y as for qmm(). Nothing is allocated, on the host or the device.
 *   - Limit: calls whose scratch (qmm_workspace_size) exceeds QMM_NOALLOC_SCRATCH_BYTES are refused with
 *     QMM_EWORKSPACE before anything is launched (for binary32 activations roughly M*K*2 bytes plus
 *     split-K partials; M*K up to about 30 million fits). Calls on the mat-vec path need no scratch.
 *   - Every GPU that loads the library keeps the array (QMM_NOALLOC_SCRATCH_BYTES) until the process
 *     exits.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that
 *     device current; make that first call before any stream capture that should contain these calls.
 *   - All calls share the one array and it keeps whatever the last call left there; no call relies on its
 *     contents (every byte a call reads, that call wrote first). Calls whose kernels can overlap on the
 *     GPU (different streams without ordering between them) race on the array: keep them ordered.
 */
#define QMM_NOALLOC_SCRATCH_BYTES (64u << 20)
int qmm_noalloc(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                void *stream);

/*
 * qmm_batch: y_i = x * dequant(W_i)^T for i < count, for up to QMM_MAX_BATCH weight matrices of one type and
 * one K that take the same activations x (the projections of one input: q/k/v, gate/up). A layer's
 * projections run back to back (candle PR 4056, "This branch, kernel level", times a layer as its seven
 * projections); on the mat-vec path (M <= 16, quantized types) the matrices that share x are served by one
 * kernel launch whose thread blocks cover the row blocks of all of them, so the fixed cost of a launch is
 * paid once. Otherwise the calls run one after the other as qmm() calls (allocation-free).
 *   wq, N, y  HOST arrays of `count` entries: device pointer, rows and output (M x N[i] binary32) of matrix i.
 * Arguments are checked as for qmm(), for every matrix, before anything is launched. Results are within the
 * same tolerance as qmm()'s; on the mat-vec path the work split of the shared launch may differ from that
 * of a single call, so the last bits may too.
 */
#define QMM_MAX_BATCH 8
int qmm_batch(int count, const void *const *wq, const int64_t *N, float *const *y, int qtype, int64_t K,
              const void *x, int64_t M, void *stream);

/*
 * qmm_id: expert-indexed mat-vec (MoE).  For each token t < M and slot j < topk, with e = ids[t*topk + j]:
 *     y[(t*topk + j)*N + n] = sum_k dequant(W_e)[n, k] * x[r*K + k]
 * where the activation row is r = t, or r = t*topk + j when qtype has QMM_X_PER_SLOT.
 *   wq    HOST array of E device pointers, one N x K weight matrix of type qtype per expert
 *         (each 16-byte aligned). The array itself is read during the call only.
 *   x     M x K (or M x topk x K with QMM_X_PER_SLOT) row-major, binary32 or bfloat16 (QMM_X_BF16).
 *   ids   DEVICE int32 array, M x topk.
 *   y     M x topk x N binary32, overwritten.
 * Every distinct expert's rows are streamed once per call for all tokens routed to it. An id outside
 * [0, E) cannot be checked on the host: that slot's output row is set to NaN and the device status word
 * (qmm_get_status) records QMM_STATUS_BAD_ID. Limits: 1 <= E <= QMM_MAX_EXPERTS,
 * 1 <= topk, M * topk <= QMM_MAX_ID_SLOTS.
 */
int qmm_id(const void *const *wq, int64_t E, int qtype, int64_t N, int64_t K, const void *x,
           const int32_t *ids, int64_t M, int topk, float *y, void *stream);

/* Which kernel qmm_id runs (qmm_id_pick_path): 1 = the expert-indexed mat-vec (binary32 products of the
 * exactly rounded weights, tolerance class 1e-5), used while an expert gets few routed pairs on average
 * (M*topk < 128 * min(E, M*topk)); 2 = the tensor-core expert kernel (x and weights rounded to bfloat16,
 * tolerance class 4e-3, like qmm's tensor-core path): each CTA takes one row block of one distinct expert
 * and runs tcgen05 MMAs over passes of up to 32/64/128 of its routed pairs, the activation rows gathered
 * by bulk copies, so each pass decodes the expert's weights once for all of them. Path 2 needs K a
 * multiple of 8 (plain types: 32). */
int qmm_id_pick_path(int qtype, int64_t E, int64_t K, int64_t M, int topk);

/* qmm_id with the path forced (tests and diagnostics): path 0 = as qmm_id picks, 1 or 2 as above.
 * QMM_ERANGE for another value. */
int qmm_id_with_path(const void *const *wq, int64_t E, int qtype, int64_t N, int64_t K, const void *x,
                     const int32_t *ids, int64_t M, int topk, float *y, int path, void *stream);

/*
 * qmm_with_tile: qmm() with the path forced, for tests and diagnostics (mirrors the pages' explicit-tile
 * entry point, candle PR 4056, section "What changes").
 *   tile = 0       mat-vec path (any M; tokens are processed 16 at a time)
 *   tile = 32/64/128  tensor-core path with that token tile
 * Output is bit-identical across tile = 32, 64, 128 for the same inputs (same K order and the same
 * split of K), which tests check.
 */
int qmm_with_tile(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                  int tile, void *stream);

/* The token-tile rule of the tensor-core path: the largest T in {32, 64, 128} whose padding
 * ceil(M/T)*T - M equals the 32-token tile's, i.e. that pads no more tokens than the 32-token tile
 * (candle PR 4056, section "Where the 64-token tile is used", extended to 128). Returns 0 for M <= 0. */
int qmm_pick_tile(int64_t M);

/* Which path qmm() takes for M tokens: 0 = mat-vec, 32/64/128 = tensor-core tile. */
int qmm_pick_path(int qtype, int64_t N, int64_t K, int64_t M);

/* The tensor-core work plan a qmm_ws() call with its workspace uses (diagnostic): the K split and the token
 * columns per thread block (before the cap at 128 that binary32 activations converted in the kernel get).
 * Returns the path as qmm_pick_path() does; on the mat-vec path (0) both outputs are 0. Without a device
 * the plan assumes unconstrained cluster packing. */
int qmm_plan_info(int qtype, int64_t N, int64_t K, int64_t M, int *ksplit, int *cols);

/* How many kernels one qmm_ws() call with these arguments and its workspace launches (diagnostic; qmm()
 * launches one kernel on the tensor-core path). The mat-vec path is planned as the call would plan it
 * (token groups of 16, halved where their activations do not fit on chip), which needs the current
 * device; without one it assumes one launch per 16 tokens. */
int qmm_launch_count(int qtype, int64_t N, int64_t K, int64_t M);

/*
 * qmm_dequant: w_out[n*K + k] = dequant(W)[n, k] as binary32. Each value is the exact value of the
 * type's formula rounded once to binary32 (bit-exact against the oracle). w_out is N x K, 16-byte aligned.
 */
int qmm_dequant(const void *wq, int qtype, int64_t N, int64_t K, float *w_out, void *stream);

/*
 * qmm_quantize: encode an N x K binary32 matrix (device, row-major) into blocks of type qtype
 * (deterministic round to nearest; decisions in binary32 so the result is reproducible bit for bit).
 * wq_out must hold N * (K/QK) * bytes_per_block bytes. Not on the matmul path.
 */
int qmm_quantize(const float *w_in, int qtype, int64_t N, int64_t K, void *wq_out, void *stream);

/* Block size in weights and bytes per block of a type (host only). */
int qmm_type_info(int qtype, int *block_weights, int *block_bytes);

/*
 * qmm_get_status: the device status word, a bit set of QMM_STATUS_* accumulated by the kernels since the
 * last call, read and cleared on `stream` (the call synchronises the stream). Returns the bits (>= 0), or
 * QMM_ECUDA when the read failed. The word is per device and shared by every stream and caller.
 */
#define QMM_STATUS_BAD_ID 0x1    /* qmm_id met an expert id outside [0, E) */
#define QMM_STATUS_TIMEOUT 0x2   /* a bounded wait in a kernel gave up (about one second); that call's
                                    output is incomplete, the device stays usable */
int qmm_get_status(void *stream);

/*
 * qmm_debug_stall (test/diagnostic only): qmm() on the mat-vec path (a quantized type, M <= 16) with
 * the warps of the first thread block made to wait for their first weight stage on a barrier that nothing
 * signals. Those bounded waits run out after about one second: each such warp records QMM_STATUS_TIMEOUT,
 * waits (bounded) for the weight copies still in flight into its shared memory, skips its share of the
 * work, and the kernel returns normally, so y is incomplete but the device and later calls are
 * unaffected. Exists to test the failure path without faulting or hanging a GPU. Returns QMM_ERANGE for
 * plain types or M > 16.
 */
int qmm_debug_stall(const void *wq, int qtype, int64_t N, int64_t K, const void *x, int64_t M, float *y,
                    void *stream);

const char *qmm_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* QMM_H */

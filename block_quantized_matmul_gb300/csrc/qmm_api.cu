// qmm_api.cu -- the extern "C" entry points of libqmm: host-side validation, then one or more
// kernel launches on the caller's stream.  Nothing here allocates device memory.
//
// Following the pages' guidance on host-side precomputation ("Op and Kernel Development
// Guidelines": shapes, strides, tiling and validation are settled on the host before the kernel
// runs), every check below happens before anything is enqueued, and the kernels trust their
// parameters.
#include "qmm_internal.cuh"

using namespace qmm;

namespace {

bool valid_type(qmm_type t) {
    return t == QMM_Q4_0 || t == QMM_Q8_0 || t == QMM_IQ4_NL || t == QMM_MXFP4 || t == QMM_Q4_1 || t == QMM_Q4_K;
}
// Flat blocks of 18 or 34 bytes are read as halfwords, Q4_1's 20-byte blocks start with a 4-byte
// (d, m) pair read as one word, Q4_K's 144-byte super-blocks are read as words, and MXFP4's
// 17-byte blocks are read byte by byte.
uintptr_t flat_align(qmm_type t) { return t == QMM_MXFP4 ? 1 : ((t == QMM_Q4_1 || t == QMM_Q4_K) ? 4 : 2); }
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_kn(int64_t K, int64_t N) { return K > 0 && (K % 32) == 0 && N > 0; }
// K must also be a whole number of the type's flat blocks (256 for Q4_K, whose tiles come from
// super-blocks).
bool valid_tkn(qmm_type t, int64_t K, int64_t N) { return valid_kn(K, N) && (K % block_len(t)) == 0; }
cudaStream_t cs(qmm_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }
qmm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

// Prefill product with a workspace: the GEMM with the token scales folded into the tensor-core operand
// for the tile types it covers, the exact-integer GEMM with a prepared token operand for the affine
// tiles (t is already a tile type).
cudaError_t launch_prefill_ws(qmm_type t, const uint8_t *w, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                              int64_t M, float *y, int64_t ldy, void *ws, cudaStream_t s) {
    if (gemm_fold_supports(t)) return launch_gemm_fold(t, w, K, N, a_q, a_d, M, y, ldy, ws, s);
    return launch_gemm_ws(t, w, K, N, a_q, a_d, M, y, ldy, ws, s);
}

// Sizes are capped so every byte offset fits comfortably in int64 arithmetic on both sides.
constexpr int64_t kMaxDim = (int64_t)1 << 31;

qmm_status check_matmul(qmm_type t, const void *w, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                        int64_t M, float *y, int64_t ldy) {
    if (!valid_type(t)) return QMM_ERR_UNSUPPORTED;
    if (!valid_tkn(t, K, N) || M <= 0 || K > kMaxMatmulK || N > kMaxDim || M > kMaxDim || ldy < N) return QMM_ERR_INVALID_ARG;
    if (!w || !a_q || !a_d || !y) return QMM_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(a_q, 16) || !aligned(a_d, 4) || !aligned(y, 4)) return QMM_ERR_MISALIGNED;
    return QMM_OK;
}

}  // namespace

extern "C" {

const char *qmm_status_str(qmm_status st) {
    switch (st) {
        case QMM_OK: return "ok";
        case QMM_ERR_INVALID_ARG: return "invalid argument";
        case QMM_ERR_UNSUPPORTED: return "unsupported type or path";
        case QMM_ERR_MISALIGNED: return "misaligned pointer or stride";
        case QMM_ERR_CUDA: return "CUDA error";
        case QMM_ERR_TIMEOUT: return "device pipeline wait timed out";
        case QMM_ERR_RANGE: return "operand row not exactly representable in the folded-scale GEMM";
        case QMM_ERR_BOUNDS: return "device bounds check failed (debug build)";
    }
    return "unknown status";
}

size_t qmm_block_size(qmm_type t) { return valid_type(t) ? (size_t)block_bytes(t) : 0; }

size_t qmm_tile_size(qmm_type t) { return valid_type(t) ? (size_t)tile_bytes(t) : 0; }

size_t qmm_tiled_size(qmm_type t, int64_t K, int64_t N) {
    if (!valid_type(t) || !valid_tkn(t, K, N) || K > kMaxDim || N > kMaxDim) return 0;
    return (size_t)((N + 31) / 32) * (size_t)(K / 32) * (size_t)tile_bytes(t);
}

size_t qmm_flat_size(qmm_type t, int64_t K, int64_t N) {
    if (!valid_type(t) || !valid_tkn(t, K, N) || K > kMaxDim || N > kMaxDim) return 0;
    return (size_t)N * (size_t)(K / 32) * (size_t)bytes_per_32(t);
}

void qmm_iq4nl_table(int8_t out[16]) {
    if (!out) return;
    for (int i = 0; i < 16; ++i) out[i] = kIq4nlTable[i];
}

int64_t qmm_decode_max_m(void) { return kDecodeMaxM; }

qmm_status qmm_quantize_weight(qmm_type t, const float *w, int64_t N, int64_t K, int64_t ldw, void *w_flat,
                               qmm_stream_t stream) {
    if (!valid_type(t)) return QMM_ERR_UNSUPPORTED;
    if (!valid_tkn(t, K, N) || K > kMaxDim || N > kMaxDim || ldw < K || !w || !w_flat) return QMM_ERR_INVALID_ARG;
    if (!aligned(w, 16) || (ldw % 4) != 0 || !aligned(w_flat, flat_align(t))) return QMM_ERR_MISALIGNED;
    return from_cuda(launch_quantize_weight(t, w, N, K, ldw, static_cast<uint8_t *>(w_flat), cs(stream)));
}

qmm_status qmm_repack(qmm_type t, const void *w_flat, int64_t K, int64_t N, void *w_tiled, qmm_stream_t stream) {
    if (!valid_type(t)) return QMM_ERR_UNSUPPORTED;
    if (!valid_tkn(t, K, N) || K > kMaxDim || N > kMaxDim || !w_flat || !w_tiled) return QMM_ERR_INVALID_ARG;
    if (!aligned(w_flat, flat_align(t)) || !aligned(w_tiled, 16)) return QMM_ERR_MISALIGNED;
    return from_cuda(launch_repack(t, static_cast<const uint8_t *>(w_flat), K, N, static_cast<uint8_t *>(w_tiled),
                                   cs(stream)));
}

qmm_status qmm_unpack(qmm_type t, const void *w_tiled, int64_t K, int64_t N, void *w_flat, qmm_stream_t stream) {
    if (!valid_type(t) || t == QMM_Q4_K) return QMM_ERR_UNSUPPORTED;   // Q4_K tiles hold rounded products
    if (!valid_kn(K, N) || K > kMaxDim || N > kMaxDim || !w_flat || !w_tiled) return QMM_ERR_INVALID_ARG;
    if (!aligned(w_flat, flat_align(t)) || !aligned(w_tiled, 16)) return QMM_ERR_MISALIGNED;
    return from_cuda(launch_unpack(t, static_cast<const uint8_t *>(w_tiled), K, N, static_cast<uint8_t *>(w_flat),
                                   cs(stream)));
}

qmm_status qmm_quantize_act(const float *x, int64_t M, int64_t K, int64_t ldx, int8_t *a_q, uint16_t *a_d,
                            qmm_stream_t stream) {
    if (M <= 0 || K <= 0 || (K % 32) != 0 || ldx < K || M > kMaxDim || K > kMaxDim || !x || !a_q || !a_d)
        return QMM_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(a_q, 16) || !aligned(a_d, 4)) return QMM_ERR_MISALIGNED;
    return from_cuda(launch_quantize_act(x, M, K, ldx, a_q, a_d, cs(stream)));
}

qmm_status qmm_matmul_path(qmm_type t, const void *w_tiled, int64_t K, int64_t N, const int8_t *a_q,
                           const uint16_t *a_d, int64_t M, float *y, int64_t ldy, qmm_path path,
                           qmm_stream_t stream) {
    qmm_status st = check_matmul(t, w_tiled, K, N, a_q, a_d, M, y, ldy);
    if (st != QMM_OK) return st;
    if (path != QMM_PATH_AUTO && path != QMM_PATH_MATVEC && path != QMM_PATH_GEMM) return QMM_ERR_UNSUPPORTED;
    const uint8_t *w = static_cast<const uint8_t *>(w_tiled);
    t = tile_type(t);
    if (path == QMM_PATH_AUTO) path = (M <= kDecodeMaxM) ? QMM_PATH_MATVEC : QMM_PATH_GEMM;
    cudaError_t e;
    if (path == QMM_PATH_MATVEC) {
        e = launch_matvec(t, w, K, N, a_q, a_d, M, y, ldy, cs(stream));
    } else {
        e = launch_gemm(t, w, K, N, a_q, a_d, M, y, ldy, cs(stream));
        if (e == cudaErrorNotSupported) return QMM_ERR_UNSUPPORTED;
    }
    return from_cuda(e);
}

qmm_status qmm_matmul(qmm_type t, const void *w_tiled, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                      int64_t M, float *y, int64_t ldy, qmm_stream_t stream) {
    return qmm_matmul_path(t, w_tiled, K, N, a_q, a_d, M, y, ldy, QMM_PATH_AUTO, stream);
}

static qmm_status check_matmul_f32(qmm_type t, const void *w_tiled, int64_t K, int64_t N, const float *x, int64_t ldx,
                                   int64_t M, float *y, int64_t ldy) {
    if (!valid_type(t)) return QMM_ERR_UNSUPPORTED;
    if (!valid_tkn(t, K, N) || M <= 0 || K > kMaxMatmulK || N > kMaxDim || M > kMaxDim || ldx < K || ldx > kMaxDim || ldy < N)
        return QMM_ERR_INVALID_ARG;
    if (!w_tiled || !x || !y) return QMM_ERR_INVALID_ARG;
    if (!aligned(w_tiled, 16) || !aligned(x, 4) || !aligned(y, 4)) return QMM_ERR_MISALIGNED;
    return QMM_OK;
}

// Where p points: 1 page-locked host memory, 0 device (or managed) memory, -1 memory the driver does
// not know (pageable host memory, which the kernels must not touch).  One driver query
// (cuPointerGetAttribute, looked up once through the runtime), or the runtime's attribute query if
// the driver entry point is unavailable.
using PointerAttrFn = CUresult (*)(void *, CUpointer_attribute, CUdeviceptr);
static int mem_where(const void *p) {
    static const PointerAttrFn fn = []() -> PointerAttrFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PointerAttrFn>(ptr);
        return nullptr;
    }();
    if (fn) {
        unsigned type = 0;
        if (fn(&type, CU_POINTER_ATTRIBUTE_MEMORY_TYPE, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return -1;
        return type == CU_MEMORYTYPE_HOST ? 1 : 0;
    }
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (at.type == cudaMemoryTypeHost) return 1;
    return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) ? 0 : -1;
}

qmm_status qmm_matmul_f32(qmm_type t, const void *w_tiled, int64_t K, int64_t N, const float *x, int64_t ldx,
                          int64_t M, float *y, int64_t ldy, qmm_stream_t stream) {
    const qmm_status st = check_matmul_f32(t, w_tiled, K, N, x, ldx, M, y, ldy);
    if (st != QMM_OK) return st;
    const int wx = mem_where(x);
    if (wx < 0 || mem_where(y) < 0) return QMM_ERR_INVALID_ARG;
    return from_cuda(launch_matvec_fused(tile_type(t), static_cast<const uint8_t *>(w_tiled), K, N, x, ldx, M, y, ldy,
                                         cs(stream), wx));
}

size_t qmm_matmul_f32_workspace_size(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || (K % 32) != 0 || M > kMaxDim || K > kMaxMatmulK) return 0;
    return ((size_t)M * (size_t)K * 4 + 255) / 256 * 256;
}

qmm_status qmm_matmul_f32_ws(qmm_type t, const void *w_tiled, int64_t K, int64_t N, const float *x, int64_t ldx,
                             int64_t M, float *y, int64_t ldy, void *workspace, size_t workspace_bytes,
                             qmm_stream_t stream) {
    const qmm_status st = check_matmul_f32(t, w_tiled, K, N, x, ldx, M, y, ldy);
    if (st != QMM_OK) return st;
    if (!workspace || workspace_bytes < qmm_matmul_f32_workspace_size(M, K)) return QMM_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return QMM_ERR_MISALIGNED;
    const uint8_t *w = static_cast<const uint8_t *>(w_tiled);
    const int wx = mem_where(x);
    if (wx < 0 || mem_where(y) < 0) return QMM_ERR_INVALID_ARG;
    if (wx == 0)                                 // device rows: the workspace is not needed
        return from_cuda(launch_matvec_fused(tile_type(t), w, K, N, x, ldx, M, y, ldy, cs(stream), 0));
    float *rows = static_cast<float *>(workspace);
    cudaError_t e = launch_stage_rows(x, M, K, ldx, rows, cs(stream));
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(launch_matvec_fused(tile_type(t), w, K, N, rows, K, M, y, ldy, cs(stream), 0));
}

qmm_status qmm_matmul_flat(qmm_type t, const void *w_flat, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                           int64_t M, float *y, int64_t ldy, qmm_stream_t stream) {
    qmm_status st = check_matmul(t, w_flat, K, N, a_q, a_d, M, y, ldy);
    if (st != QMM_OK) return st;
    if (((K / 32) * bytes_per_32(t)) % 16 != 0) return QMM_ERR_UNSUPPORTED;   // rows are copied as 16-byte units
    return from_cuda(launch_matvec_flat(t, static_cast<const uint8_t *>(w_flat), K, N, a_q, a_d, M, y, ldy, cs(stream)));
}

size_t qmm_matmul_workspace_size(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || (K % 32) != 0 || M > kMaxDim || K > kMaxDim) return 0;
    return gemm_workspace_bytes(M, K);
}

qmm_status qmm_matmul_ws(qmm_type t, const void *w_tiled, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                         int64_t M, float *y, int64_t ldy, void *workspace, size_t workspace_bytes,
                         qmm_stream_t stream) {
    qmm_status st = check_matmul(t, w_tiled, K, N, a_q, a_d, M, y, ldy);
    if (st != QMM_OK) return st;
    const uint8_t *w = static_cast<const uint8_t *>(w_tiled);
    t = tile_type(t);
    if (M <= kDecodeMaxM) return from_cuda(launch_matvec(t, w, K, N, a_q, a_d, M, y, ldy, cs(stream)));
    if (!workspace || workspace_bytes < gemm_workspace_bytes(M, K)) return QMM_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return QMM_ERR_MISALIGNED;
    return from_cuda(launch_prefill_ws(t, w, K, N, a_q, a_d, M, y, ldy, workspace, cs(stream)));
}

qmm_status qmm_matmul_noalloc(qmm_type t, const void *w_tiled, int64_t K, int64_t N, const int8_t *a_q,
                              const uint16_t *a_d, int64_t M, float *y, int64_t ldy, qmm_stream_t stream) {
    qmm_status st = check_matmul(t, w_tiled, K, N, a_q, a_d, M, y, ldy);
    if (st != QMM_OK) return st;
    const uint8_t *w = static_cast<const uint8_t *>(w_tiled);
    t = tile_type(t);
    if (M <= kDecodeMaxM) return from_cuda(launch_matvec(t, w, K, N, a_q, a_d, M, y, ldy, cs(stream)));
    if (gemm_workspace_bytes(M, K) > kNoAllocScratchBytes) return QMM_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return QMM_ERR_CUDA;
    return from_cuda(launch_prefill_ws(t, w, K, N, a_q, a_d, M, y, ldy, scratch, cs(stream)));
}

size_t qmm_matmul_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

qmm_status qmm_selftest_timeout(int unit, uint64_t limit_ns, int *flags_dev, qmm_stream_t stream) {
    if (unit < 0 || unit > 2 || limit_ns < 1000000ull || limit_ns > 2000000000ull || !flags_dev)
        return QMM_ERR_INVALID_ARG;
    if (!aligned(flags_dev, 4)) return QMM_ERR_MISALIGNED;
    return from_cuda(unit == 0   ? launch_selftest_wait_mv(limit_ns, flags_dev, cs(stream))
                     : unit == 1 ? launch_selftest_wait_gemm(limit_ns, flags_dev, cs(stream))
                                 : launch_selftest_wait_fold(limit_ns, flags_dev, cs(stream)));
}

qmm_status qmm_device_status(qmm_stream_t stream) {
    unsigned v = 0, w = 0, f = 0;
    cudaError_t e = read_and_clear_device_status(&v, cs(stream));
    if (e == cudaSuccess) e = read_and_clear_matvec_status(&w, cs(stream));
    if (e == cudaSuccess) e = read_and_clear_fold_status(&f, cs(stream));
    // the bounds-check words (always 0 unless the library was built with QMM_DEBUG)
    unsigned d[5] = {0, 0, 0, 0, 0};
    if (e == cudaSuccess) e = read_dcheck_matvec(&d[0], cs(stream));
    if (e == cudaSuccess) e = read_dcheck_gemm(&d[1], cs(stream));
    if (e == cudaSuccess) e = read_dcheck_fold(&d[2], cs(stream));
    if (e == cudaSuccess) e = read_dcheck_quant(&d[3], cs(stream));
    if (e == cudaSuccess) e = read_dcheck_repack(&d[4], cs(stream));
    if (e != cudaSuccess) return QMM_ERR_CUDA;
    if (d[0] | d[1] | d[2] | d[3] | d[4]) return QMM_ERR_BOUNDS;
    if (v | w | (f & 1u)) return QMM_ERR_TIMEOUT;
    return (f & 2u) ? QMM_ERR_RANGE : QMM_OK;
}

}  // extern "C"

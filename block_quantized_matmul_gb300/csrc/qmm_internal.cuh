// qmm_internal.cuh -- declarations shared by the libqmm translation units (product code only).
#pragma once

#include <cuda.h>   // CUtensorMap and its enums (the encoder is fetched through the runtime)
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/qmm.h"

namespace qmm {

constexpr int kTileRows = 32;         // rows (N) per tile
constexpr int kTileCols = 32;         // columns (K) per tile = elements per GGML block
constexpr int kTile4Bytes = 576;      // Q4_0 / IQ4_NL tile
constexpr int kTile8Bytes = 1088;     // Q8_0 tile
constexpr int kScale4Off = 512;       // FP16 row scales inside a 4-bit tile
constexpr int kScale8Off = 1024;      // FP16 row scales inside a Q8_0 tile
constexpr int kBlock4Bytes = 18;      // flat GGML block: fp16 d + 16 nibble bytes
constexpr int kBlock8Bytes = 34;      // flat GGML block: fp16 d + 32 int8
constexpr int kTileMxBytes = 544;     // MXFP4 tile: 512 nibble bytes + 32 E8M0 exponent bytes
constexpr int kBlockMxBytes = 17;     // flat MXFP4 block: E8M0 e + 16 nibble bytes
constexpr int kTile41Bytes = 640;     // Q4_1 tile: 512 nibble bytes + 32 fp16 (d, m) pairs
constexpr int kBlock41Bytes = 20;     // flat Q4_1 block: fp16 d + fp16 m + 16 nibble bytes
constexpr int kSuperQ4KBytes = 144;   // flat Q4_K super-block of 256: fp16 d, fp16 dmin, 12 scale bytes, 128 nibble bytes
constexpr int kQ4KBytesPer32 = 18;    // the same, per 32 weights

inline int tile_bytes(qmm_type t) {
    return t == QMM_Q8_0 ? kTile8Bytes
                         : (t == QMM_MXFP4 ? kTileMxBytes : ((t == QMM_Q4_1 || t == QMM_Q4_K) ? kTile41Bytes : kTile4Bytes));
}
// Bytes of one flat GGML block (Q4_K: one super-block of 256 weights).
inline int block_bytes(qmm_type t) {
    return t == QMM_Q8_0 ? kBlock8Bytes
                         : (t == QMM_MXFP4 ? kBlockMxBytes
                                           : (t == QMM_Q4_1 ? kBlock41Bytes : (t == QMM_Q4_K ? kSuperQ4KBytes : kBlock4Bytes)));
}
// Flat bytes per 32 weights (every type's row is K/32 times this).
inline int bytes_per_32(qmm_type t) { return t == QMM_Q4_K ? kQ4KBytesPer32 : block_bytes(t); }
// Elements per flat block.
inline int block_len(qmm_type t) { return t == QMM_Q4_K ? 256 : 32; }
// The tile a type is stored in for the tiled kernels: a Q4_K tile is a Q4_1 tile.
inline qmm_type tile_type(qmm_type t) { return t == QMM_Q4_K ? QMM_Q4_1 : t; }

// Per-type constants for the kernels.
template <int TYPE>
struct TileFmt {
    static constexpr int kBytes = TYPE == QMM_Q8_0                        ? kTile8Bytes
                                  : TYPE == QMM_MXFP4                     ? kTileMxBytes
                                  : (TYPE == QMM_Q4_1 || TYPE == QMM_Q4_K) ? kTile41Bytes
                                                                          : kTile4Bytes;
    static constexpr int kScaleOff = TYPE == QMM_Q8_0 ? kScale8Off : kScale4Off;   // MXFP4, Q4_1: 512 too
    static constexpr bool kLut = TYPE == QMM_IQ4_NL || TYPE == QMM_MXFP4;         // codes go through a table
    static constexpr bool kE8M0 = TYPE == QMM_MXFP4;                              // one exponent byte per row
    static constexpr bool kAffine = TYPE == QMM_Q4_1 || TYPE == QMM_Q4_K;         // (d, m) per row: d*q + m
    static constexpr bool kNibbleInt = TYPE == QMM_Q4_0 || kAffine;               // integer nibble codes
};

// The built-in IQ4_NL table (16 int8 levels, ascending): the levels of GGML's published IQ4_NL
// format, so that IQ4_NL weights quantized elsewhere (GGUF files) decode to their own values.  The
// pages name the table (iq4_nl_to_fp16_lut) without printing it.  Every level is an integer in
// [-127, 113], so every block sum stays an exact integer.
constexpr int8_t kIq4nlTable[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};

// Table passed by value to kernels (host-side precomputed parameters, no device-global state).
struct Lut16 {
    int8_t v[16];
};
inline Lut16 iq4nl_lut() {
    Lut16 l;
    for (int i = 0; i < 16; ++i) l.v[i] = kIq4nlTable[i];
    return l;
}

// MXFP4 codes as integers: twice the OCP FP4 (E2M1) value of code = sign<<3 | exponent<<1 | mantissa
// ({0, 0.5, 1, 1.5, 2, 3, 4, 6} with the sign), so that the block sums stay exact integers.  The
// matching block scale is half the fp16 scale (mx_half_scale).
constexpr int8_t kMxfp4Twice[16] = {0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12};
inline Lut16 mxfp4_lut() {
    Lut16 l;
    for (int i = 0; i < 16; ++i) l.v[i] = kMxfp4Twice[i];
    return l;
}
inline Lut16 lut_for(qmm_type t) { return t == QMM_MXFP4 ? mxfp4_lut() : iq4nl_lut(); }

// The pages' E8M0 -> fp16 scale: fp16 bits f << 10 with f = clamp(e - 112, 0, 30), i.e. 2^(f - 15), or 0
// when f = 0.  Half of it (the scale of the doubled integer codes) as an exact fp32: 2^(f - 16).
__host__ __device__ __forceinline__ float mx_half_scale(uint32_t e) {
    int f = (int)e - 112;
    f = f < 0 ? 0 : (f > 30 ? 30 : f);
    const uint32_t bits = f ? (uint32_t)(f + 127 - 16) << 23 : 0u;
    float v;
    memcpy(&v, &bits, 4);
    return v;
}

// ---- the dynamic Q8_0 activation rule, per block of 32 (also the Q8_0 weight rule) ----
// amax = max|x|, d = amax/127, id = d ? 1/d : 0, q = round half away from zero of x*id clamped to
// [-127, 127] (a NaN product, 0*inf after 1/d overflowed, gives 0); the stored scale is fp16(d).
// IEEE-rounded fp32 intrinsics throughout, so nothing is contracted or reassociated.
__device__ __forceinline__ float q8_scale(float amax) { return __fdiv_rn(amax, 127.0f); }
__device__ __forceinline__ float inv_or_zero(float d) { return d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f; }
__device__ __forceinline__ int q8_code(float x, float id) {
    float v = __fmul_rn(x, id);
    if (isnan(v)) return 0;
    float r = roundf(v);                       // halfway cases away from zero
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int)r;
}

// Activation source of the decode kernels: quantized rows (a_q, a_d) or fp32 rows x quantized
// inside the kernel (x != nullptr).
struct ActSrc {
    const int8_t *a_q;
    const uint16_t *a_d;
    const float *x;
    int64_t ldx;
    int x_host;       // x lives in host memory (read over NVLink-C2C)
};

// Launchers (each returns cudaGetLastError() after enqueueing).
cudaError_t launch_quantize_act(const float *x, int64_t M, int64_t K, int64_t ldx, int8_t *a_q,
                                uint16_t *a_d, cudaStream_t s);
cudaError_t launch_stage_rows(const float *x, int64_t M, int64_t K, int64_t ldx, float *dst, cudaStream_t s);
cudaError_t launch_quantize_weight(qmm_type t, const float *w, int64_t N, int64_t K, int64_t ldw,
                                   uint8_t *flat, cudaStream_t s);
cudaError_t launch_repack(qmm_type t, const uint8_t *flat, int64_t K, int64_t N, uint8_t *tiled,
                          cudaStream_t s);
cudaError_t launch_unpack(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, uint8_t *flat,
                          cudaStream_t s);
cudaError_t launch_matvec(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                          const uint16_t *a_d, int64_t M, float *y, int64_t ldy, cudaStream_t s);
// 2-D tensor map: rows of `inner` elements (row stride `row_bytes`), box {box_inner, box_rows}.
cudaError_t make_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw);
// 3-D tensor map of the tiled weight as [n_col_tiles][n_k_tiles][tile bytes / 8] 8-byte words, one box
// = 4 column tiles x 2 K tiles (column tiles past the end read as zeros).
cudaError_t make_weight_map(CUtensorMap *map, const uint8_t *tiled, int tile_bytes, int64_t nkt, int64_t nct);
// Decode matmul straight from flat GGML rows (row bytes a multiple of 16, flat 16-byte aligned).
cudaError_t launch_matvec_flat(qmm_type t, const uint8_t *flat, int64_t K, int64_t N, const int8_t *a_q,
                               const uint16_t *a_d, int64_t M, float *y, int64_t ldy, cudaStream_t s);
// x_host: the rows are in page-locked host memory (the int8 path then shares them across clusters).
cudaError_t launch_matvec_fused(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const float *x, int64_t ldx,
                                int64_t M, float *y, int64_t ldy, cudaStream_t s, int x_host);
cudaError_t launch_gemm(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                        const uint16_t *a_d, int64_t M, float *y, int64_t ldy, cudaStream_t s);
cudaError_t launch_gemm_ws(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                           const uint16_t *a_d, int64_t M, float *y, int64_t ldy, void *ws, cudaStream_t s);
size_t gemm_workspace_bytes(int64_t M, int64_t K);
// The folded-scale GEMM (block scales inside exact hi + lo fp16 operands): Q4_0, Q8_0, IQ4_NL tiles.
bool gemm_fold_supports(qmm_type t);
cudaError_t launch_gemm_fold(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                             const uint16_t *a_d, int64_t M, float *y, int64_t ldy, void *ws, cudaStream_t s);
cudaError_t read_and_clear_fold_status(unsigned *out, cudaStream_t s);

// Workspace of the tensor-core GEMMs, each region 256-byte aligned.  The exact-integer kernel uses
// hi (fp16 copies of the int8 quants), dT (block scales transposed, [K/32][M_pad] fp16) and cA
// (Q4_1: d_a * sum(a_q), [K/32][M_pad] fp32); the folded-scale kernel uses hi and lo (the two fp16
// terms of d_a * a_q, [M][K] each) and ts (per token row, the power of two it was scaled by).
struct GemmWsLayout {
    size_t hi, lo, dT, cA, ts, total;
};
inline size_t round256(size_t v) { return (v + 255) / 256 * 256; }
inline GemmWsLayout gemm_ws_layout(int64_t M, int64_t K) {
    const size_t m_pad = (size_t)((M + 7) / 8 * 8), nkt = (size_t)(K / 32), mk2 = (size_t)M * (size_t)K * 2;
    GemmWsLayout L;
    L.hi = 0;
    L.lo = round256(mk2);
    L.dT = L.lo + round256(mk2);
    L.cA = L.dT + round256(nkt * m_pad * 2);
    L.ts = L.cA + round256(nkt * m_pad * 4);
    L.total = L.ts + round256((size_t)M * 4);
    return L;
}

// ---- device bounds checks (QMM_DEBUG builds) ----
// QMM_DCHECK(cond) is `true` in release builds, so the compiler drops it and the branch it guards.
// Built with -DQMM_DEBUG it evaluates cond; when cond fails it records the source line in this
// translation unit's check word (the first failure stays) and yields false, and the caller skips the
// access it guards -- nothing traps.  qmm_device_status() reports a recorded failure as
// QMM_ERR_BOUNDS.  Each file with kernels defines its word's reader with QMM_DCHECK_READER(name).
#ifdef QMM_DEBUG
static __device__ unsigned g_dcheck_line = 0;
__device__ __forceinline__ bool dcheck(bool ok, unsigned line) {
    if (!ok) atomicCAS(&g_dcheck_line, 0u, line);
    return ok;
}
#define QMM_DCHECK(cond) (::qmm::dcheck((cond), __LINE__))
#define QMM_DCHECK_READER(name)                                                                       \
    cudaError_t name(unsigned *out, cudaStream_t s) {                                                 \
        unsigned zero = 0;                                                                            \
        cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_dcheck_line, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s); \
        if (e == cudaSuccess)                                                                         \
            e = cudaMemcpyToSymbolAsync(g_dcheck_line, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s); \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                                           \
        return e;                                                                                     \
    }
#else
#define QMM_DCHECK(cond) (true)
#define QMM_DCHECK_READER(name)                        \
    cudaError_t name(unsigned *out, cudaStream_t) {    \
        *out = 0;                                      \
        return cudaSuccess;                            \
    }
#endif
// The readers: the source line of the first failed check in each file since the last read, or 0.
cudaError_t read_dcheck_matvec(unsigned *out, cudaStream_t s);
cudaError_t read_dcheck_gemm(unsigned *out, cudaStream_t s);
cudaError_t read_dcheck_fold(unsigned *out, cudaStream_t s);
cudaError_t read_dcheck_quant(unsigned *out, cudaStream_t s);
cudaError_t read_dcheck_repack(unsigned *out, cudaStream_t s);

// Fixed device scratch used by qmm_matmul_noalloc (bytes, per device).
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
cudaError_t noalloc_scratch(void **out);
cudaError_t read_and_clear_device_status(unsigned *out, cudaStream_t s);   // tensor-core GEMM
cudaError_t read_and_clear_matvec_status(unsigned *out, cudaStream_t s);   // decode matvec
// One CTA whose bounded waits run out on purpose (decode kernels' and GEMM's wait helpers).
cudaError_t launch_selftest_wait_mv(unsigned long long limit_ns, int *out, cudaStream_t s);
cudaError_t launch_selftest_wait_gemm(unsigned long long limit_ns, int *out, cudaStream_t s);
cudaError_t launch_selftest_wait_fold(unsigned long long limit_ns, int *out, cudaStream_t s);

// Raises a kernel's dynamic shared-memory limit once per device (the attribute is per device and
// per function, and setting it on every call costs host time on the launch path).
// `done_mask` must be a static owned by the caller's (kernel-specific) launcher: bit d is set once the
// attribute is in place on device d (devices 0..127; others set it on every call).
template <typename Kern>
inline cudaError_t ensure_smem_limit(Kern kern, size_t bytes, int (&done_mask)[4]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < 128;
    if (cacheable && (__atomic_load_n(&done_mask[dev >> 5], __ATOMIC_ACQUIRE) >> (dev & 31)) & 1) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && cacheable) __atomic_fetch_or(&done_mask[dev >> 5], 1 << (dev & 31), __ATOMIC_RELEASE);
    return e;
}

// Largest M handled by one decode-matvec launch (two 8-token mma fragments).
constexpr int kDecodeMaxM = 16;

// Blocks of 32 that the exact-integer GEMM sums per output in a register before adding the partial
// into y, and the largest K any product call accepts: the fp32 accumulation error of every kernel
// stays below 1e-5 * sum_k |w_k x_k| up to this K (131072 = 4096 blocks).
constexpr int kGemmChunkBlocks = 128;
constexpr int64_t kMaxMatmulK = (int64_t)1 << 17;

}  // namespace qmm

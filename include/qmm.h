/*
 * qmm.h -- C ABI of libqmm: matrix multiply over block-32 quantized weights stored in 32-row tiles,
 * with activations dynamically quantized to Q8_0 blocks, on one NVIDIA GB300 GPU (sm_103a).
 *
 * Layouts follow "Hexagon backend developer details", section "Tiled Weight Formats":
 *   - "Tile Dimensions and Grid Layout": a weight of logical shape [ne0 = K, ne1 = N] is cut into
 *     tiles of 32 rows (N) x 32 columns (K).  n_k_tiles = K/32, n_col_tiles = (N+31)/32,
 *     tile_idx = ct*n_k_tiles + kt and the tile starts at byte tile_idx*tile_size.
 *   - "Block-32 Quantized Formats": Q4_0 and IQ4_NL tiles are 576 bytes (byte cp*32+row holds
 *     column 2cp in its low nibble and 2cp+1 in its high nibble, cp = 0..15; 32 FP16 row scales at
 *     bytes 512..575); Q8_0 tiles are 1088 bytes (bytes cp*64+2*row and cp*64+2*row+1 hold columns
 *     2cp and 2cp+1 as int8; 32 FP16 row scales at bytes 1024..1087).  IQ4_NL quants are indices
 *     into a 16-entry non-linear table.
 *
 * Conventions for every call below:
 *   - Pointers named *_dev are addresses the GPU accesses directly: device memory, except where a
 *     call says otherwise (qmm_matmul_f32 also takes x and y in page-locked host memory, which on
 *     GB300 its kernel reads and writes over the coherent NVLink-C2C link).  The caller owns every
 *     buffer and the stream.  The library allocates no device memory and keeps no per-call state.
 *   - Calls that take a stream only validate their arguments on the host and enqueue work on that
 *     stream; they return before the GPU has run.  `stream` is a cudaStream_t (NULL = legacy
 *     default stream).  Calls on different streams with distinct outputs may run concurrently.
 *   - Argument errors are reported before anything is enqueued; a failed launch returns
 *     QMM_ERR_CUDA.  Nothing is thrown and nothing aborts across this interface.
 *   - fp16 values are IEEE binary16 bit patterns in uint16_t, little-endian in memory.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                        /* cudaStream_t is `struct CUstream_st *` */
typedef struct CUstream_st *qmm_stream_t;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1,   /* a size, stride or required pointer is invalid */
    QMM_ERR_UNSUPPORTED = 2,   /* type or path not implemented */
    QMM_ERR_MISALIGNED = 3,    /* a pointer or stride violates the stated alignment */
    QMM_ERR_CUDA = 4,          /* the CUDA runtime reported an error at launch */
    QMM_ERR_TIMEOUT = 5,       /* a kernel gave up waiting on its own pipeline (see qmm_device_status) */
    QMM_ERR_RANGE = 6,         /* the folded-scale GEMM met an operand row it cannot represent exactly
                                  (see qmm_matmul_ws and qmm_device_status) */
    QMM_ERR_BOUNDS = 7         /* a device bounds check failed (builds with QMM_DEBUG only; see
                                  qmm_device_status) */
} qmm_status;

/* Weight formats ("Block-32 Quantized Formats").  MXFP4 tiles (544 B) hold OCP FP4 (E2M1) codes in
 * the Q4_0 nibble layout and one E8M0 exponent byte per row at byte 512 + row; a weight is the FP4
 * value of its code times the power-of-two fp16 scale with bits clamp(e - 112, 0, 30) << 10.
 * Q4_1 tiles (640 B) keep the Q4_0 nibble layout and one FP16 pair (d, m) per row at bytes
 * 512 + 4*row; a weight is d*q + m (q = 0..15).
 * Q4_K ("K-Quants Formats"): flat rows are GGML super-blocks of 256 weights (144 B: fp16 d, fp16 dmin,
 * 12 bytes packing a 6-bit scale sc_j and min m_j for each sub-block j of 32, then 128 nibble bytes;
 * weight i of sub-block j is nibble (j & 1) of byte 32*(j/2) + i, worth d*sc_j*q - dmin*m_j).  Each
 * super-block becomes 8 tiles of 32 k in the Q4_1 tile layout with the row pair
 * (fp16(d*sc_j), fp16(-dmin*m_j)), so every tiled call reads a Q4_K weight exactly as a Q4_1 one.
 * For Q4_K, K must be a multiple of 256 in every call. */
typedef enum { QMM_Q4_0 = 0, QMM_Q8_0 = 1, QMM_IQ4_NL = 2, QMM_MXFP4 = 3, QMM_Q4_1 = 4, QMM_Q4_K = 5 } qmm_type;

/* Which kernel qmm_matmul_path runs: AUTO picks the decode matvec for M <= qmm_decode_max_m()
 * and the exact-integer tensor-core GEMM otherwise (the folded-scale GEMM needs a workspace and
 * runs through qmm_matmul_ws / qmm_matmul_noalloc). */
typedef enum { QMM_PATH_AUTO = 0, QMM_PATH_MATVEC = 1, QMM_PATH_GEMM = 2 } qmm_path;

/* Human-readable name of a status code (static string, never NULL). */
QMM_API const char *qmm_status_str(qmm_status st);

/* Bytes of one flat GGML block of 32 weights: 18 (Q4_0, IQ4_NL: fp16 d + 16 nibble bytes, element
 * j in the low nibble of byte j, element j+16 in its high nibble), 34 (Q8_0: fp16 d + 32 int8) or
 * 17 (MXFP4: the E8M0 exponent byte + 16 nibble bytes in the same order) or 20 (Q4_1: fp16 d, fp16 m
 * + 16 nibble bytes); for Q4_K the 144-byte super-block of 256 weights.  0 for an unknown type. */
QMM_API size_t qmm_block_size(qmm_type t);

/* Bytes of one tile ("Block-32 Quantized Formats"): 576 (Q4_0, IQ4_NL), 1088 (Q8_0), 544 (MXFP4) or
 * 640 (Q4_1, Q4_K); 0 if unknown. */
QMM_API size_t qmm_tile_size(qmm_type t);

/* Bytes of the tiled weight [K, N] ("Tile Dimensions and Grid Layout"):
 * n_col_tiles * n_k_tiles * tile_size.  0 if K <= 0, K % 32 != 0, N <= 0 or the type is unknown. */
QMM_API size_t qmm_tiled_size(qmm_type t, int64_t K, int64_t N);

/* Bytes of the flat weight: N rows of K/32 GGML blocks (K/256 super-blocks for Q4_K).  0 on the
 * same invalid inputs, and for Q4_K when K % 256 != 0. */
QMM_API size_t qmm_flat_size(qmm_type t, int64_t K, int64_t N);

/* The 16-entry IQ4_NL table the kernels use (int8 values, ascending).  The pages name the table
 * (iq4_nl_to_fp16_lut) without printing it; the built-in one holds the 16 levels of GGML's
 * published IQ4_NL format {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113},
 * so IQ4_NL weights from GGUF files decode to their own values.  Writes 16 bytes to `out`. */
QMM_API void qmm_iq4nl_table(int8_t out[16]);

/* Largest activation row count M that QMM_PATH_AUTO sends to the decode matvec. */
QMM_API int64_t qmm_decode_max_m(void);

/*
 * qmm_quantize_weight -- fp32 weight rows -> flat GGML blocks (model-load helper, not the hot path).
 *   w_dev      fp32, N rows of K values, row n at w_dev + n*ldw; 16-byte aligned, ldw % 4 == 0.
 *   w_flat_dev output, qmm_flat_size(t, K, N) bytes, row-major blocks; 2-byte aligned (4-byte for
 *              Q4_1 and Q4_K, any address for MXFP4).
 * Rules per 32-element block (x = the block, m = its signed element of largest magnitude, first on
 * ties): Q8_0 d = max|x|/127, q = round-half-away(x/d) (computed as x * (1/d));  Q4_0 d = m/-8,
 * q = min(15, trunc(x*(1/d) + 8.5));  IQ4_NL d = m/table[0], q = the table index whose level
 * fp16(d)*table[q] is nearest to x (lowest index on ties).  d is stored rounded to fp16.
 * MXFP4: e = floor(log2 max|x|) - 2 + 127 (0 for an all-zero block, at most 254), then the code whose
 * level s * fp4(code) is nearest to x (lowest code on ties), s the dequantizing fp16 scale.
 * Q4_1: d = (max - min)/15, q = min(15, trunc((x - min)*(1/d) + 0.5)), m = min; d and m as fp16.
 * Q4_K, per super-block: for each sub-block mn = min(0, min x), scale = (max x - mn)/15, min = -mn;
 * d = max scale/63, dmin = max min/63 (fp16); sc, m = min(63, trunc(v*(63/max) + 0.5)); then
 * q = min(15, trunc((x + dmin*m) * (1/(d*sc)) + 0.5)) (0 when d*sc = 0).
 * Errors: INVALID_ARG (N <= 0, K <= 0, K % 32 (K % 256 for Q4_K), ldw < K, NULL), UNSUPPORTED
 * (type), MISALIGNED.
 */
QMM_API qmm_status qmm_quantize_weight(qmm_type t, const float *w_dev, int64_t N, int64_t K, int64_t ldw,
                               void *w_flat_dev, qmm_stream_t stream);

/*
 * qmm_repack -- flat GGML rows -> tiles ("Tiled Weight Formats"; the pages repack at model load,
 * in set_tensor() or rt-repack).
 *   w_flat_dev  N rows of K/32 blocks (qmm_flat_size bytes); 2-byte aligned (4-byte for Q4_1 and
 *               Q4_K, any address for MXFP4).
 *   w_tiled_dev output, qmm_tiled_size bytes; 16-byte aligned.  Rows past N in the last column tile
 *               are written as zero bytes (scale 0, quants 0).  The buffers must not overlap.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED.  Bit-exact, lossless, except for Q4_K, whose tile
 * pairs are d*sc and -dmin*m rounded to fp16 (exact fp32 products, round to nearest even; d and dmin
 * must be finite).
 */
QMM_API qmm_status qmm_repack(qmm_type t, const void *w_flat_dev, int64_t K, int64_t N, void *w_tiled_dev,
                      qmm_stream_t stream);

/* qmm_unpack -- inverse of qmm_repack (tiles -> flat rows); used to check a tiled buffer. Same
 * arguments and alignment rules with the roles of the two buffers swapped.  UNSUPPORTED for Q4_K
 * (its tiles cannot be split back into a super-block). */
QMM_API qmm_status qmm_unpack(qmm_type t, const void *w_tiled_dev, int64_t K, int64_t N, void *w_flat_dev,
                      qmm_stream_t stream);

/*
 * qmm_quantize_act -- dynamic Q8_0 quantization of activations (the pages quantize activations into
 * Q8_0 blocks before the matmul; "Memory buffers").
 *   x_dev  fp32, M rows of K values, row m at x_dev + m*ldx; 4-byte aligned (16-byte aligned with
 *          ldx % 4 == 0 takes the vectorised path).
 *   a_q_dev output int8 [M][K] (row stride K); 16-byte aligned.
 *   a_d_dev output fp16 bits [M][K/32], the scale of each block; 4-byte aligned.
 * Per block of 32: amax = max|x|, d = amax/127, id = (d != 0) ? 1/d : 0, q = round half away from
 * zero of x*id, clamped to [-127, 127] (a NaN product gives 0); a_d = fp16(d).  IEEE fp32 division
 * and rounding, no fused multiply-add, no flush-to-zero.  Inputs must be finite.
 * Errors: INVALID_ARG (M <= 0, K <= 0, K % 32, ldx < K, NULL), MISALIGNED.
 */
QMM_API qmm_status qmm_quantize_act(const float *x_dev, int64_t M, int64_t K, int64_t ldx, int8_t *a_q_dev,
                            uint16_t *a_d_dev, qmm_stream_t stream);

/*
 * qmm_matmul -- Y = A * W^T over tiled weights:
 *   Y[m, n] = sum_b fp32(d_w[n, b]) * fp32(d_a[m, b]) * S_b[m, n],
 *   S_b[m, n] = sum_{j<32} w_int[n, 32b+j] * a_q[m, 32b+j]  (exact integer block dot products),
 *   w_int = q-8 (Q4_0), q (Q8_0), table[q] (IQ4_NL), 2*fp4(q) with d_w = half the E8M0 scale
 *   (MXFP4); Q4_1 adds fp32(m_w[n, b]) * fp32(d_a[m, b]) * sum_j a_q[m, 32b+j] with w_int = q, and
 *   so does Q4_K, whose tile pair (d, m) is (d*sc, -dmin*m) of the super-block.
 *   w_tiled_dev  qmm_tiled_size bytes from qmm_repack; 16-byte aligned.
 *   a_q_dev, a_d_dev  as written by qmm_quantize_act for M rows and the same K.
 *   y_dev  fp32 output, y[m*ldy + n] for n < N (other columns untouched); 4-byte aligned.
 * Accumulation is fp32 in a fixed order (results are reproducible run to run); the error against
 * the exact value stays below 1e-5 * sum_k |w_k * x_k| (dequantized) for every accepted K: the
 * tensor-core GEMM runs K in passes of at most 4096 that add into y in order.  K may be at most
 * 131072 in every product call (qmm_matmul*, INVALID_ARG beyond).
 * Launch overlap (M <= qmm_decode_max_m()): the decode kernel is a programmatic dependent launch.
 * It may start while the kernel before it on the stream is finishing, and it starts streaming the
 * weight tiles at once; it waits for that kernel to complete before it reads a_q, a_d or y.  So
 * the tiles must not be written by the kernel launched immediately before this call if that
 * kernel itself lets dependents start early.  Tiles from qmm_repack (which makes its stores
 * visible before it exits), from a copy, or from any earlier kernel are fine.  qmm_quantize_act
 * is launched the same way and waits before it reads x.
 * Errors: INVALID_ARG (sizes, ldy < N, NULL), UNSUPPORTED, MISALIGNED, CUDA.
 */
QMM_API qmm_status qmm_matmul(qmm_type t, const void *w_tiled_dev, int64_t K, int64_t N, const int8_t *a_q_dev,
                      const uint16_t *a_d_dev, int64_t M, float *y_dev, int64_t ldy, qmm_stream_t stream);

/*
 * qmm_matmul_f32 -- the same product with the activation quantization fused into the decode kernel:
 * Y = Q8_0(x) * W^T, x given as fp32 rows.  The pages quantize the activations into Q8_0 blocks in
 * VTCM inside the op before the weight loop ("Memory buffers"); here every CTA quantizes the rows
 * it needs into shared memory while its weight stream starts.
 *   w_tiled_dev  as for qmm_matmul.
 *   x_dev  fp32, M rows of K values, row m at x_dev + m*ldx; 4-byte aligned (16-byte aligned with
 *          ldx % 4 == 0 takes the vectorised loads).  Inputs must be finite.
 *   y_dev  fp32 output as for qmm_matmul.
 * The quantization is the rule of qmm_quantize_act, bit for bit, and the result equals
 * qmm_quantize_act followed by qmm_matmul (same kernels' arithmetic, same order) for
 * M <= qmm_decode_max_m().  Meant for decode shapes: larger M runs the decode kernel on groups
 * of qmm_decode_max_m() rows, far slower than quantize + the tensor-core GEMM.  Nothing is
 * written but y; no workspace.  Launch overlap as for qmm_matmul (x is read only after the
 * preceding kernel has completed).
 * x and y may also live in page-locked host memory mapped for the device (cudaHostAlloc, or
 * cudaHostRegister with cudaHostRegisterMapped); the call checks where each points (one driver query
 * per pointer) and refuses pageable host memory, which the GPU must not touch, with INVALID_ARG
 * before anything is enqueued.  A decode step then reads x and writes y over NVLink-C2C inside the
 * kernel (same results, bit for bit).  Host memory is not cached in the GPU's L2, so every CTA that
 * reads x pays the link for it: with x in host memory and M <= 4 the decode kernel runs in
 * thread-block clusters of C = 2 to 8 CTAs, each CTA reading 1/C of the blocks and sharing them
 * through distributed shared memory (C is the largest whose clusters all fit on the GPU at once).
 * qmm_matmul_f32_ws reads x over the link only once.
 * Errors: INVALID_ARG (sizes, ldx < K, ldy < N, NULL, x or y in pageable host memory),
 * UNSUPPORTED, MISALIGNED, CUDA.
 */
QMM_API qmm_status qmm_matmul_f32(qmm_type t, const void *w_tiled_dev, int64_t K, int64_t N, const float *x_dev,
                                  int64_t ldx, int64_t M, float *y_dev, int64_t ldy, qmm_stream_t stream);

/* Bytes of device workspace qmm_matmul_f32_ws needs for M rows of length K: 4*M*K rounded up to
 * 256 (0 if invalid). */
QMM_API size_t qmm_matmul_f32_workspace_size(int64_t M, int64_t K);

/*
 * qmm_matmul_f32_ws -- qmm_matmul_f32 with a caller-provided device workspace, for activation rows
 * in page-locked host memory.  The pages' decode path brings each operand into on-chip memory once
 * per op ("DDR -> DMA -> VTCM Execution Pipeline"); here a first kernel copies the rows over
 * NVLink-C2C once into the workspace (dense, row stride K), and the fused decode kernel reads them
 * from there (its CTAs then share the copy through L2).  Same arguments and results, bit for bit,
 * as qmm_matmul_f32, plus:
 *   workspace_dev  >= qmm_matmul_f32_workspace_size(M, K) bytes, 256-byte aligned, owned by the
 *                  caller; overwritten when x is in host memory, untouched otherwise.  Calls that
 *                  overlap on the GPU must use different workspaces.
 * The copy is a programmatic dependent launch: it lets the decode kernel launch at once (the decode
 * kernel takes the SMs as the kernel before the call leaves them and starts streaming the weight
 * tiles), and waits for the kernel before it on the stream before it reads x or writes the
 * workspace; the decode kernel reads the rows and writes y only after the copy has completed.  So
 * the launch-overlap rule of qmm_matmul applies to the kernel launched immediately before this call.
 * x and y are located as for qmm_matmul_f32 (pageable host memory is refused).
 * Errors: those of qmm_matmul_f32, plus INVALID_ARG (workspace missing or too small) and
 * MISALIGNED (workspace not 256-byte aligned).
 */
QMM_API qmm_status qmm_matmul_f32_ws(qmm_type t, const void *w_tiled_dev, int64_t K, int64_t N, const float *x,
                                     int64_t ldx, int64_t M, float *y, int64_t ldy, void *workspace_dev,
                                     size_t workspace_bytes, qmm_stream_t stream);

/*
 * qmm_matmul_flat -- the product of qmm_matmul taken straight from flat GGML rows, without tiles.
 * "Hexagon backend developer details", "Op and Kernel Development Guidelines", section "supports_op
 * Independence from Buffer and Repack State": tensors that are not repacked stay flat, so every
 * supported type must work both tiled and flat.
 *   w_flat_dev  N rows of K/32 blocks (qmm_flat_size bytes, the layout qmm_quantize_weight writes);
 *               16-byte aligned, and a row must be a whole number of 16-byte units:
 *               (K/32) * qmm_block_size(t) % 16 == 0 (true for every type when K % 512 == 0).
 *   a_q_dev, a_d_dev, y_dev  as for qmm_matmul.
 * The same block products and the same error bound as qmm_matmul (the summation order differs, so
 * results agree within that bound, not bit for bit).  A decode kernel: rows of A are processed in
 * groups of 4, each group streaming the whole weight once; for prefill shapes repack and use
 * qmm_matmul.  Launch overlap as for qmm_matmul.
 * Errors: INVALID_ARG (sizes, ldy < N, NULL), UNSUPPORTED (type, or a row length that is not a
 * multiple of 16 bytes), MISALIGNED, CUDA.
 */
QMM_API qmm_status qmm_matmul_flat(qmm_type t, const void *w_flat_dev, int64_t K, int64_t N,
                                   const int8_t *a_q_dev, const uint16_t *a_d_dev, int64_t M, float *y_dev,
                                   int64_t ldy, qmm_stream_t stream);

/* qmm_matmul_path -- qmm_matmul with the kernel chosen by the caller.  QMM_PATH_MATVEC accepts any
 * M (rows are processed in groups of qmm_decode_max_m()); QMM_PATH_GEMM any M >= 1. */
QMM_API qmm_status qmm_matmul_path(qmm_type t, const void *w_tiled_dev, int64_t K, int64_t N,
                           const int8_t *a_q_dev, const uint16_t *a_d_dev, int64_t M, float *y_dev,
                           int64_t ldy, qmm_path path, qmm_stream_t stream);

/* Bytes of device workspace qmm_matmul_ws needs for M activation rows of length K (0 if invalid). */
QMM_API size_t qmm_matmul_workspace_size(int64_t M, int64_t K);

/*
 * qmm_matmul_ws -- the product of qmm_matmul, with caller-provided scratch memory for the tensor-core
 * path ("Hexagon backend developer details", "Tiled Weight Formats"; the pages' prefill path
 * dequantizes tiles to FP16 and contracts them on the matrix unit).
 *   workspace_dev  >= qmm_matmul_workspace_size(M, K) bytes, 256-byte aligned, owned by the caller;
 *                  its contents on entry do not matter and are overwritten.  Calls that overlap on the
 *                  GPU must use different workspaces.
 * For M > qmm_decode_max_m() a first kernel prepares the token operand in the workspace, and the GEMM
 * loads it with TMA straight into its operand layout (each token tile prepared once, not once per
 * weight tile):
 *   - Q4_0, Q8_0, IQ4_NL tiles: the folded-scale GEMM.  Every dequantized value d*q (an fp16 scale
 *     times an integer code of at most 8 bits) is split exactly into two fp16 terms hi + lo, for
 *     the activations in the workspace and for the weights inside the kernel.  The sum is
 *     Y = sum_k (a_hi w_hi + a_hi w_lo + a_lo w_hi) on the tensor cores, in fp32, over 128-wide K
 *     chunks added in fp32.  The dropped a_lo w_lo is below 2^-22 |a w|; rounding stays below about
 *     5e-6 * sum_k |w_k * x_k|, inside the bound of qmm_matmul, with a different summation order.
 *     A token row whose largest |d_a| * 127 (or a weight row whose largest |d_w| * max|w_int|)
 *     reaches 2^15 is scaled by a power of two 2^-t and its outputs by 2^t; that is exact when every
 *     block scale of the row survives the scaling (fp16(d * 2^-t) * 2^t == d), which fails only
 *     for rows holding values of at least 32768 whose block scales also span more than about
 *     2^28 / 127.  Every scaled row is checked; a row that fails the check is reported as
 *     QMM_ERR_RANGE by the next qmm_device_status() (the result of that call is then not exact).
 *     K runs in passes of at most 4096 that add into y in order.
 *   - MXFP4, Q4_1, Q4_K tiles: the exact-integer GEMM of qmm_matmul, with the quants copied to fp16
 *     and the block scales transposed in the workspace (results identical to qmm_matmul's).
 * For smaller M the workspace is not touched and the decode kernel runs.  Launch overlap: the
 * preparation kernel and the GEMM are programmatic dependent launches; the preparation waits for
 * the kernel before it on the stream before it reads a_q / a_d or writes the workspace.
 * Errors: those of qmm_matmul, plus INVALID_ARG (workspace missing or too small) and MISALIGNED
 * (workspace not 256-byte aligned).
 */
QMM_API qmm_status qmm_matmul_ws(qmm_type t, const void *w_tiled_dev, int64_t K, int64_t N,
                                 const int8_t *a_q_dev, const uint16_t *a_d_dev, int64_t M, float *y_dev,
                                 int64_t ldy, void *workspace_dev, size_t workspace_bytes,
                                 qmm_stream_t stream);

/*
 * qmm_matmul_noalloc -- qmm_matmul_ws for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for users of this library.
 *
 * Some callers may not allocate device memory: code running inside a custom allocator or memory
 * pool that must not see foreign allocations, serving runtimes that plan every byte of device memory
 * up front, or sections that must not enter the CUDA allocator at all.  This call takes the same
 * inputs and outputs as qmm_matmul and allocates nothing: for M > qmm_decode_max_m() the
 * tensor-core path's workspace is a fixed scratch array of qmm_matmul_noalloc_max_workspace() bytes
 * (16 MiB) that the library holds on every GPU that loads it, until the process exits.  The kernels
 * and results are those of qmm_matmul_ws.
 *   - Sizes: if qmm_matmul_workspace_size(M, K) exceeds that limit the call returns
 *     QMM_ERR_INVALID_ARG without launching anything (the workspace is about 4.2 bytes per
 *     activation element: M = 960 tokens at K = 4096 fit, 1024 do not).
 *   - Every call with M > qmm_decode_max_m() looks up the scratch array's device address in the
 *     current context (a host-side lookup, no device work), so it follows a device reset that loads
 *     the library's device code again.  The first such call in a context may load that code; make it
 *     before any stream capture.
 *   - The scratch array is shared by all calls and keeps the last call's contents; nothing in it
 *     needs to start at zero (each call rewrites what it reads).  Calls that overlap on the GPU (on
 *     different streams, or from different threads) race on it and must be serialized by the caller.
 *   - For M <= qmm_decode_max_m() no scratch is used (the decode kernel needs none).
 * Errors: those of qmm_matmul, plus INVALID_ARG for sizes beyond the scratch limit.
 */
QMM_API qmm_status qmm_matmul_noalloc(qmm_type t, const void *w_tiled_dev, int64_t K, int64_t N,
                                      const int8_t *a_q_dev, const uint16_t *a_d_dev, int64_t M,
                                      float *y_dev, int64_t ldy, qmm_stream_t stream);

/* Size in bytes of the fixed scratch array qmm_matmul_noalloc uses (per device). */
QMM_API size_t qmm_matmul_noalloc_max_workspace(void);

/*
 * qmm_device_status -- synchronizes `stream`, then returns and clears the library's device status
 * words for the current device: QMM_OK; QMM_ERR_BOUNDS (only in a library built with QMM_DEBUG,
 * whose kernels check every tile index against n_col_tiles * n_k_tiles, every block index against
 * K / 32 and every ring slot against the ring's depth, and skip an access that fails) when such a
 * check failed since the last read; else QMM_ERR_TIMEOUT when a pipelined kernel gave up on one of
 * its bounded waits (its outputs are then undefined); else QMM_ERR_RANGE when a qmm_matmul_ws /
 * qmm_matmul_noalloc call since the last read met an operand row the folded-scale GEMM cannot
 * represent exactly (that call's outputs may be off by more than the stated bound; qmm_matmul,
 * the exact-integer GEMM, computes such data within it).  QMM_ERR_CUDA if the synchronization fails.
 */
QMM_API qmm_status qmm_device_status(qmm_stream_t stream);

/*
 * qmm_selftest_timeout -- test hook for the failure detection above; not part of the hot path.
 * Launches one CTA that uses the pipelined kernels' own bounded-wait helper (unit 0: the decode
 * kernels', unit 1: the exact-integer GEMM's, unit 2: the folded-scale GEMM's, each with its own
 * device status word) on a barrier phase that nothing completes: one warp waits with a
 * limit of limit_ns, a second with the normal 2 s limit and must give up as soon as the first has
 * raised the CTA's abort flag.  flags_dev[0..1] (int32, device) receive 1 for a wait that returned
 * success (neither should), 0 otherwise.  Afterwards qmm_device_status() reports QMM_ERR_TIMEOUT,
 * and the context stays usable: nothing faults, traps or hangs.
 * Errors: INVALID_ARG (unit not 0, 1 or 2, limit_ns outside [1 ms, 2 s], NULL), MISALIGNED, CUDA.
 */
QMM_API qmm_status qmm_selftest_timeout(int unit, uint64_t limit_ns, int *flags_dev, qmm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */

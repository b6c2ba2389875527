// matvec.cu -- decode-shaped matmul (M <= 16 activation rows per pass) over 32-row weight tiles, and
// over flat GGML rows.
//
// What it computes ("Hexagon backend developer details", "Tiled Weight Formats"):
//   Y[m, n] = sum_b fp32(d_w[n,b]) * fp32(d_a[m,b]) * S_b[m,n],  S_b = sum_j w_int[n,32b+j] * a_q[m,32b+j]
// with w_int = q-8 (Q4_0), q (Q8_0), table[q] (IQ4_NL), twice the FP4 value (MXFP4, with half the
// E8M0 scale) read from the tile layouts of "Block-32 Quantized Formats"; the affine tiles (Q4_1, and
// Q4_K through the same tile) add d_a * m_w * sum_j a_q per block.  The pages' decode kernel is an
// HVX 32x1 / 32x2 vector dot product fed by a DDR -> DMA -> VTCM multi-buffered pipeline ("DDR -> DMA
// -> VTCM Execution Pipeline"); this file is the GB300 counterpart of both.
//
// GB300 design:
//   * Persistent CTAs (one wide or two narrow per SM) each own a set of column tiles.  The K tiles of
//     a column tile are contiguous in memory (tile_idx = ct*n_k_tiles + kt), so one producer warp
//     streams them with 1-D cp.async.bulk copies of one stage into a deep ring (mbarrier complete_tx /
//     consumer release) -- the pipelined multi-buffering of the pages, with the TMA engine as the DMA
//     queue.
//   * Up to 4 activation rows (matvec_dp4a_kernel): each lane takes 4 rows x 8 columns of a tile,
//     byte-transposes them into int8x4 words (nibble masks, or a 16-entry table held in registers
//     for IQ4_NL / MXFP4) and takes dp4a against int8 activations staged once per CTA.
//   * 5 to 16 rows (matvec_kernel): quants become fp16 holding exact integers (biased: 1024+q or
//     1152+q, see decode_*), activations are staged once per CTA as fp16 in the mma fragment order,
//     and mma.sync.m16n8k16 (fp32 accumulate) yields block sums that are exact integers; subtracting
//     the exact per-(token, block) bias gives S_b.  fp16 mma.sync runs at ~4x the int8 mma.sync rate
//     on sm_103a, where int8 tcgen05 does not exist.
//   * Per block the result is rescaled by d_w*d_a with packed f32x2 arithmetic and accumulated.
//   * The fused variants (qmm_matmul_f32) quantize the fp32 activation rows into shared memory
//     themselves, by the rule of qmm_quantize_act, while the first weight stages stream in.  With the
//     rows in host memory (read over NVLink-C2C, whose bytes set the cost) the int8 path runs in
//     thread-block clusters: each CTA reads and quantizes only its share of the blocks and writes the
//     records into every CTA of its cluster through distributed shared memory.
//   * Flat GGML rows (matvec_flat_kernel, qmm_matmul_flat): 2-D tensor copies of 32 rows x 32 blocks,
//     one block per lane, dp4a.
//   * Launched as a programmatic dependent: weight streaming overlaps the end of the preceding grid
//     (the activation quantizer), and only the activation staging waits for it.
//   * No atomics and no scratch memory: each column tile is reduced across the warps in a fixed
//     order; if the staged activations would not fit, K is processed in passes that add into y.
#include "pipeline.cuh"
#include "qmm_internal.cuh"

namespace qmm {
namespace {

// Independent tiles per warp and stage of the fp16 mma path (ILP); measured best for 8 and 16 tokens
// alike (one tile per warp at 16 tokens, which avoids a few spilled registers, is 3-7 % slower).
constexpr int kTilesPerWarp = 2;
// Independent tiles per warp and stage for the int8 dot-product consumers: 4 where decoding a tile takes
// many instructions per byte (4-bit codes, table lookups), 2 for the plain Q8_0 bytes (measured).
template <int TYPE>
constexpr int kDp4aTilesPerWarp = TYPE == QMM_Q8_0 ? 2 : 4;
constexpr int kDp4aMaxM = 4;                            // tokens up to which the int8 dot-product path runs
// Parts per ring stage of the int8 path: each its own bulk copy and barrier, consumed by CW / parts
// warps that take contiguous tiles, so a stage's first parts are worked on while the rest lands.  Four
// for the 4-bit types, whose decode makes the work per byte large (Q4_0 K=N=4096: 3.64 -> 3.37 us);
// one for Q8_0, which streams at the bandwidth limit and only pays for the extra copies (measured).
template <int TYPE>
constexpr int kDp4aSub = TYPE == QMM_Q8_0 ? 1 : 4;
constexpr int kLutCopies = 32;                          // byte-indexed table copies (one per lane: no bank conflicts)
constexpr int kActBudget = 64 * 1024;                   // bytes of staged activations per CTA
// Deepest ring of the tiled decode kernels.  Their barriers come first in shared memory, laid out for
// this many stages, so that their place does not depend on the launch parameters: thread 0
// initialises them while the parameters are still being fetched at kernel start.
constexpr int kMaxRingStages = 12;
constexpr int kSmemLimit = 227 * 1024;
using namespace pipe;

struct MvParams {
    const uint8_t *tiled;
    const int8_t *a_q;
    const uint16_t *a_d;
    float *y;
    int64_t K, nkt, N, ldy, n_col_tiles;
    int M;            // tokens in this launch (<= 8 * NF)
    int kt0, nkc;     // K-tile range of this pass: [kt0, kt0 + nkc)
    int accumulate;   // 0: y = result, 1: y += result
    int stages;       // ring depth
    Lut16 lut;
    const float *x;   // fused activation quantization: fp32 rows (a_q / a_d unused), else nullptr
    int64_t ldx;
    int x_vec;        // x 16-byte aligned and ldx % 4 == 0: float4 loads
};

__device__ unsigned g_mv_status = 0;   // set when a bounded wait gave up (reported with the GEMM's word)

// Bounded wait (pipeline.cuh) reporting to this file's status word.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort,
                                             unsigned long long limit_ns = kWaitLimitNs) {
    return wait_bounded_on(bar, parity, abort, &g_mv_status, limit_ns);
}

// Runs the bounded wait out on purpose (the failure-detection test): warp 0 waits, with limit_ns,
// for a barrier phase that nothing completes; warp 1 waits for the same phase with the normal limit
// and must give up once warp 0 has raised the abort flag.  out[w] = 1 if warp w's wait returned
// true (neither should); the device status word is set as by any timed-out pipeline wait.
__global__ void __launch_bounds__(64) selftest_wait_kernel(unsigned long long limit_ns, int *out) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    volatile int *abort = &abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const bool ok = wait_bounded(smem_u32(&bar), 0u, abort, warp == 0 ? limit_ns : kWaitLimitNs);
    if ((threadIdx.x & 31) == 0) out[warp] = ok ? 1 : 0;
}
// Producer warp: streams the K tiles [kt0, kt0 + nkc) of every column tile this CTA owns into the
// ring, one stage of TPS consecutive tiles at a time in NSUB 1-D bulk copies of TPS / NSUB tiles, each
// completing its own barrier full[stage * NSUB + q] (so the consumers of the first part of a stage can
// start before the rest has landed), and returns once the copies in flight have landed.
template <int TS, int TPS, int NSUB = 1>
__device__ __forceinline__ void produce(const MvParams &p, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                        volatile int *abort, int lane) {
    static_assert(TPS % NSUB == 0, "sub-copies split a stage evenly");
    constexpr int kSubTiles = TPS / NSUB;
    const int stages = p.stages, nkc = p.nkc;
    uint32_t it = 0;
    bool ok = true;
    for (int64_t ct = blockIdx.x; ct < p.n_col_tiles && ok; ct += gridDim.x) {
        const uint8_t *src = p.tiled + (ct * p.nkt + p.kt0) * TS;
        for (int j0 = 0; j0 < nkc; j0 += TPS, ++it) {
            const int s = (int)(it % (uint32_t)stages);
            const uint32_t ph = (it / (uint32_t)stages) & 1u;
            if (!wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort)) { ok = false; break; }
            if (lane == 0) {
                const int nt = (nkc - j0) < TPS ? (nkc - j0) : TPS;
#pragma unroll
                for (int q = 0; q < NSUB; ++q) {
                    // tiles [ct * nkt + kt0 + j0 + t0, .. + t1) of this column tile, into ring slot s
                    const int t0 = q * kSubTiles, t1 = (t0 + kSubTiles) < nt ? (t0 + kSubTiles) : nt;
                    const uint32_t fb = smem_u32(&full[s * NSUB + q]);
                    if (t1 > t0 && QMM_DCHECK(s < stages && ct < p.n_col_tiles && p.kt0 + j0 + t1 <= p.nkt)) {
                        const uint32_t bytes = (uint32_t)((t1 - t0) * TS);
                        mbar_arrive_expect_tx(fb, bytes);
                        bulk_g2s(smem_u32(ring + (s * TPS + t0) * TS), src + (int64_t)(j0 + t0) * TS, bytes, fb);
                    } else {
                        mbar_arrive(fb);           // nothing of this part in a short last stage
                    }
                }
            }
            __syncwarp();
        }
    }
    // copies in flight land before the CTA may exit
    if (lane == 0 && it > 0) {
        const uint32_t last = it - 1;
        for (uint32_t k = 0; k < (uint32_t)stages && k <= last; ++k) {
            const uint32_t i = last - k;
            for (int q = 0; q < NSUB; ++q) wait_drain(smem_u32(&full[(i % stages) * NSUB + q]), (i / stages) & 1u);
        }
    }
}

template <int CW>
__device__ __forceinline__ void consumer_sync() {      // named barrier over the consumer warps
    asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");
}

// Fused activation quantization.  The 4 lanes q = 0..3 of an aligned lane quad quantize one block
// of 32 (columns 8q..8q+7 each) by the rule of qmm_quantize_act, sharing amax through two
// shuffles; every lane of the warp must call quantize_loaded (dead lanes load with live = false).
// load_quarter fetches the lane's 8 fp32 values (so that a thread can have several blocks in
// flight before it quantizes any); quantize_loaded returns the 8 int8 codes (columns 8q..8q+7, in
// order) and sets da = fp32(fp16(d)).
__device__ __forceinline__ void load_quarter(const MvParams &p, bool live, int tok, int64_t kt, int q, float (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = 0.0f;
    if (live && QMM_DCHECK(kt < p.nkt && tok < p.M)) {
        const float *src = p.x + (int64_t)tok * p.ldx + kt * 32 + 8 * q;
        if (p.x_vec) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(src)), b = __ldg(reinterpret_cast<const float4 *>(src + 4));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __ldg(src + k);
        }
    }
}
// The int8 codes of a quarter loaded by load_quarter (the 4 lanes of a quad hold one block's quarters
// and take the block's amax together) and fp32(d_a).
__device__ __forceinline__ uint2 quantize_loaded(const float (&v)[8], float &da) {
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = q8_scale(amax), id = inv_or_zero(d);
    uint32_t lo = 0u, hi = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        lo |= (uint32_t)(q8_code(v[k], id) & 0xFF) << (8 * k);
        hi |= (uint32_t)(q8_code(v[k + 4], id) & 0xFF) << (8 * k);
    }
    da = __half2float(__float2half_rn(d));
    return make_uint2(lo, hi);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// The scales of tile rows r0 .. r0+3 (r0 a multiple of 4) as fp32: fp16 row scales (Q4_1: the d of each
// (d, m) pair), or for MXFP4 half the power of two of each row's E8M0 byte (the doubled integer codes
// carry the other factor 2).  row_mins: the m of Q4_1's pairs.
template <int TYPE>
__device__ __forceinline__ void row_mins(const uint8_t *scales, int r0, float (&m)[4]) {
    const uint4 dm = *reinterpret_cast<const uint4 *>(scales + 4 * r0);
    m[0] = __high2float(bits_h2(dm.x)); m[1] = __high2float(bits_h2(dm.y));
    m[2] = __high2float(bits_h2(dm.z)); m[3] = __high2float(bits_h2(dm.w));
}
template <int TYPE>
__device__ __forceinline__ void row_scales(const uint8_t *scales, int r0, float (&d)[4]) {
    if constexpr (TileFmt<TYPE>::kAffine) {
        const uint4 dm = *reinterpret_cast<const uint4 *>(scales + 4 * r0);    // (d, m) of 4 rows
        d[0] = __low2float(bits_h2(dm.x)); d[1] = __low2float(bits_h2(dm.y));
        d[2] = __low2float(bits_h2(dm.z)); d[3] = __low2float(bits_h2(dm.w));
    } else if constexpr (TileFmt<TYPE>::kE8M0) {
        const uint32_t e4 = *reinterpret_cast<const uint32_t *>(scales + r0);
#pragma unroll
        for (int r = 0; r < 4; ++r) d[r] = mx_half_scale((e4 >> (8 * r)) & 0xFFu);
    } else {
        const uint2 sc = *reinterpret_cast<const uint2 *>(scales + 2 * r0);
        const float2 d01 = __half22float2(bits_h2(sc.x)), d23 = __half22float2(bits_h2(sc.y));
        d[0] = d01.x; d[1] = d01.y; d[2] = d23.x; d[3] = d23.y;
    }
}

__device__ __forceinline__ float2 pack2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ void unpack2(float2 v, float &a, float &b) {
    a = v.x;
    b = v.y;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- weight decode: 16 half2 H[q][r] = (column 2cp, 2cp+1) of tile row 4g+r, cp = t + 4q ----
// Q4_0: byte -> half2(1024 + lo, 1024 + 16*hi).  With the odd-column activations staged divided by
// 16 (exact), the mma sums (1024+lo)*a_even + (64+hi)*a_odd; the bias 1032*sum(a_even) +
// 72*sum(a_odd) (which also removes the -8 offset) is subtracted per token and block.
template <int I>
__device__ __forceinline__ uint32_t q4_biased(uint32_t w) {
    const uint32_t y = __byte_perm(w, 0u, 0x4040u | (I << 8) | I);
    uint32_t h;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(h) : "r"(y), "r"(0x00F0000Fu), "r"(0x64006400u));
    return h;
}
// Q8_0: two int8 -> half2(1152 + b0, 1152 + b1) (b ^ 0x80 = b + 128 placed in the mantissa of 1024);
// bias 1152*sum(a) per token and block.
template <int SEL>
__device__ __forceinline__ uint32_t q8_biased(uint32_t w_xor) { return __byte_perm(w_xor, 0x64646464u, SEL); }

template <int TYPE>
__device__ __forceinline__ void decode_tile(const uint8_t *tile, int g, int t, uint32_t (&H)[4][4],
                                            const uint32_t *lut_lane) {
    if constexpr (TYPE == QMM_Q8_0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint2 v = *reinterpret_cast<const uint2 *>(tile + (t + 4 * q) * 64 + 8 * g);
            const uint32_t x = v.x ^ 0x80808080u, z = v.y ^ 0x80808080u;
            H[q][0] = q8_biased<0x4140>(x);
            H[q][1] = q8_biased<0x4342>(x);
            H[q][2] = q8_biased<0x4140>(z);
            H[q][3] = q8_biased<0x4342>(z);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(tile + (t + 4 * q) * 32 + 4 * g);
            if constexpr (TileFmt<TYPE>::kNibbleInt) {
                H[q][0] = q4_biased<0>(w);
                H[q][1] = q4_biased<1>(w);
                H[q][2] = q4_biased<2>(w);
                H[q][3] = q4_biased<3>(w);
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) H[q][r] = lut_lane[__byte_perm(w, 0u, 0x4440u | (uint32_t)r) * kLutCopies];
            }
        }
    }
}

// Staged fp16 activation pairs (column 2cp, 2cp+1) for the biased decode, the odd column divided by 16
// (exact) for the nibble types, whose high nibble is decoded as 16*hi; for a whole int8x4 word w
// (columns c..c+3): lo = (c, c+1), hi = (c+2, c+3).  Byte b ^ 0x80
// under the exponent byte 0x64 is the fp16 number 1152 + b (exact), and one fp16 subtract (or, for the
// nibble types, an fma by (1, 1/16) minus (1152, 72)) leaves b (or b/16) exactly.
template <int TYPE>
__device__ __forceinline__ void act_pairs4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x80808080u;
    const __half2 b01 = bits_h2(__byte_perm(x, 0x64646464u, 0x5140u));
    const __half2 b23 = bits_h2(__byte_perm(x, 0x64646464u, 0x7362u));
    if constexpr (TileFmt<TYPE>::kNibbleInt) {
        const __half2 sc = __halves2half2(__float2half_rn(1.0f), __float2half_rn(0.0625f));
        const __half2 off = __halves2half2(__float2half_rn(-1152.0f), __float2half_rn(-72.0f));
        lo = h2_bits(__hfma2(b01, sc, off));
        hi = h2_bits(__hfma2(b23, sc, off));
    } else {
        const __half2 off = __float2half2_rn(1152.0f);
        lo = h2_bits(__hsub2(b01, off));
        hi = h2_bits(__hsub2(b23, off));
    }
}
// The exact bias of the biased weight decode for one (token, block).
template <int TYPE>
__device__ __forceinline__ float act_bias(int sum_even, int sum_odd) {
    if (TYPE == QMM_Q4_0) return 1032.0f * (float)sum_even + 72.0f * (float)sum_odd;
    if (TYPE == QMM_Q4_1) return 1024.0f * (float)sum_even + 64.0f * (float)sum_odd;   // no -8 offset
    if (TYPE == QMM_Q8_0) return 1152.0f * (float)(sum_even + sum_odd);
    return 0.0f;
}

// Token stride of the staged activations in uint4 units: an odd multiple of 4, so the 8 lanes of a
// quarter-warp (2 tokens x 4 column groups) read 8 distinct 16-byte bank groups.
__host__ __device__ inline int act_tok_stride(int nkc) { return nkc * 4 + ((nkc & 1) ? 0 : 4); }

// Shared-memory layout (offsets in bytes from a 128-byte aligned base).
struct MvLayout {
    int ring, bars, act, da, corr, asum, red, lut, total;
};
template <int TYPE, int NF, int CW>
__host__ __device__ inline MvLayout mv_layout(int M, int nkc, int stages) {
    constexpr int TS = TileFmt<TYPE>::kBytes;
    constexpr int kTilesPerStage = CW * kTilesPerWarp;
    MvLayout L;
    int off = 0;
    L.bars = off;  off += 2 * kMaxRingStages * 8 + 16;       // full, empty, abort flag: a fixed place
    off = (off + 127) & ~127;
    L.ring = off;  off += stages * kTilesPerStage * TS;
    off = (off + 15) & ~15;
    L.act = off;   off += M * act_tok_stride(nkc) * 16;     // [M][stride] uint4 (16 half2 per block)
    L.da = off;    off += nkc * 8 * NF * 4;                 // [nkc][8*NF] float
    L.corr = off;  off += nkc * 8 * NF * 4;                 // [nkc][8*NF] float
    L.asum = off;  off += TileFmt<TYPE>::kAffine ? nkc * 8 * NF * 4 : 0;   // Q4_1: [nkc][8*NF] sum of a_q
    L.red = off;   off += CW * 2 * NF * 4 * 32 * 4;
    L.lut = off;   off += TileFmt<TYPE>::kLut ? 256 * kLutCopies * 4 : 0;
    L.total = off;
    return L;
}

// The TPW tiles cw, cw + CW, ... of one ring stage for lane (g, t): all of them decoded first, then
// contracted with the staged tokens (act_s[act_off[nf] + 4 j]: block j of this lane's activation row
// of token group nf) and rescaled into acc.  jt0 = the K tile of the warp's first tile;
// FULL: every tile of the stage is live, else tiles at or past nkc are skipped.
template <int TYPE, int NF, int CW, int TPW, bool FULL>
__device__ __forceinline__ void mma_stage(const uint8_t *tile, int jt0, int nkc, const uint4 *act_s, const int (&act_off)[NF],
                                          const float *da_s, const float *corr_s, const float *asum_s,
                                          const uint32_t *lut_lane, int g, int t, float2 (&acc)[2][NF][2]) {
    constexpr int TS = TileFmt<TYPE>::kBytes;
    constexpr int SOFF = TileFmt<TYPE>::kScaleOff;
    constexpr int TOK = 8 * NF;
    uint32_t H[TPW][4][4];
    float dwr[TPW][4];
    float mwr[TPW][4];              // Q4_1 row mins
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        if (FULL || jt0 + CW * u < nkc) {
            decode_tile<TYPE>(tile + CW * u * TS, g, t, H[u], lut_lane);
            row_scales<TYPE>(tile + CW * u * TS + SOFF, 4 * g, dwr[u]);            // rows 4g .. 4g+3
            if constexpr (TileFmt<TYPE>::kAffine) row_mins<TYPE>(tile + CW * u * TS + SOFF, 4 * g, mwr[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        const int j = jt0 + CW * u;
        if (!FULL && j >= nkc) continue;
#pragma unroll
        for (int nf = 0; nf < NF; ++nf) {
            const uint4 b = act_s[act_off[nf] + 4 * j];
            const float2 da = *reinterpret_cast<const float2 *>(da_s + j * TOK + 8 * nf + 2 * t);
            const float2 cr = *reinterpret_cast<const float2 *>(corr_s + j * TOK + 8 * nf + 2 * t);
            const float2 ncorr = pack2(-cr.x, -cr.y);
            float2 as2 = make_float2(0.0f, 0.0f);
            if constexpr (TileFmt<TYPE>::kAffine) as2 = *reinterpret_cast<const float2 *>(asum_s + j * TOK + 8 * nf + 2 * t);
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(c, H[u][0][2 * rb], H[u][0][2 * rb + 1], H[u][1][2 * rb], H[u][1][2 * rb + 1], b.x, b.y);
                mma16816(c, H[u][2][2 * rb], H[u][2][2 * rb + 1], H[u][3][2 * rb], H[u][3][2 * rb + 1], b.z, b.w);
                // c0,c1: row 4g+2rb, tokens 2t,2t+1;  c2,c3: row 4g+2rb+1
                const float2 s01 = fadd2(pack2(c[0], c[1]), ncorr);
                const float2 s23 = fadd2(pack2(c[2], c[3]), ncorr);
                const float2 p01 = fmul2(pack2(dwr[u][2 * rb], dwr[u][2 * rb]), da);
                const float2 p23 = fmul2(pack2(dwr[u][2 * rb + 1], dwr[u][2 * rb + 1]), da);
                acc[rb][nf][0] = ffma2(s01, p01, acc[rb][nf][0]);
                acc[rb][nf][1] = ffma2(s23, p23, acc[rb][nf][1]);
                if constexpr (TileFmt<TYPE>::kAffine) {
                    // + m_w * d_a * sum(a_q) of the block, per row and token
                    const float2 m01 = fmul2(pack2(mwr[u][2 * rb], mwr[u][2 * rb]), da);
                    const float2 m23 = fmul2(pack2(mwr[u][2 * rb + 1], mwr[u][2 * rb + 1]), da);
                    acc[rb][nf][0] = ffma2(as2, m01, acc[rb][nf][0]);
                    acc[rb][nf][1] = ffma2(as2, m23, acc[rb][nf][1]);
                }
            }
        }
    }
}

// CW consumer warps per CTA: 8 (two CTAs per SM) for grids with many column tiles, 16 (one wide CTA
// per SM) for small ones.
template <int TYPE, int NF, int CW, bool FUSED>
__global__ void __launch_bounds__(32 * (1 + CW), 16 / CW) matvec_kernel(const MvParams p) {
    constexpr int kConsumerWarps = CW;
    constexpr int kTilesPerStage = CW * kTilesPerWarp;
    constexpr int TS = TileFmt<TYPE>::kBytes;
    constexpr int TOK = 8 * NF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const MvLayout L = mv_layout<TYPE, NF, CW>(p.M, p.nkc, p.stages);
    uint8_t *ring = smem + L.ring;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kMaxRingStages;
    volatile int *abort = reinterpret_cast<volatile int *>(empty + kMaxRingStages);
    uint4 *act_s = reinterpret_cast<uint4 *>(smem + L.act);      // [M][act_tok_stride] uint4
    const int tok_stride = act_tok_stride(p.nkc);
    float *da_s = reinterpret_cast<float *>(smem + L.da);         // [nkc][TOK]
    float *corr_s = reinterpret_cast<float *>(smem + L.corr);     // [nkc][TOK]
    float *asum_s = reinterpret_cast<float *>(smem + L.asum);     // [nkc][TOK] (Q4_1 only)
    float *red_s = reinterpret_cast<float *>(smem + L.red);
    uint32_t *lut_s = reinterpret_cast<uint32_t *>(smem + L.lut);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stages = p.stages;
    const int nkc = p.nkc;

    if (threadIdx.x == 0) {
        // every stage the ring could have: no dependence on the launch parameters
#pragma unroll
        for (int s = 0; s < kMaxRingStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // A grid launched after this one as a programmatic dependent may start now: it waits for this
    // grid to complete before it reads anything this grid writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        produce<TS, kTilesPerStage>(p, ring, full, empty, abort, lane);
        return;
    }

    // ============================== consumers ==============================
    const int cw = warp - 1;                  // consumer warp 0..7
    const int ctid = threadIdx.x - 32;        // 0..255
    const int g = lane >> 2, t = lane & 3;

    // Once the thread's first activation loads are in flight, it builds its share of the byte -> half2
    // table (which depends on the parameters only) while they land.  Runs once per thread.
    bool requested = false;
    auto on_loads_issued = [&]() {
        if (requested) return;
        requested = true;
        if constexpr (TileFmt<TYPE>::kLut) {
            for (int i = ctid; i < 256 * kLutCopies; i += kConsumerWarps * 32) {
                const int b = i / kLutCopies;
                lut_s[i] = h2_bits(__halves2half2(__int2half_rn(p.lut.v[b & 15]), __int2half_rn(p.lut.v[b >> 4])));
            }
        }
    };

    // The weights never depend on the kernel launched just before on the stream, so the producer
    // starts streaming at once; the activations may, so the consumers wait for that grid first
    // (a no-op unless this grid was launched as its programmatic dependent).
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- stage activations once: per (token, block) 16 half2 in fragment order, plus the
    //      per-block scale and the exact bias of the biased weight decode ----
    if constexpr (!FUSED) {
        // two (token, block) entries per thread and pass, both loaded before either is converted (the
        // loop runs warp-uniformly: every lane of a warp takes part in every pass)
        constexpr int kStep = kConsumerWarps * 32;
        for (int w0 = cw * 32; w0 < TOK * nkc; w0 += 2 * kStep) {
            const int i0 = w0 + lane;
            uint4 ld[2][2];
            uint16_t dbits[2] = {0, 0};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * kStep, j = i / TOK, tok = i - j * TOK;
                ld[u][0] = ld[u][1] = make_uint4(0u, 0u, 0u, 0u);
                if (i < TOK * nkc && tok < p.M && QMM_DCHECK(p.kt0 + j < p.nkt)) {
                    const int64_t kt = p.kt0 + j;
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.a_q + (int64_t)tok * p.K + kt * 32);
                    ld[u][0] = __ldg(src);
                    ld[u][1] = __ldg(src + 1);
                    dbits[u] = p.a_d[(int64_t)tok * p.nkt + kt];
                }
            }
            on_loads_issued();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * kStep;
                if (i >= TOK * nkc) break;
                const int j = i / TOK, tok = i - j * TOK;
                float d = 0.0f, corr = 0.0f, asum = 0.0f;
                if (tok < p.M) {
                    const uint4 v0 = ld[u][0], v1 = ld[u][1];
                    const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                    int sum_even = 0, sum_odd = 0;
                    uint32_t hp[16];                 // half2 of column pair cp, in cp order
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) {
                        act_pairs4<TYPE>(wv[wi], hp[2 * wi], hp[2 * wi + 1]);
                        sum_even = __dp4a((int)wv[wi], 0x00010001, sum_even);     // columns 4wi, 4wi + 2
                        sum_odd = __dp4a((int)wv[wi], 0x01000100, sum_odd);       // columns 4wi + 1, 4wi + 3
                    }
                    // fragment order: position 4t + q holds column pair t + 4q
                    uint4 *dst = act_s + tok * tok_stride + j * 4;
#pragma unroll
                    for (int tt = 0; tt < 4; ++tt) dst[tt] = make_uint4(hp[tt], hp[tt + 4], hp[tt + 8], hp[tt + 12]);
                    d = __half2float(__ushort_as_half(dbits[u]));
                    corr = act_bias<TYPE>(sum_even, sum_odd);
                    asum = (float)(sum_even + sum_odd);
                }
                da_s[j * TOK + tok] = d;
                corr_s[j * TOK + tok] = corr;
                if constexpr (TileFmt<TYPE>::kAffine) asum_s[j * TOK + tok] = asum;
            }
        }
    } else {
        // 4 lanes per (block, token), 8 columns each; lane q holds column pairs 4q..4q+3, which go to
        // word q of fragment positions 0..3
        const int total = TOK * nkc * 4;
        for (int base = cw * 32; base < total; base += kConsumerWarps * 32) {
            const int e = base + lane, q = e & 3, jt = (e >> 2) / TOK, tok = (e >> 2) - jt * TOK;
            const bool live = e < total && tok < p.M;
            float v[8], d;
            load_quarter(p, live, tok, p.kt0 + jt, q, v);
            on_loads_issued();
            const uint2 c = quantize_loaded(v, d);
            uint32_t hp[4];
            act_pairs4<TYPE>(c.x, hp[0], hp[1]);
            act_pairs4<TYPE>(c.y, hp[2], hp[3]);
            int sum_even = __dp4a((int)c.y, 0x00010001, __dp4a((int)c.x, 0x00010001, 0));
            int sum_odd = __dp4a((int)c.y, 0x01000100, __dp4a((int)c.x, 0x01000100, 0));
            sum_even += __shfl_xor_sync(0xffffffffu, sum_even, 1);
            sum_odd += __shfl_xor_sync(0xffffffffu, sum_odd, 1);
            sum_even += __shfl_xor_sync(0xffffffffu, sum_even, 2);
            sum_odd += __shfl_xor_sync(0xffffffffu, sum_odd, 2);
            if (live) {
                uint32_t *dst = reinterpret_cast<uint32_t *>(act_s + tok * tok_stride + jt * 4);
#pragma unroll
                for (int u = 0; u < 4; ++u) dst[4 * u + q] = hp[u];
            }
            if (e < total && q == 0) {
                da_s[jt * TOK + tok] = live ? d : 0.0f;
                corr_s[jt * TOK + tok] = live ? act_bias<TYPE>(sum_even, sum_odd) : 0.0f;
                if constexpr (TileFmt<TYPE>::kAffine) asum_s[jt * TOK + tok] = live ? (float)(sum_even + sum_odd) : 0.0f;
            }
        }
    }
    on_loads_issued();             // threads that had no activation entries
    consumer_sync<CW>();

    // After a timed-out wait a warp stops waiting and computing but keeps the loop structure, so
    // every consumer warp still reaches the same named barriers.
    const uint32_t *lut_lane = lut_s + (lane & (kLutCopies - 1));
    // this lane's activation row per token group: token 8 nf + g, or for a token past the live ones
    // (its output column is dropped) the last live token's row, so that every read stays in the
    // staged rows
    int act_off[NF];
#pragma unroll
    for (int nf = 0; nf < NF; ++nf) act_off[nf] = min(8 * nf + g, p.M - 1) * tok_stride + t;
    uint32_t it = 0;
    bool ok = true;
    for (int64_t ct = blockIdx.x; ct < p.n_col_tiles; ct += gridDim.x) {
        float2 acc[2][NF][2];     // [rb][nf][row pair half]: (tok 2t, 2t+1) of rows 4g+2rb(+1)
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int nf = 0; nf < NF; ++nf) acc[rb][nf][0] = acc[rb][nf][1] = make_float2(0.0f, 0.0f);

        for (int j0 = 0; j0 < nkc; j0 += kTilesPerStage, ++it) {
            const int s = (int)(it % (uint32_t)stages);
            const uint32_t ph = (it / (uint32_t)stages) & 1u;
            if (ok) ok = __all_sync(0xffffffffu, wait_bounded(smem_u32(&full[s]), ph, abort));
            if (ok && QMM_DCHECK(s < stages)) {
                // tiles cw, cw + CW, ... of this stage; only the last stage of a pass can be partial
                const uint8_t *tile = ring + (s * kTilesPerStage + cw) * TS;
                if (j0 + kTilesPerStage <= nkc)
                    mma_stage<TYPE, NF, CW, kTilesPerWarp, true>(tile, j0 + cw, nkc, act_s, act_off, da_s, corr_s, asum_s, lut_lane, g, t, acc);
                else
                    mma_stage<TYPE, NF, CW, kTilesPerWarp, false>(tile, j0 + cw, nkc, act_s, act_off, da_s, corr_s, asum_s, lut_lane, g, t, acc);
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }

        // ---- reduce the 8 warps in a fixed order, write (or add into) y ----
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int nf = 0; nf < NF; ++nf)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float a, b;
                    unpack2(acc[rb][nf][h], a, b);
                    red_s[((((cw * 2 + rb) * NF + nf) * 2 + h) * 2 + 0) * 32 + lane] = a;
                    red_s[((((cw * 2 + rb) * NF + nf) * 2 + h) * 2 + 1) * 32 + lane] = b;
                }
        consumer_sync<CW>();
        if (cw == 0) {
#pragma unroll
            for (int rb = 0; rb < 2; ++rb)
#pragma unroll
                for (int nf = 0; nf < NF; ++nf)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float sum = 0.0f;
#pragma unroll
                            for (int w = 0; w < kConsumerWarps; ++w)
                                sum += red_s[((((w * 2 + rb) * NF + nf) * 2 + h) * 2 + e) * 32 + lane];
                            const int row = 4 * g + 2 * rb + h;
                            const int tok = 8 * nf + 2 * t + e;
                            const int64_t n = ct * 32 + row;
                            if (ok && tok < p.M && n < p.N) {
                                float *dst = p.y + (int64_t)tok * p.ldy + n;
                                *dst = p.accumulate ? (*dst + sum) : sum;
                            }
                        }
        }
        consumer_sync<CW>();
    }
}

// ================= small-M path: int8 dot products straight from the tile bytes =================
// For a handful of tokens the fp16 decode above costs more issue slots than the weight bytes take
// to arrive.  Here the quants stay 8-bit: lane (i, j) = (lane & 7, lane >> 3) of a warp owns tile
// rows 4i..4i+3 and column pairs cp = 4j..4j+3 of one tile, gathers each row's bytes into int8x4
// words with a 4x4 byte transpose (Q4_0 / IQ4_NL: byte cp*32 + row; Q8_0: bytes cp*64 + 2*row,
// +1) and takes dp4a against the int8 activations.  The column pairs are visited in the rotated
// order cp_c = 4j + ((c + j) & 3), which puts the 32 lanes' shared-memory words in distinct banks;
// the activations are staged once per CTA in that same order, so the rotation costs nothing later.
//   Q4_0:   low and high nibbles are two int8x4 words (0..15) of the even and odd columns; the -8
//           offset enters as the dp4a chain's start value -8 * (sum of the lane's 8 activations).
//   IQ4_NL: each nibble indexes the 16-entry table held in 4 registers with two byte permutes and
//           a third that picks the half by the index's top bit.
//   Q8_0:   the int8 quants are the operands as they are.
// Each lane keeps, per token, fp32 sums for its 4 rows: y += float(S) * (d_w * d_a), where S, the
// product of the two fp16 scales and float(S) are exact; the four column quarters and then the
// warps are added in a fixed order at the end of a column tile.

// Row words of one tile for lane (i, j): R[r][0], R[r][1] are the int8x4 weights of row 4i + r in
// the staged activation order (see dp4a_record).
template <int TYPE>
__device__ __forceinline__ void tile_rows_dp4a(const uint8_t *tile, int i, int j, uint32_t (&R)[4][2],
                                               const uint32_t (&tb)[4]) {
    if constexpr (TYPE == QMM_Q8_0) {
        uint2 w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint2 *>(tile + (4 * j + ((c + j) & 3)) * 64 + 8 * i);
        // w[c].x = (row 4i: col 2cp, 2cp+1; row 4i+1: col 2cp, 2cp+1), w[c].y likewise rows 4i+2, 4i+3
        R[0][0] = __byte_perm(w[0].x, w[1].x, 0x5410); R[0][1] = __byte_perm(w[2].x, w[3].x, 0x5410);
        R[1][0] = __byte_perm(w[0].x, w[1].x, 0x7632); R[1][1] = __byte_perm(w[2].x, w[3].x, 0x7632);
        R[2][0] = __byte_perm(w[0].y, w[1].y, 0x5410); R[2][1] = __byte_perm(w[2].y, w[3].y, 0x5410);
        R[3][0] = __byte_perm(w[0].y, w[1].y, 0x7632); R[3][1] = __byte_perm(w[2].y, w[3].y, 0x7632);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint32_t *>(tile + (4 * j + ((c + j) & 3)) * 32 + 4 * i);
        // 4x4 byte transpose: T[r] = byte r (tile row 4i + r) of w[0..3]
        const uint32_t x01 = __byte_perm(w[0], w[1], 0x5140), x23 = __byte_perm(w[2], w[3], 0x5140);
        const uint32_t y01 = __byte_perm(w[0], w[1], 0x7362), y23 = __byte_perm(w[2], w[3], 0x7362);
        uint32_t T[4];
        T[0] = __byte_perm(x01, x23, 0x5410);
        T[1] = __byte_perm(x01, x23, 0x7632);
        T[2] = __byte_perm(y01, y23, 0x5410);
        T[3] = __byte_perm(y01, y23, 0x7632);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if constexpr (TileFmt<TYPE>::kNibbleInt) {
                R[r][0] = T[r] & 0x0F0F0F0Fu;             // even columns 2cp_c
                R[r][1] = (T[r] >> 4) & 0x0F0F0F0Fu;      // odd columns 2cp_c + 1
            } else {
                // nibbles in column order: lo(b0), hi(b0), lo(b1), hi(b1) | lo(b2), hi(b2), lo(b3), hi(b3)
                const uint32_t m = T[r] & 0x77777777u;                         // index & 7 per nibble
                const uint32_t sel0 = ((T[r] >> 1) & 0x4444u) | 0x3210u;       // + 4 where index & 8
                const uint32_t sel1 = ((T[r] >> 17) & 0x4444u) | 0x3210u;
                const uint32_t m1 = m >> 16;
                R[r][0] = __byte_perm(__byte_perm(tb[0], tb[1], m), __byte_perm(tb[2], tb[3], m), sel0);
                R[r][1] = __byte_perm(__byte_perm(tb[0], tb[1], m1), __byte_perm(tb[2], tb[3], m1), sel1);
            }
        }
    }
}

// Staged activation record of (token, block, quarter j): the 8 int8 v of columns 8j..8j+7 as two
// int8x4 words in the order of tile_rows_dp4a, the dp4a start value (Q4_1: the sum of the 8 values,
// for the min term), and fp32(d_a).
__device__ __forceinline__ uint4 dp4a_record(int type, uint2 v, int j, float da) {
    unsigned long long V = (unsigned long long)v.x | ((unsigned long long)v.y << 32);
    if (j) V = (V >> (16 * j)) | (V << (64 - 16 * j));       // column pair c <- local pair (c + j) & 3
    const uint32_t lo = (uint32_t)V, hi = (uint32_t)(V >> 32);
    uint4 rec;
    int corr = 0;
    if (type == QMM_Q4_0 || type == QMM_Q4_1) {
        rec.x = __byte_perm(lo, hi, 0x6420);      // even columns
        rec.y = __byte_perm(lo, hi, 0x7531);      // odd columns
        const int asum = __dp4a((int)v.x, 0x01010101, __dp4a((int)v.y, 0x01010101, 0));
        corr = (type == QMM_Q4_0) ? -8 * asum : asum;   // Q4_0: chain start; Q4_1: sum for the min term
    } else {
        rec.x = lo;
        rec.y = hi;
    }
    rec.z = (uint32_t)corr;
    rec.w = __float_as_uint(da);
    return rec;
}

// One tile for lane (i, j): the int8 dot products of its rows 4i..4i+3 with the MT staged tokens
// (act[4 t + j]: token t's record of the tile's block for this lane's column pairs), rescaled by
// d_w * d_a and added to acc.  Tokens past the live ones have all-zero records and add nothing.
template <int TYPE, int MT>
__device__ __forceinline__ void dp4a_tile(const uint8_t *tile, const uint4 *act, int i, int j, const uint32_t (&tb)[4],
                                          float2 (&acc)[MT][2]) {
    constexpr int SOFF = TileFmt<TYPE>::kScaleOff;
    uint32_t R[4][2];
    tile_rows_dp4a<TYPE>(tile, i, j, R, tb);
    float dws[4];
    row_scales<TYPE>(tile + SOFF, 4 * i, dws);                  // rows 4i .. 4i+3
    const float2 dw01 = pack2(dws[0], dws[1]), dw23 = pack2(dws[2], dws[3]);
    float2 mw01 = make_float2(0.0f, 0.0f), mw23 = make_float2(0.0f, 0.0f);
    if constexpr (TileFmt<TYPE>::kAffine) {
        float mws[4];
        row_mins<TYPE>(tile + SOFF, 4 * i, mws);
        mw01 = pack2(mws[0], mws[1]);
        mw23 = pack2(mws[2], mws[3]);
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const uint4 a = act[4 * t + j];
        int S[4];
        const int c0 = TileFmt<TYPE>::kAffine ? 0 : (int)a.z;
#pragma unroll
        for (int r = 0; r < 4; ++r) S[r] = __dp4a((int)R[r][0], (int)a.x, __dp4a((int)R[r][1], (int)a.y, c0));
        const float da = __uint_as_float(a.w);
        const float2 da2 = pack2(da, da);
        acc[t][0] = ffma2(pack2((float)S[0], (float)S[1]), fmul2(dw01, da2), acc[t][0]);
        acc[t][1] = ffma2(pack2((float)S[2], (float)S[3]), fmul2(dw23, da2), acc[t][1]);
        if constexpr (TileFmt<TYPE>::kAffine) {
            // + m_w * d_a * (sum of this lane's 8 activations); the 4 quarters add up to the block's sum
            const float as = (float)(int)a.z;
            const float2 as2 = pack2(as, as);
            acc[t][0] = ffma2(as2, fmul2(mw01, da2), acc[t][0]);
            acc[t][1] = ffma2(as2, fmul2(mw23, da2), acc[t][1]);
        }
    }
}

struct Dp4aLayout {
    int ring, bars, act, red, total;
};
template <int TYPE, int MT, int CW, int TPW>
__host__ __device__ inline Dp4aLayout dp4a_layout(int nkc, int stages) {
    constexpr int TS = TileFmt<TYPE>::kBytes;
    Dp4aLayout L;
    int off = 0;
    L.bars = off;  off += (kDp4aSub<TYPE> + 1) * kMaxRingStages * 8 + 16;   // full [stage][part], empty [stage], abort flag
    off = (off + 127) & ~127;
    L.ring = off;  off += stages * CW * TPW * TS;
    off = (off + 15) & ~15;
    L.act = off;   off += MT * nkc * 4 * 16;                 // [nkc][MT][4] uint4
    L.red = off;   off += CW * MT * 32 * 4;                  // [CW][MT][32] float
    L.total = off;
    return L;
}

// MT = token capacity (1, 2 or 4); p.M <= MT tokens are live.  TPW independent tiles per warp and stage.
// SHARE_X (fused only, launched in clusters): CTA r of a cluster of C quantizes the blocks jt with
// jt % C == r and stores each record into all C CTAs' shared memory; one thread per CTA then arrives
// on every CTA's exchange barrier, which completes once all C CTAs have published their share.
template <int TYPE, int MT, int CW, bool FUSED, int TPW, bool SHARE_X = false>
__global__ void __launch_bounds__(32 * (1 + CW), 16 / CW) matvec_dp4a_kernel(const MvParams p) {
    static_assert(FUSED || !SHARE_X, "the shared staging quantizes fp32 rows");
    constexpr int kTilesPerStage = CW * TPW;
    constexpr int TS = TileFmt<TYPE>::kBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const Dp4aLayout L = dp4a_layout<TYPE, MT, CW, TPW>(p.nkc, p.stages);
    uint8_t *ring = smem + L.ring;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kMaxRingStages * kDp4aSub<TYPE>;     // full: [stage][part]
    volatile int *abort = reinterpret_cast<volatile int *>(empty + kMaxRingStages);
    uint64_t *xbar = empty + kMaxRingStages + 1;          // exchange barrier (SHARE_X), after the abort flag
    uint4 *act_s = reinterpret_cast<uint4 *>(smem + L.act);
    float *red_s = reinterpret_cast<float *>(smem + L.red);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stages = p.stages, nkc = p.nkc;

    if (threadIdx.x == 0) {
        // every stage the ring could have: no dependence on the launch parameters
#pragma unroll
        for (int s = 0; s < kMaxRingStages; ++s) {
#pragma unroll
            for (int q = 0; q < kDp4aSub<TYPE>; ++q) mbar_init(smem_u32(&full[s * kDp4aSub<TYPE> + q]), 1);
            mbar_init(smem_u32(&empty[s]), CW);
        }
        if constexpr (SHARE_X) mbar_init(smem_u32(xbar), cluster_size());
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // SHARE_X: every thread signals the cluster barrier once, here (this CTA's barriers exist); each
    // waits on it before it leaves or touches another CTA's barrier, so no CTA arrives on a barrier
    // that is not initialised yet and none exits while its cluster peers may still write to it.
    if constexpr (SHARE_X) asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
    // A grid launched after this one as a programmatic dependent may start now: it waits for this
    // grid to complete before it reads anything this grid writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        produce<TS, kTilesPerStage, kDp4aSub<TYPE>>(p, ring, full, empty, abort, lane);
        if constexpr (SHARE_X) asm volatile("barrier.cluster.wait;" ::: "memory");
        return;
    }

    const int cw = warp - 1;
    const int i = lane & 7, j = lane >> 3;

    // the activations may come from the grid launched just before this one (see produce)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // records e = (block jt, token t, quarter q) at act_s[(jt * MT + t) * 4 + q]; each thread first
    // issues the loads of its records (up to MT of them at a time), then builds them
    constexpr int kStageBatch = MT;
    const int total = MT * nkc * 4;
    bool x_ok = true;
    if constexpr (!FUSED) {
        for (int w0 = cw * 32; w0 < total; w0 += CW * 32 * kStageBatch) {     // warp-uniform passes
            const int base = w0 + lane;
            uint2 v[kStageBatch];
            uint16_t db[kStageBatch];
#pragma unroll
            for (int u = 0; u < kStageBatch; ++u) {
                const int e = base + u * CW * 32, q = e & 3, tok = (e >> 2) % MT, jt = (e >> 2) / MT;
                v[u] = make_uint2(0u, 0u);
                db[u] = 0;
                if (e < total && tok < p.M && QMM_DCHECK(p.kt0 + jt < p.nkt)) {
                    const int64_t kt = p.kt0 + jt;
                    db[u] = p.a_d[(int64_t)tok * p.nkt + kt];
                    v[u] = *reinterpret_cast<const uint2 *>(p.a_q + (int64_t)tok * p.K + kt * 32 + 8 * q);
                }
            }
#pragma unroll
            for (int u = 0; u < kStageBatch; ++u) {
                const int e = base + u * CW * 32, q = e & 3, tok = (e >> 2) % MT;
                if (e < total)
                    act_s[e] = tok < p.M ? dp4a_record(TYPE, v[u], q, __half2float(__ushort_as_half(db[u]))) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
    } else if constexpr (!SHARE_X) {
        // a record is made by the lane quad of its 4 quarters (all lanes of a warp iterate together)
        for (int base = cw * 32; base < total; base += CW * 32 * kStageBatch) {
            float v[kStageBatch][8];
#pragma unroll
            for (int u = 0; u < kStageBatch; ++u) {
                const int e = base + u * CW * 32 + lane, q = e & 3, tok = (e >> 2) % MT, jt = (e >> 2) / MT;
                load_quarter(p, e < total && tok < p.M, tok, p.kt0 + jt, q, v[u]);
            }
#pragma unroll
            for (int u = 0; u < kStageBatch; ++u) {
                const int e = base + u * CW * 32 + lane, q = e & 3, tok = (e >> 2) % MT;
                float da;
                const uint2 c = quantize_loaded(v[u], da);
                if (e < total) act_s[e] = tok < p.M ? dp4a_record(TYPE, c, q, da) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
    } else {
        // this CTA's share: blocks jt = rank + C * l; local record index el = (l * MT + tok) * 4 + q
        const int rank = (int)cluster_rank(), csize = (int)cluster_size();
        const int nloc = (nkc - rank + csize - 1) / csize;
        const int total_l = MT * nloc * 4;
        for (int base = cw * 32; base < total_l; base += CW * 32 * kStageBatch) {
            float v[kStageBatch][8];
#pragma unroll
            for (int u = 0; u < kStageBatch; ++u) {
                const int el = base + u * CW * 32 + lane, q = el & 3, tok = (el >> 2) % MT;
                const int jt = rank + csize * ((el >> 2) / MT);
                load_quarter(p, el < total_l && tok < p.M, tok, p.kt0 + jt, q, v[u]);
            }
#pragma unroll
            for (int u = 0; u < kStageBatch; ++u) {
                const int el = base + u * CW * 32 + lane, q = el & 3, tok = (el >> 2) % MT;
                const int jt = rank + csize * ((el >> 2) / MT);
                float da;
                const uint2 c = quantize_loaded(v[u], da);
                if (el < total_l && QMM_DCHECK(jt < nkc)) {
                    const uint4 rec = tok < p.M ? dp4a_record(TYPE, c, q, da) : make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t dst = smem_u32(&act_s[(jt * MT + tok) * 4 + q]);
                    for (int r = 0; r < csize; ++r) st_peer_v4(peer_addr(dst, (uint32_t)r), rec);
                }
            }
        }
        // publish: this CTA's stores are done (named barrier), then one thread releases them to every
        // CTA of the cluster; every consumer thread then acquires all C shares
        consumer_sync<CW>();
        asm volatile("barrier.cluster.wait;" ::: "memory");
        if (cw == 0 && lane == 0) {
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            for (int r = 0; r < csize; ++r) mbar_arrive_peer(peer_addr(smem_u32(xbar), (uint32_t)r));
        }
        if (!wait_cluster_bounded(smem_u32(xbar), 0u, abort, &g_mv_status, kWaitLimitNs)) {
            // a share never came: keep this CTA (and its shared memory) alive for a late writer as
            // long as a second bounded wait allows, then skip the tiles
            wait_drain(smem_u32(xbar), 0u);
            x_ok = false;
        }
    }
    uint32_t tb[4] = {0u, 0u, 0u, 0u};
    if constexpr (TileFmt<TYPE>::kLut) {
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
            for (int b = 0; b < 4; ++b) tb[w] |= ((uint32_t)(p.lut.v[4 * w + b] & 0xFF)) << (8 * b);
    }
    consumer_sync<CW>();

    uint32_t it = 0;
    bool ok = true;
    if constexpr (SHARE_X) ok = __all_sync(0xffffffffu, x_ok);
    for (int64_t ct = blockIdx.x; ct < p.n_col_tiles; ct += gridDim.x) {
        float2 acc[MT][2];           // per token: rows (4i, 4i+1), (4i+2, 4i+3)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = make_float2(0.0f, 0.0f);

        for (int j0 = 0; j0 < nkc; j0 += kTilesPerStage, ++it) {
            const int s = (int)(it % (uint32_t)stages);
            const uint32_t ph = (it / (uint32_t)stages) & 1u;
            // warp cw takes tiles cw * TPW .. cw * TPW + TPW - 1 of the stage, which arrive with part
            // cw / (CW / kDp4aSub<TYPE>) of its copies
            if (ok) ok = __all_sync(0xffffffffu, wait_bounded(smem_u32(&full[s * kDp4aSub<TYPE> + cw / (CW / kDp4aSub<TYPE>)]), ph, abort));
            if (ok && QMM_DCHECK(s < stages)) {
                // only the last stage of a pass can be partial
                const uint8_t *tile = ring + (s * kTilesPerStage + cw * TPW) * TS;
                const uint4 *act = act_s + (j0 + cw * TPW) * MT * 4;
                if (j0 + kTilesPerStage <= nkc) {
#pragma unroll
                    for (int u = 0; u < TPW; ++u) dp4a_tile<TYPE, MT>(tile + u * TS, act + u * MT * 4, i, j, tb, acc);
                } else {
#pragma unroll
                    for (int u = 0; u < TPW; ++u)
                        if (j0 + cw * TPW + u < nkc) dp4a_tile<TYPE, MT>(tile + u * TS, act + u * MT * 4, i, j, tb, acc);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }

        // ---- quarters (lanes i, i+8, i+16, i+24), then warps, in a fixed order ----
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float v[4];
            unpack2(acc[t][0], v[0], v[1]);
            unpack2(acc[t][1], v[2], v[3]);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                v[r] += __shfl_xor_sync(0xffffffffu, v[r], 8);
                v[r] += __shfl_xor_sync(0xffffffffu, v[r], 16);
            }
            if (j == 0) *reinterpret_cast<float4 *>(red_s + (cw * MT + t) * 32 + 4 * i) = make_float4(v[0], v[1], v[2], v[3]);
        }
        consumer_sync<CW>();
        if (cw < MT && cw < p.M) {
            const int t = cw;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < CW; ++w) sum += red_s[(w * MT + t) * 32 + lane];
            const int64_t n = ct * 32 + lane;
            if (ok && n < p.N) {
                float *dst = p.y + (int64_t)t * p.ldy + n;
                *dst = p.accumulate ? (*dst + sum) : sum;
            }
        }
        consumer_sync<CW>();
    }
}

struct Plan {
    int nkc, stages, ctas_per_sm;
    size_t smem;
};

// Ring depth from what is left of the CTA's share of shared memory: CW = 16 runs one wide CTA per
// SM (all of it), CW = 8 two narrow CTAs per SM (half each).
template <int TS, int CW, int TPW>
Plan plan_ring(int nkc, int fixed_bytes) {
    constexpr int kTilesPerStage = CW * TPW;
    Plan pl;
    pl.nkc = nkc;
    const int stage_bytes = kTilesPerStage * TS + 16;
    const int budget = (CW == 16) ? kSmemLimit : kSmemLimit / 2;
    const int st = (budget - 1024 - fixed_bytes - 128) / stage_bytes;
    pl.stages = st > kMaxRingStages ? kMaxRingStages : (st < 2 ? 2 : st);
    pl.ctas_per_sm = 16 / CW;
    return pl;
}

int chunk_tiles(int64_t nkt, int64_t bytes_per_tile) {
    int64_t nkc = kActBudget / bytes_per_tile;
    if (nkc > nkt) nkc = nkt;
    if (nkc < 1) nkc = 1;
    return (int)nkc;
}

// SM count of the device current at the first call (thread-safe static initialization).
int num_sms() {
    static const int sms = []() {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 152;
        return n;
    }();
    return sms;
}

// CTAs of one launch: one persistent CTA per SM (two narrow ones), at most one per column tile.
inline int64_t decode_grid(const Plan &pl, int64_t N) {
    const int64_t nct = (N + 31) / 32;
    const int64_t grid = (int64_t)num_sms() * pl.ctas_per_sm;
    return grid > nct ? nct : grid;
}

// Cluster size for the shared activation staging: the largest C in {8, 4, 2} for which the grid,
// rounded up to a multiple of C, fits in clusters that can all be resident at once
// (cudaOccupancyMaxActiveClusters); 1 if none does.  A cluster of C CTAs reads 1/C of the host rows
// per CTA instead of all of them.  The answer depends on the kernel only: its ring is sized to fill
// its share of shared memory, which pins it to one CTA per SM (16 consumer warps) or two (8), so it
// is cached per kernel (cache[i] = clusters + 1 once known).  A stale or refused answer costs
// speed, never correctness: clusters that do not fit at once run one after another.
constexpr int kShareSizes[3] = {8, 4, 2};
template <typename Kern>
int share_cluster_size(Kern kern, int threads, size_t smem, int64_t grid, int (&cache)[3]) {
    for (int i = 0; i < 3; ++i) {
        const int c = kShareSizes[i];
        const int64_t g = (grid + c - 1) / c * c;
        int n = __atomic_load_n(&cache[i], __ATOMIC_RELAXED) - 1;
        if (n < 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)g, 1, 1);
            cfg.blockDim = dim3((unsigned)threads, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 0) {
                n = 0;
                (void)cudaGetLastError();        // a refused query is an answer (no clusters), not an error
            }
            __atomic_store_n(&cache[i], n + 1, __ATOMIC_RELAXED);
        }
        if ((int64_t)n * c >= g) return c;
    }
    return 1;
}

// Launch `kern` once per K pass (passes after the first add into y).  Each launch is a programmatic
// dependent of the grid before it on the stream: it may start while that grid is still running (if
// that grid allows it), and the kernel waits for it before reading activations or y.  cs > 1: in
// clusters of cs CTAs, the grid rounded up to a multiple of cs (CTAs past the last column tile only
// stage their share of the activations).
template <typename Kern>
cudaError_t launch_passes(Kern kern, int threads, const Plan &pl, const Lut16 &lut, const uint8_t *tiled, int64_t K,
                          int64_t N, const ActSrc &a, int M, float *y, int64_t ldy, cudaStream_t s, int cs = 1) {
    const int64_t nkt = K / 32, nct = (N + 31) / 32;
    if (pl.smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;   // a ring of two stages must fit
    int64_t grid = decode_grid(pl, N);
    if (cs > 1) grid = (grid + cs - 1) / cs * cs;
    for (int64_t kt0 = 0; kt0 < nkt; kt0 += pl.nkc) {
        MvParams p;
        p.tiled = tiled;
        p.a_q = a.a_q;
        p.a_d = a.a_d;
        p.x = a.x;
        p.ldx = a.ldx;
        p.x_vec = a.x != nullptr && (reinterpret_cast<uintptr_t>(a.x) & 15u) == 0 && a.ldx % 4 == 0;
        p.y = y;
        p.K = K;
        p.nkt = nkt;
        p.N = N;
        p.ldy = ldy;
        p.n_col_tiles = nct;
        p.M = M;
        p.kt0 = (int)kt0;
        p.nkc = (int)((nkt - kt0) < pl.nkc ? (nkt - kt0) : pl.nkc);
        p.accumulate = kt0 > 0;
        p.stages = pl.stages;
        p.lut = lut;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3((unsigned)threads, 1, 1);
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)cs;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = cs > 1 ? 2 : 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int TYPE, int NF, int CW, bool FUSED>
cudaError_t run_mma(const uint8_t *tiled, int64_t K, int64_t N, const ActSrc &a, int M, float *y, int64_t ldy,
                    cudaStream_t s) {
    constexpr int TS = TileFmt<TYPE>::kBytes;
    const int nkc = chunk_tiles(K / 32, 64 * (int64_t)M);
    Plan pl = plan_ring<TS, CW, kTilesPerWarp>(nkc, mv_layout<TYPE, NF, CW>(M, nkc, 0).total);
    pl.smem = (size_t)mv_layout<TYPE, NF, CW>(M, nkc, pl.stages).total + 128;
    auto kern = matvec_kernel<TYPE, NF, CW, FUSED>;
    static int attr_done[4] = {0, 0, 0, 0};
    const cudaError_t e = ensure_smem_limit(kern, kSmemLimit, attr_done);
    if (e != cudaSuccess) return e;
    return launch_passes(kern, 32 * (1 + CW), pl, lut_for((qmm_type)TYPE), tiled, K, N, a, M, y, ldy, s);
}

template <int TYPE, int MT, int CW, bool FUSED>
cudaError_t run_dp4a(const uint8_t *tiled, int64_t K, int64_t N, const ActSrc &a, int M, float *y, int64_t ldy,
                     cudaStream_t s) {
    constexpr int TS = TileFmt<TYPE>::kBytes;
    constexpr int TPW = kDp4aTilesPerWarp<TYPE>;
    const int nkc = chunk_tiles(K / 32, 64 * (int64_t)MT);
    Plan pl = plan_ring<TS, CW, TPW>(nkc, dp4a_layout<TYPE, MT, CW, TPW>(nkc, 0).total);
    pl.smem = (size_t)dp4a_layout<TYPE, MT, CW, TPW>(nkc, pl.stages).total + 128;
    if constexpr (FUSED) {
        if (a.x_host) {
            // rows in host memory: one read of them per cluster instead of one per CTA
            auto kx = matvec_dp4a_kernel<TYPE, MT, CW, true, TPW, true>;
            static int attr_x[4] = {0, 0, 0, 0};
            static int clusters[3] = {0, 0, 0};
            const cudaError_t e = ensure_smem_limit(kx, kSmemLimit, attr_x);
            if (e != cudaSuccess) return e;
            const int cs = share_cluster_size(kx, 32 * (1 + CW), pl.smem, decode_grid(pl, N), clusters);
            if (cs > 1) return launch_passes(kx, 32 * (1 + CW), pl, lut_for((qmm_type)TYPE), tiled, K, N, a, M, y, ldy, s, cs);
        }
    }
    auto kern = matvec_dp4a_kernel<TYPE, MT, CW, FUSED, TPW>;
    static int attr_done[4] = {0, 0, 0, 0};
    const cudaError_t e = ensure_smem_limit(kern, kSmemLimit, attr_done);
    if (e != cudaSuccess) return e;
    return launch_passes(kern, 32 * (1 + CW), pl, lut_for((qmm_type)TYPE), tiled, K, N, a, M, y, ldy, s);
}

// Up to kDp4aMaxM tokens: int8 dot products; more: fp16 mma.sync.  Many column tiles: two narrow
// CTAs per SM hide latency best; few: one wide CTA per SM streams each column tile twice as fast,
// which keeps the rounds of a small grid short and balanced.
template <int TYPE, bool FUSED>
cudaError_t run(const uint8_t *tiled, int64_t K, int64_t N, const ActSrc &a, int M, float *y, int64_t ldy,
                cudaStream_t s) {
    const bool narrow = (N + 31) / 32 >= (int64_t)num_sms() * 8;
#define QMM_MV_ARGS tiled, K, N, a, M, y, ldy, s
    if (M <= kDp4aMaxM) {
        if (M == 1) return narrow ? run_dp4a<TYPE, 1, 8, FUSED>(QMM_MV_ARGS) : run_dp4a<TYPE, 1, 16, FUSED>(QMM_MV_ARGS);
        if (M == 2) return narrow ? run_dp4a<TYPE, 2, 8, FUSED>(QMM_MV_ARGS) : run_dp4a<TYPE, 2, 16, FUSED>(QMM_MV_ARGS);
        return narrow ? run_dp4a<TYPE, 4, 8, FUSED>(QMM_MV_ARGS) : run_dp4a<TYPE, 4, 16, FUSED>(QMM_MV_ARGS);
    }
    if (M <= 8) return narrow ? run_mma<TYPE, 1, 8, FUSED>(QMM_MV_ARGS) : run_mma<TYPE, 1, 16, FUSED>(QMM_MV_ARGS);
    return narrow ? run_mma<TYPE, 2, 8, FUSED>(QMM_MV_ARGS) : run_mma<TYPE, 2, 16, FUSED>(QMM_MV_ARGS);
#undef QMM_MV_ARGS
}

// ================= flat (untiled) rows: decode straight from the GGML blocks =================
// The pages keep every supported type usable from its flat row-major GGML layout as well as from the
// tiles.  Here a chunk is 32 consecutive weight rows; a stage holds those rows x kFlatKB blocks, brought
// in by one 2-D tensor copy (the flat weight seen as rows of 8-byte words; a row must be a whole
// number of 16-byte units).  Warp w of the 16 consumer warps takes rows w and w + 16 of the chunk and
// lane b block b of the stage: it loads the block's bytes as aligned words (blocks are 17..34 bytes,
// so most are unaligned), extracts the head and the codes with funnel shifts, turns the codes into 8
// int8x4 words and takes dp4a against the staged activations, whose byte order matches those words
// (natural order for Q4_0 / Q4_1 / Q8_0; for the table types the order of the table lookup, see
// stage_flat).  Row sums: a fixed butterfly over the 32 lanes at the end of the chunk.
constexpr int kFlatKB = 32;            // blocks per row and stage
constexpr int kFlatCW = 16;            // consumer warps
constexpr int kFlatMT = 4;             // tokens per launch
// Parts per stage: 8-row tensor copies, each completing its own barrier; warp w takes rows 2w and
// 2w + 1, so the warps of a stage's first rows compute while the rest lands.
constexpr int kFlatSub = 4;
constexpr int kFlatMaxStages = 8;      // ring depth cap; the barriers are laid out for this many

template <int TYPE>
struct FlatFmt {
    // bytes per 32 weights (Q4_K: an eighth of a 144-byte super-block)
    static constexpr int kBlock = TYPE == QMM_Q8_0    ? kBlock8Bytes
                                  : TYPE == QMM_MXFP4 ? kBlockMxBytes
                                  : TYPE == QMM_Q4_1  ? kBlock41Bytes
                                  : TYPE == QMM_Q4_K  ? kQ4KBytesPer32
                                                      : kBlock4Bytes;
    static constexpr int kHead = TYPE == QMM_MXFP4 ? 1 : (TYPE == QMM_Q4_1 ? 4 : 2);
    // Block words u[i] (bytes 4i..4i+3 of the block) that the code words touch: the last code word
    // starts at byte kBlock - 4 and spans u[(kBlock - 4) / 4] and, unless it is word aligned, the next.
    static constexpr int kU = (kBlock - 4) / 4 + ((kBlock - 4) % 4 ? 1 : 0) + 1;
};

struct FlatParams {
    const int8_t *a_q;
    const uint16_t *a_d;
    float *y;
    int64_t K, nkt, N, ldy, n_chunks;
    int M, stages, kt0, nkc, accumulate;
    Lut16 lut;
};

struct FlatLayout {
    int ring, bars, act, aux, total;
};
template <int TYPE, int MT>
__host__ __device__ inline FlatLayout flat_layout(int nkc, int stages) {
    FlatLayout L;
    int off = 0;
    L.bars = off;  off += (kFlatSub + 1) * kFlatMaxStages * 8 + 16;   // full [stage][part], empty [stage], abort flag
    off = (off + 127) & ~127;
    L.ring = off;  off += stages * 32 * kFlatKB * FlatFmt<TYPE>::kBlock;
    off += 16;                                                // word reads of the last block run past the ring
    off = (off + 15) & ~15;
    L.act = off;   off += MT * nkc * 32;                      // [MT][nkc] 32 int8 in the decode order
    L.aux = off;   off += MT * nkc * 8;                       // [MT][nkc] {fp32 d_a, int corr or sum}
    L.total = off;
    return L;
}

// The 8 int8x4 words of one flat block (blk_off = its byte offset from a 16-byte aligned base) in the
// staged activation order, and its scale (and Q4_1 min).  The block is read as aligned words, shifted
// into block-relative words u[] by one funnel shift each (blocks of 17, 18 or 34 bytes start at any
// byte offset), then code word k at byte kHead + 4k is a fixed funnel shift of two u[].
template <int TYPE>
__device__ __forceinline__ void flat_block_words(const uint8_t *base, int blk_off, uint32_t (&W)[8], float &dw, float &mw,
                                                 const uint32_t (&tb)[4]) {
    constexpr int BB = FlatFmt<TYPE>::kBlock, H = FlatFmt<TYPE>::kHead, NU = FlatFmt<TYPE>::kU;
    uint32_t u[NU];
    if constexpr (BB % 4 == 0) {
        const uint32_t *w32 = reinterpret_cast<const uint32_t *>(base + blk_off);
#pragma unroll
        for (int i = 0; i < NU; ++i) u[i] = w32[i];
    } else {
        const uint32_t *w32 = reinterpret_cast<const uint32_t *>(base + (blk_off & ~3));
        const uint32_t sh = 8u * (uint32_t)(blk_off & 3);
        uint32_t w[NU + 1];
#pragma unroll
        for (int i = 0; i <= NU; ++i) w[i] = w32[i];
#pragma unroll
        for (int i = 0; i < NU; ++i) u[i] = __funnelshift_r(w[i], w[i + 1], sh);
    }
    // code word at block byte H + 4k
    auto at = [&](int k) -> uint32_t {
        constexpr int s = 8 * (H & 3);
        const int q = (H >> 2) + k;
        if constexpr (s == 0) return u[q];
        else return __funnelshift_r(u[q], u[q + 1], s);
    };
    mw = 0.0f;
    if constexpr (TYPE == QMM_MXFP4) {
        dw = mx_half_scale(u[0] & 0xFFu);
    } else {
        dw = __low2float(bits_h2(u[0]));
        if constexpr (TYPE == QMM_Q4_1) mw = __high2float(bits_h2(u[0]));
    }
    if constexpr (TYPE == QMM_Q8_0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) W[k] = at(k);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t qk = at(k);                      // quant bytes 4k..4k+3: elements 4k.. (low), 16+4k.. (high)
            if constexpr (TileFmt<TYPE>::kNibbleInt) {
                W[k] = qk & 0x0F0F0F0Fu;
                W[4 + k] = (qk >> 4) & 0x0F0F0F0Fu;
            } else {
                // table values in nibble order lo(b0), hi(b0), lo(b1), hi(b1) | lo(b2), hi(b2), lo(b3), hi(b3)
                const uint32_t m = qk & 0x77777777u;
                const uint32_t sel0 = ((qk >> 1) & 0x4444u) | 0x3210u;
                const uint32_t sel1 = ((qk >> 17) & 0x4444u) | 0x3210u;
                const uint32_t m1 = m >> 16;
                W[2 * k] = __byte_perm(__byte_perm(tb[0], tb[1], m), __byte_perm(tb[2], tb[3], m), sel0);
                W[2 * k + 1] = __byte_perm(__byte_perm(tb[0], tb[1], m1), __byte_perm(tb[2], tb[3], m1), sel1);
            }
        }
    }
}

// Q4_K: sub-block j (0..7) of the super-block at `sb` (4-byte aligned): its 8 code words in natural
// order, and the row pair of its tile, fp16(d*sc_j) and fp16(-dmin*m_j), so that the flat product
// is the tiled one.
__device__ __forceinline__ void flat_q4k_words(const uint8_t *sb_bytes, int j, uint32_t (&W)[8], float &dw, float &mw) {
    const uint32_t *sb = reinterpret_cast<const uint32_t *>(sb_bytes);
    const int jj = j & 3;
    const uint32_t head = sb[0];
    const uint32_t b0 = (sb[1] >> (8 * jj)) & 0xFF, b1 = (sb[2] >> (8 * jj)) & 0xFF, b2 = (sb[3] >> (8 * jj)) & 0xFF;
    const uint32_t sc = j < 4 ? (b0 & 63) : ((b2 & 15) | ((b0 >> 6) << 4));
    const uint32_t m = j < 4 ? (b1 & 63) : ((b2 >> 4) | ((b1 >> 6) << 4));
    const float d = __low2float(bits_h2(head)), dmin = __high2float(bits_h2(head));
    dw = __half2float(__float2half_rn(__fmul_rn(d, (float)sc)));
    mw = __half2float(__float2half_rn(-__fmul_rn(dmin, (float)m)));
    const uint4 *qs = reinterpret_cast<const uint4 *>(sb + 4 + 8 * (j >> 1));   // 16-byte aligned
    const uint4 q0 = qs[0], q1 = qs[1];
    const int sh = 4 * (j & 1);
    const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) W[k] = (q[k] >> sh) & 0x0F0F0F0Fu;
}

// Stage the 32 activations of one (token, block) in the order of flat_block_words, plus d_a and the
// Q4_0 start value -8 * sum(a) (Q4_1: the sum itself, for the min term).
template <int TYPE>
__device__ __forceinline__ void stage_flat(const int8_t *a32, float da, uint32_t *dst_words, uint2 *dst_aux) {
    const uint4 v0 = *reinterpret_cast<const uint4 *>(a32), v1 = *reinterpret_cast<const uint4 *>(a32 + 16);
    const uint32_t a[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};   // natural order
    if constexpr (TileFmt<TYPE>::kLut) {
        // table lookup order: for k = 0..3, [a(4k), a(4k+16), a(4k+1), a(4k+17)], [a(4k+2), a(4k+18), a(4k+3), a(4k+19)]
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            dst_words[2 * k] = __byte_perm(a[k], a[4 + k], 0x5140);
            dst_words[2 * k + 1] = __byte_perm(a[k], a[4 + k], 0x7362);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) dst_words[k] = a[k];
    }
    int asum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) asum = __dp4a((int)a[k], 0x01010101, asum);
    const int aux = TYPE == QMM_Q4_0 ? -8 * asum : (TileFmt<TYPE>::kAffine ? asum : 0);
    *dst_aux = make_uint2(__float_as_uint(da), (uint32_t)aux);
}

// MT = token capacity (1, 2 or 4); p.M <= MT tokens are live.
template <int TYPE, int MT>
__global__ void __launch_bounds__(32 * (1 + kFlatCW), 1)
    matvec_flat_kernel(const FlatParams p, const __grid_constant__ CUtensorMap w_map) {
    constexpr int BB = FlatFmt<TYPE>::kBlock;
    constexpr int kRowStage = kFlatKB * BB;                     // bytes of one row in a stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const FlatLayout L = flat_layout<TYPE, MT>(p.nkc, p.stages);
    uint8_t *ring = smem + L.ring;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kFlatMaxStages * kFlatSub;     // full: [stage][part]
    volatile int *abort = reinterpret_cast<volatile int *>(empty + kFlatMaxStages);
    uint32_t *act_w = reinterpret_cast<uint32_t *>(smem + L.act);
    uint2 *act_x = reinterpret_cast<uint2 *>(smem + L.aux);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stages = p.stages, nkc = p.nkc;

    if (threadIdx.x == 0) {
        // every stage the ring could have: no dependence on the launch parameters
#pragma unroll
        for (int s = 0; s < kFlatMaxStages; ++s) {
#pragma unroll
            for (int q = 0; q < kFlatSub; ++q) mbar_init(smem_u32(&full[s * kFlatSub + q]), 1);
            mbar_init(smem_u32(&empty[s]), kFlatCW);
        }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---- producer: per chunk and stage, kFlatSub 2-D tensor copies of 32 / kFlatSub rows x kFlatKB
        // blocks (rows past N and blocks past the row end arrive as zeros and are never used) ----
        uint32_t it = 0;
        bool ok = true;
        for (int64_t ch = blockIdx.x; ch < p.n_chunks && ok; ch += gridDim.x) {
            for (int kb0 = 0; kb0 < nkc; kb0 += kFlatKB, ++it) {
                const int s = (int)(it % (uint32_t)stages);
                const uint32_t ph = (it / (uint32_t)stages) & 1u;
                if (!__all_sync(0xffffffffu, wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort))) { ok = false; break; }
                if (lane == 0) {
#pragma unroll
                    for (int q = 0; q < kFlatSub; ++q) {
                        constexpr int kRows = 32 / kFlatSub;
                        const uint32_t fb = smem_u32(&full[s * kFlatSub + q]);
                        // rows ch*32 + kRows*q .. of blocks kt0 + kb0.. into part q of ring slot s
                        if (QMM_DCHECK(s < stages && ch < p.n_chunks && p.kt0 + kb0 < p.nkt)) {
                            mbar_arrive_expect_tx(fb, (uint32_t)(kRows * kRowStage));
                            tma_load_2d(smem_u32(ring + (s * 32 + kRows * q) * kRowStage), &w_map, (p.kt0 + kb0) * BB / 8,
                                        (int)(ch * 32 + kRows * q), fb);
                        } else {
                            mbar_arrive(fb);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0 && it > 0) {
            const uint32_t last = it - 1;
            for (uint32_t k = 0; k < (uint32_t)stages && k <= last; ++k) {
                const uint32_t i = last - k;
                for (int q = 0; q < kFlatSub; ++q) wait_drain(smem_u32(&full[(i % stages) * kFlatSub + q]), (i / stages) & 1u);
            }
        }
        return;
    }

    const int cw = warp - 1, ctid = threadIdx.x - 32;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int e = ctid; e < MT * nkc; e += kFlatCW * 32) {
        const int tok = e / nkc, jt = e - tok * nkc;
        if (tok < p.M) {
            const int64_t kt = p.kt0 + jt;
            const float da = __half2float(__ushort_as_half(p.a_d[(int64_t)tok * p.nkt + kt]));
            stage_flat<TYPE>(p.a_q + (int64_t)tok * p.K + kt * 32, da, act_w + (size_t)e * 8, act_x + e);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) act_w[(size_t)e * 8 + k] = 0u;
            act_x[e] = make_uint2(0u, 0u);
        }
    }
    uint32_t tb[4] = {0u, 0u, 0u, 0u};
    if constexpr (TileFmt<TYPE>::kLut) {
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
            for (int b = 0; b < 4; ++b) tb[w] |= ((uint32_t)(p.lut.v[4 * w + b] & 0xFF)) << (8 * b);
    }
    consumer_sync<kFlatCW>();

    uint32_t it = 0;
    bool ok = true;
    for (int64_t ch = blockIdx.x; ch < p.n_chunks; ch += gridDim.x) {
        float acc[2][MT];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[r][t] = 0.0f;
        for (int kb0 = 0; kb0 < nkc; kb0 += kFlatKB, ++it) {
            const int s = (int)(it % (uint32_t)stages);
            const uint32_t ph = (it / (uint32_t)stages) & 1u;
            // rows 2cw, 2cw + 1 arrive with part cw / (kFlatCW / kFlatSub) of the stage
            if (ok) ok = __all_sync(0xffffffffu, wait_bounded(smem_u32(&full[s * kFlatSub + cw / (kFlatCW / kFlatSub)]), ph, abort));
            const int jt = kb0 + lane;                         // this lane's block
            if (ok && jt < nkc) {
                const uint8_t *st = ring + s * 32 * kRowStage;
                uint4 aw[MT][2];
                uint2 ax[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(act_w + ((size_t)t * nkc + jt) * 8);
                    aw[t][0] = src[0];
                    aw[t][1] = src[1];
                    ax[t] = act_x[t * nkc + jt];
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = 2 * cw + r;
                    uint32_t W[8];
                    float dw, mw;
                    if constexpr (TYPE == QMM_Q4_K)
                        flat_q4k_words(st + row * kRowStage + (lane >> 3) * kSuperQ4KBytes, lane & 7, W, dw, mw);
                    else
                        flat_block_words<TYPE>(st, row * kRowStage + lane * BB, W, dw, mw, tb);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        if (t >= p.M) break;
                        const int c0 = TYPE == QMM_Q4_0 ? (int)ax[t].y : 0;
                        int S = __dp4a((int)W[0], (int)aw[t][0].x, c0);
                        S = __dp4a((int)W[1], (int)aw[t][0].y, S);
                        S = __dp4a((int)W[2], (int)aw[t][0].z, S);
                        S = __dp4a((int)W[3], (int)aw[t][0].w, S);
                        S = __dp4a((int)W[4], (int)aw[t][1].x, S);
                        S = __dp4a((int)W[5], (int)aw[t][1].y, S);
                        S = __dp4a((int)W[6], (int)aw[t][1].z, S);
                        S = __dp4a((int)W[7], (int)aw[t][1].w, S);
                        const float da = __uint_as_float(ax[t].x);
                        acc[r][t] = fmaf((float)S, __fmul_rn(dw, da), acc[r][t]);
                        if constexpr (TileFmt<TYPE>::kAffine)
                            acc[r][t] = fmaf((float)(int)ax[t].y, __fmul_rn(mw, da), acc[r][t]);
                    }
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }
        // ---- row sums over the lanes (fixed butterfly), then y ----
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = acc[r][t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                const int64_t n = ch * 32 + 2 * cw + r;
                if (ok && lane == 0 && t < p.M && n < p.N) {
                    float *dst = p.y + (int64_t)t * p.ldy + n;
                    *dst = p.accumulate ? (*dst + v) : v;
                }
            }
    }
}

template <int TYPE, int MT>
cudaError_t run_flat(const uint8_t *flat, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d, int M, float *y,
                     int64_t ldy, cudaStream_t s) {
    constexpr int BB = FlatFmt<TYPE>::kBlock;
    const int64_t nkt = K / 32;
    int64_t nkc = kActBudget / (kFlatMT * 40);                  // staged bytes per (token, block): 32 + 8
                                                                // (the same K passes for every MT)
    nkc = nkc / kFlatKB * kFlatKB;
    if (nkc > nkt) nkc = nkt;
    const int fixed = flat_layout<TYPE, MT>((int)nkc, 0).total;
    const int stage_bytes = 32 * kFlatKB * BB + 16;
    int st = (kSmemLimit - 1024 - fixed - 128) / stage_bytes;
    st = st > kFlatMaxStages ? kFlatMaxStages : (st < 2 ? 2 : st);
    const size_t smem = (size_t)flat_layout<TYPE, MT>((int)nkc, st).total + 128;
    auto kern = matvec_flat_kernel<TYPE, MT>;
    static int attr_done[4] = {0, 0, 0, 0};
    cudaError_t e = ensure_smem_limit(kern, kSmemLimit, attr_done);
    if (e != cudaSuccess) return e;
    const int64_t n_chunks = (N + 31) / 32;
    int64_t grid = num_sms();
    if (grid > n_chunks) grid = n_chunks;
    // The flat weight as N rows of row_bytes / 8 eight-byte words; one box = 32 / kFlatSub rows x kFlatKB
    // blocks (a stage part).
    alignas(64) CUtensorMap w_map;
    e = make_map_2d(&w_map, CU_TENSOR_MAP_DATA_TYPE_UINT64, flat, (uint64_t)(nkt * BB / 8), (uint64_t)N,
                    (uint64_t)(nkt * BB), (uint32_t)(kFlatKB * BB / 8), (uint32_t)(32 / kFlatSub), CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    for (int64_t kt0 = 0; kt0 < nkt; kt0 += nkc) {
        FlatParams p;
        p.a_q = a_q;
        p.a_d = a_d;
        p.y = y;
        p.K = K;
        p.nkt = nkt;
        p.N = N;
        p.ldy = ldy;
        p.n_chunks = n_chunks;
        p.M = M;
        p.stages = st;
        p.kt0 = (int)kt0;
        p.nkc = (int)((nkt - kt0) < nkc ? (nkt - kt0) : nkc);
        p.accumulate = kt0 > 0;
        p.lut = lut_for((qmm_type)TYPE);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(32 * (1 + kFlatCW), 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, p, w_map);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int TYPE>
cudaError_t run_flat_mt(const uint8_t *flat, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d, int M, float *y,
                        int64_t ldy, cudaStream_t s) {
    if (M == 1) return run_flat<TYPE, 1>(flat, K, N, a_q, a_d, M, y, ldy, s);
    if (M == 2) return run_flat<TYPE, 2>(flat, K, N, a_q, a_d, M, y, ldy, s);
    return run_flat<TYPE, 4>(flat, K, N, a_q, a_d, M, y, ldy, s);
}

// Groups of at most kDecodeMaxM rows, one launch sequence each.
template <bool FUSED>
cudaError_t run_groups(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const ActSrc &a, int64_t M, float *y,
                       int64_t ldy, cudaStream_t s) {
    const int64_t nkt = K / 32;
    for (int64_t m0 = 0; m0 < M; m0 += kDecodeMaxM) {
        const int mm = (int)((M - m0) < kDecodeMaxM ? (M - m0) : kDecodeMaxM);
        ActSrc g = a;
        if (FUSED) {
            g.x = a.x + m0 * a.ldx;
        } else {
            g.a_q = a.a_q + m0 * K;
            g.a_d = a.a_d + m0 * nkt;
        }
        float *yy = y + m0 * ldy;
        cudaError_t e;
        switch (t) {
            case QMM_Q4_0: e = run<QMM_Q4_0, FUSED>(tiled, K, N, g, mm, yy, ldy, s); break;
            case QMM_IQ4_NL: e = run<QMM_IQ4_NL, FUSED>(tiled, K, N, g, mm, yy, ldy, s); break;
            case QMM_MXFP4: e = run<QMM_MXFP4, FUSED>(tiled, K, N, g, mm, yy, ldy, s); break;
            case QMM_Q4_1: e = run<QMM_Q4_1, FUSED>(tiled, K, N, g, mm, yy, ldy, s); break;
            default: e = run<QMM_Q8_0, FUSED>(tiled, K, N, g, mm, yy, ldy, s); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_matvec(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                          const uint16_t *a_d, int64_t M, float *y, int64_t ldy, cudaStream_t s) {
    const ActSrc a = {a_q, a_d, nullptr, 0, 0};
    return run_groups<false>(t, tiled, K, N, a, M, y, ldy, s);
}

cudaError_t launch_matvec_fused(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const float *x, int64_t ldx,
                                int64_t M, float *y, int64_t ldy, cudaStream_t s, int x_host) {
    const ActSrc a = {nullptr, nullptr, x, ldx, x_host};
    return run_groups<true>(t, tiled, K, N, a, M, y, ldy, s);
}

cudaError_t launch_matvec_flat(qmm_type t, const uint8_t *flat, int64_t K, int64_t N, const int8_t *a_q,
                               const uint16_t *a_d, int64_t M, float *y, int64_t ldy, cudaStream_t s) {
    const int64_t nkt = K / 32;
    for (int64_t m0 = 0; m0 < M; m0 += kFlatMT) {
        const int mm = (int)((M - m0) < kFlatMT ? (M - m0) : kFlatMT);
        const int8_t *aq = a_q + m0 * K;
        const uint16_t *ad = a_d + m0 * nkt;
        float *yy = y + m0 * ldy;
        cudaError_t e;
        switch (t) {
            case QMM_Q4_0: e = run_flat_mt<QMM_Q4_0>(flat, K, N, aq, ad, mm, yy, ldy, s); break;
            case QMM_IQ4_NL: e = run_flat_mt<QMM_IQ4_NL>(flat, K, N, aq, ad, mm, yy, ldy, s); break;
            case QMM_MXFP4: e = run_flat_mt<QMM_MXFP4>(flat, K, N, aq, ad, mm, yy, ldy, s); break;
            case QMM_Q4_1: e = run_flat_mt<QMM_Q4_1>(flat, K, N, aq, ad, mm, yy, ldy, s); break;
            case QMM_Q4_K: e = run_flat_mt<QMM_Q4_K>(flat, K, N, aq, ad, mm, yy, ldy, s); break;
            default: e = run_flat_mt<QMM_Q8_0>(flat, K, N, aq, ad, mm, yy, ldy, s); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_selftest_wait_mv(unsigned long long limit_ns, int *out, cudaStream_t s) {
    selftest_wait_kernel<<<1, 64, 0, s>>>(limit_ns, out);
    return cudaGetLastError();
}

cudaError_t read_and_clear_matvec_status(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_mv_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_mv_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

QMM_DCHECK_READER(read_dcheck_matvec)

}  // namespace qmm

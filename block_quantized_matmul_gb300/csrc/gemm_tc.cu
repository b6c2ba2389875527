// gemm_tc.cu -- prefill-shaped matmul over 32-row weight tiles on the sm_103a tensor cores (tcgen05).
//
// What it computes ("Hexagon backend developer details", "Tiled Weight Formats"):
//   Y[m, n] = sum_b fp32(d_w[n,b]) * fp32(d_a[m,b]) * S_b[m,n],  S_b = sum_j w_int[n,32b+j] * a_q[m,32b+j]
// The pages' prefill path dequantizes tiles to FP16 in VTCM and feeds the 32x32 HMX array (folding the
// scale into the FP16 value, which rounds).  Here the block sums stay exact:
//   * int8 tcgen05 (kind::i8) does not exist on sm_103a, so quants are expanded to fp16 holding the
//     exact integer (|w| <= 127, |a| <= 127) and contracted with tcgen05.mma.kind::f16; every partial
//     sum of a 32-element block is an integer below 2^24, so the fp32 accumulator in TMEM is exact.
//   * Each block's sums S_b go to their own TMEM slot; the CUDA cores then apply the two scales,
//     y += (S_b * d_a) * d_w, with packed f32x2 multiplies and FMAs in registers (affine tiles, Q4_1
//     and Q4_K: + m_w * (d_a * sum_j a_q), one more FMA).  w_int is q-8 (Q4_0), q (Q8_0, Q4_1),
//     table[q] (IQ4_NL) or twice the FP4 value (MXFP4, with half the E8M0 scale).
//
// Tile: 128 weight rows (4 column tiles, the UMMA M dimension) x 128 tokens (UMMA N), all of K.
// The pipeline moves K in pairs of 32-wide blocks; TMEM holds S of four single blocks (4 x 128
// columns).
// Warp roles (480 threads):
//   warp 0      W producer: per block pair, one 3-D TMA of the 4 x 2 raw weight tiles plus one TMA of
//               the pair's token data (fp16 scales, or the raw int8 rows), into a W ring.
//   warp 1      TMEM owner and MMA issuer (one thread): per block, 2 MMAs (K = 16 each) into a
//               4-slot TMEM ring.
//   warps 2-5   converters: thread c turns weight row c of the pair into fp16 in the canonical K-major
//               128-byte-swizzled layout and writes the pair's fp32 d_w / d_a (and, for int8
//               activations, converts token row c).
//   warps 6-13  rescale: tcgen05.ld of S_b, y += (S_b * d_a) * d_w in registers, then the fp32 store.
//   warp 14     B producer (prepared variant): one 128-byte-swizzled TMA of the fp16 token operand of
//               the pair, straight into the layout the MMA reads.
// Two token-operand variants: int8 quants converted in the kernel (no scratch memory), or a prepared
// fp16 copy in a caller workspace (every token tile is then converted once instead of once per
// weight tile).
// Long K: one launch covers at most kGemmChunkBlocks blocks (K = 4096); longer rows run in passes, each
// adding its partial sums into y in order.  Error: two roundings per block (S_b * d_a, then the FMA)
// along a pass and one per pass add, at most (kGemmChunkBlocks + 2 + n_passes) * 2^-24 *
// sum_k |w_k x_k|: 7.9e-6 at K = 4096, 9.7e-6 at the largest accepted K (131072).
// Every mbarrier wait is bounded in time; on expiry the kernel records QMM_ERR_TIMEOUT in a device
// status word, lets its copies and MMAs in flight land, frees TMEM and returns.
#include <cuda.h>   // CUtensorMap and its enums (the encoder is fetched through the runtime)


#include "pipeline.cuh"
#include "qmm_internal.cuh"
#include "tc_common.cuh"

namespace qmm {

namespace {

__device__ unsigned g_device_status = 0;   // non-zero once a bounded wait gave up

constexpr int BM = 128;                    // weight rows per CTA
constexpr int BN = 128;                    // tokens per CTA
constexpr int kTmemStages = 4;
constexpr int kTmemCols = 512;             // 4 slots x 128 fp32 columns (S of one block each)
constexpr int kConvWarp0 = 2, kNumConvWarps = 4;
constexpr int kRescaleWarp0 = 6, kNumRescaleWarps = 8;
constexpr int kBProducerWarp = kRescaleWarp0 + kNumRescaleWarps;    // warp 14
constexpr int kThreads = (kBProducerWarp + 1) * 32;
constexpr int kOp2Bytes = BM * 128;        // 128 rows x 128 bytes: a block pair (SW128)
constexpr int kLutCopies = 32;          // byte-indexed table copies (one per lane: no bank conflicts)

using namespace pipe;
using namespace tc;

struct GemmParams {
    const uint8_t *tiled;
    const int8_t *a_q;
    const uint16_t *a_d;
    float *y;
    int64_t K, nkt, N, M, ldy;
    int64_t n_col_tiles;
    int kt0, nkc;       // K blocks of this pass: [kt0, kt0 + nkc)
    int accumulate;     // 0: y = result, 1: y += result (passes after the first)
    Lut16 lut;
};

// Bounded wait (pipeline.cuh) reporting to this file's status word.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort,
                                             unsigned long long limit_ns = kWaitLimitNs) {
    return wait_bounded_on(bar, parity, abort, &g_device_status, limit_ns);
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

// Warp-uniform bounded wait: every lane waits, and the warp gives up together if any lane did, so
// the .sync.aligned tcgen05 instructions that follow are always executed by the full warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = wait_bounded(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both K-major, M = 128, N = BN.
constexpr uint32_t kIdesc = idesc_f16(BM, BN);

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    mma_f16_ss(d_tmem, adesc, bdesc, kIdesc, accumulate);
}

// ---------------------------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------------------------
// ACT: how the token operand reaches shared memory.
//   kActInt8      the int8 quants are copied raw (2-D TMA) and converted by the converter warps;
//   kActPrepared  a prepared fp16 copy of the quants (exact integers) is copied by TMA straight into
//                 the 64-byte-swizzled operand layout, and the block scales come transposed
//                 ([K/32][M_pad] fp16), one 256-byte row per block.
enum { kActInt8 = 0, kActPrepared = 1 };

// Shared-memory plan: three decoupled rings whose stages each cover a pair of K blocks.
//   W ring   W producer -> converters: the raw weight tiles [4 column tiles][2 blocks] (one 3-D TMA)
//            and the pair's token data: 2 x 128 fp16 scales (prepared variant) or 128 rows x 64 int8
//            (int8 variant);
//   B ring   B producer -> MMA (prepared variant only): the fp16 token operand of the pair, 128 rows x
//            128 bytes, swizzled by the TMA unit;
//   op ring  converters -> MMA and rescale: A (weights, 128 x 128 B, 128-byte swizzle), for the int8
//            variant B (128 x 128 B), and the pair's fp32 scales d_w[2][128] and d_a[2][128].  A stage
//            is released by the rescale warps once they have applied both blocks' scales (the MMAs
//            that read A and B have completed by then).
template <int TYPE, int ACT>
struct GemmPlan {
    static constexpr bool kPrep = ACT == kActPrepared;
    static constexpr int TS = TileFmt<TYPE>::kBytes;
    static constexpr int kWTiles = 8 * TS;                                   // [4 ct][2 kt] raw tiles
    static constexpr bool kAff = TileFmt<TYPE>::kAffine;                   // Q4_1: + m_w * d_a * sum(a_q)
    // token data of a pair: fp16 scales (+ fp32 d_a * sum(a_q) for Q4_1), or the int8 rows
    static constexpr int kWTok = kPrep ? 2 * BN * 2 + (kAff ? 2 * BN * 4 : 0) : BN * 64;
    static constexpr int kWStageBytes = (kWTiles + kWTok + 127) / 128 * 128;
    // d_w[2][128], d_a[2][128] (+ Q4_1: m_w[2][128], d_a * sum(a_q)[2][128])
    static constexpr int kScaleBytes = (kAff ? 4 : 2) * 2 * 128 * 4;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOp2Bytes;                                  // int8 variant only
    static constexpr int kOffScale = kPrep ? kOp2Bytes : 2 * kOp2Bytes;
    static constexpr int kOpStage = (kOffScale + kScaleBytes + 1023) / 1024 * 1024;
    static constexpr int kOpStages = 3;
    static constexpr int kBStages = kPrep ? 4 : 0;
    static constexpr int kBRing = kBStages > 0 ? kBStages : 1;               // modulus, never 0
    static constexpr int kLutBytes = TileFmt<TYPE>::kLut ? 256 * kLutCopies * 4 : 0;
    static constexpr int kFixed = kOpStages * kOpStage + kBStages * kOp2Bytes + kLutBytes + 1024 + 512;
    static constexpr int kWStagesFit = (227 * 1024 - kFixed) / kWStageBytes;
    static constexpr int kWStages = kWStagesFit > 8 ? 8 : kWStagesFit;
    // byte offsets from the 1024-aligned base
    static constexpr int kOp = 0;
    static constexpr int kB = kOp + kOpStages * kOpStage;
    static constexpr int kW = kB + kBStages * kOp2Bytes;
    static constexpr int kLut = kW + kWStages * kWStageBytes;
    static constexpr int kBars = kLut + kLutBytes;
    static constexpr int kNumBars = 2 * kWStages + 2 * kBStages + 2 * kOpStages + 2 * kTmemStages;
    static constexpr int kEnd = kBars + kNumBars * 8 + 16;
    static constexpr size_t kSmem = 1024 + (size_t)kEnd;
    static_assert(kWStages >= 3, "W ring too shallow");
};

// 15 warps put 4 warps on some SM sub-partitions, whose 16K-register files then allow at most
// 128 registers per thread.
template <int TYPE, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap act_map,
            const __grid_constant__ CUtensorMap da_map, const __grid_constant__ CUtensorMap ca_map) {
    using P = GemmPlan<TYPE, ACT>;
    constexpr int TS = P::TS;
    constexpr int SOFF = TileFmt<TYPE>::kScaleOff;
    constexpr int WS = P::kWStages, BR = P::kBRing, OS = P::kOpStages;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base_u32 & 1023u)) & 1023u);
    uint8_t *op_s = smem + P::kOp;
    uint8_t *b_s = smem + P::kB;
    uint8_t *w_s = smem + P::kW;
    uint32_t *lut_s = reinterpret_cast<uint32_t *>(smem + P::kLut);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::kBars);
    uint64_t *w_full = bars, *w_empty = bars + WS;
    uint64_t *b_full = bars + 2 * WS, *b_empty = b_full + P::kBStages;
    uint64_t *op_full = bars + 2 * WS + 2 * P::kBStages, *op_empty = op_full + OS;
    uint64_t *tm_full = op_empty + OS, *tm_empty = tm_full + kTmemStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tm_empty + kTmemStages);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ct0 = (int64_t)blockIdx.x * 4;
    const int64_t m0 = (int64_t)blockIdx.y * BN;
    const int n_tiles = (int)((p.n_col_tiles - ct0) < 4 ? (p.n_col_tiles - ct0) : 4);
    const int n_tok = (int)((p.M - m0) < BN ? (p.M - m0) : BN);
    const int64_t nkt = p.nkt;                  // row stride of a_d (all K blocks)
    const int nkt32 = p.nkc;                     // blocks of this pass
    const int kt0 = p.kt0;
    const int npairs = (nkt32 + 1) >> 1;

    // ---- set-up: barriers, IQ4_NL table, TMEM ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < WS; ++s) { mbar_init(smem_u32(&w_full[s]), 1); mbar_init(smem_u32(&w_empty[s]), kNumConvWarps * 32); }
        for (int s = 0; s < P::kBStages; ++s) { mbar_init(smem_u32(&b_full[s]), 1); mbar_init(smem_u32(&b_empty[s]), 1); }
        for (int s = 0; s < OS; ++s) {
            mbar_init(smem_u32(&op_full[s]), kNumConvWarps * 32);
            mbar_init(smem_u32(&op_empty[s]), kNumRescaleWarps * 32);
        }
        for (int s = 0; s < kTmemStages; ++s) { mbar_init(smem_u32(&tm_full[s]), 1); mbar_init(smem_u32(&tm_empty[s]), kNumRescaleWarps * 32); }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (TileFmt<TYPE>::kLut) {
        for (int i = threadIdx.x; i < 256 * kLutCopies; i += kThreads) {
            const int b = i / kLutCopies;
            lut_s[i] = h2_bits(__halves2half2(__int2half_rn(p.lut.v[b & 15]), __int2half_rn(p.lut.v[b >> 4])));
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ============================== W producer ==============================
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&w_map)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(P::kPrep ? &da_map : &act_map)) : "memory");
        }
        int issued = 0, s = 0;
        uint32_t ph = 0;
        for (int pr = 0; pr < npairs; ++pr) {
            if (!wait_warp(smem_u32(&w_empty[s]), ph ^ 1u, abort)) break;
            if (lane == 0 && !QMM_DCHECK(s < WS && ct0 < p.n_col_tiles && kt0 + 2 * pr < nkt)) {
                mbar_arrive(smem_u32(&w_full[s]));      // a failed check: skip the copies of this pair
            } else if (lane == 0) {
                const uint32_t fb = smem_u32(&w_full[s]);
                const uint32_t dst = smem_u32(w_s + s * P::kWStageBytes);
                mbar_arrive_expect_tx(fb, (uint32_t)(P::kWTiles + P::kWTok));
                tma_load_3d(dst, &w_map, 0, kt0 + 2 * pr, (int)ct0, fb);
                if constexpr (P::kPrep) {
                    tma_load_2d(dst + P::kWTiles, &da_map, (int)m0, kt0 + 2 * pr, fb);
                    if constexpr (P::kAff) tma_load_2d(dst + P::kWTiles + 2 * BN * 2, &ca_map, (int)m0, kt0 + 2 * pr, fb);
                } else {
                    tma_load_2d(dst + P::kWTiles, &act_map, 32 * kt0 + 64 * pr, (int)m0, fb);
                }
            }
            __syncwarp();
            issued = pr + 1;
            if (++s == WS) { s = 0; ph ^= 1u; }
        }
        // let every copy issued land before the CTA can exit
        for (int i = (issued > WS ? issued - WS : 0); i < issued; ++i)
            wait_drain(smem_u32(&w_full[i % WS]), (uint32_t)((i / WS) & 1));
    } else if (warp == kBProducerWarp) {
        // ============================== B producer ==============================
        if (P::kPrep) {
            int issued = 0, s = 0;
            uint32_t ph = 0;
            for (int pr = 0; pr < npairs; ++pr) {
                if (!wait_warp(smem_u32(&b_empty[s]), ph ^ 1u, abort)) break;
                if (lane == 0) {
                    const uint32_t fb = smem_u32(&b_full[s]);
                    if (QMM_DCHECK(s < BR && kt0 + 2 * pr < nkt && m0 < p.M)) {
                        mbar_arrive_expect_tx(fb, (uint32_t)kOp2Bytes);
                        tma_load_2d(smem_u32(b_s + s * kOp2Bytes), &act_map, 32 * kt0 + 64 * pr, (int)m0, fb);
                    } else {
                        mbar_arrive(fb);
                    }
                }
                __syncwarp();
                issued = pr + 1;
                if (++s == BR) { s = 0; ph ^= 1u; }
            }
            for (int i = (issued > BR ? issued - BR : 0); i < issued; ++i)
                wait_drain(smem_u32(&b_full[i % BR]), (uint32_t)((i / BR) & 1));
        }
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        int committed = 0;
        int os = 0, bs = 0, ts = 0;
        uint32_t oph = 0, bph = 0, tph = 0;
        bool ok = true;
        for (int pr = 0; pr < npairs && ok; ++pr) {
            if (!wait_warp(smem_u32(&op_full[os]), oph, abort)) break;
            if (P::kPrep && !wait_warp(smem_u32(&b_full[bs]), bph, abort)) break;
            const uint32_t op = smem_u32(op_s + os * P::kOpStage);
            const uint32_t bbase = P::kPrep ? smem_u32(b_s + bs * kOp2Bytes) : op + P::kOffB;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (2 * pr + j >= nkt32) break;
                if (!wait_warp(smem_u32(&tm_empty[ts]), tph ^ 1u, abort)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a = op + P::kOffA + 64 * j, b = bbase + 64 * j;
                    const uint32_t d_s = tmem_base + (uint32_t)(ts * BN);
                    mma_f16(d_s, smem_desc_sw128(a), smem_desc_sw128(b), 0u);
                    mma_f16(d_s, smem_desc_sw128(a + 32), smem_desc_sw128(b + 32), 1u);
                    mma_commit(smem_u32(&tm_full[ts]));
                }
                __syncwarp();
                committed += 1;
                if (++ts == kTmemStages) { ts = 0; tph ^= 1u; }
            }
            if (!ok) break;
            if (P::kPrep) {
                if (lane == 0) mma_commit(smem_u32(&b_empty[bs]));
                __syncwarp();
                if (++bs == BR) { bs = 0; bph ^= 1u; }
            }
            if (++os == OS) { os = 0; oph ^= 1u; }
        }
        for (int i = (committed > kTmemStages ? committed - kTmemStages : 0); i < committed; ++i)
            wait_drain(smem_u32(&tm_full[i % kTmemStages]), (uint32_t)((i / kTmemStages) & 1));
    } else if (warp < kRescaleWarp0) {
        // ================================ converters ================================
        // Thread c owns weight row c (tile q = c/32, tile row c%32) and token row c of the pair.
        const int c = threadIdx.x - kConvWarp0 * 32;
        const int q = c >> 5, tr = c & 31;
        const bool w_ok = q < n_tiles;
        const uint32_t *lut_lane = lut_s + (lane & (kLutCopies - 1));
        const bool tok_ok = c < n_tok;
        // int8 variant: block scales of this token, loaded 8 blocks (4 pairs) ahead
        uint16_t da_cur[8], da_nxt[8];
        if (!P::kPrep) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                da_cur[u] = (tok_ok && u < nkt32) ? p.a_d[(m0 + c) * nkt + kt0 + u] : (uint16_t)0;
                da_nxt[u] = (tok_ok && 8 + u < nkt32) ? p.a_d[(m0 + c) * nkt + kt0 + 8 + u] : (uint16_t)0;
            }
        }
        bool ok = true;
        int ws = 0, os = 0;
        uint32_t wph = 0, oph = 0;
        for (int pg = 0; pg < npairs && ok; pg += 4) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int pr = pg + u;
                if (pr >= npairs || !ok) break;
                if (!wait_bounded(smem_u32(&w_full[ws]), wph, abort)) { ok = false; break; }
                if (!wait_bounded(smem_u32(&op_empty[os]), oph ^ 1u, abort)) { ok = false; break; }
                const uint8_t *raw = w_s + ws * P::kWStageBytes;
                uint8_t *op = op_s + os * P::kOpStage;
                float *sc = reinterpret_cast<float *>(op + P::kOffScale);        // [d_w 2][128], [d_a 2][128]
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // -- weight row c of block j: 32 columns -> 16 half2 in column order --
                    uint32_t h[16];
                    float dw = 0.0f, mw = 0.0f;
                    if (w_ok) {
                        const uint8_t *tile = raw + (q * 2 + j) * TS;
                        if constexpr (TYPE == QMM_Q8_0) {
#pragma unroll
                            for (int cp = 0; cp < 16; ++cp) {
                                const uint32_t v = *reinterpret_cast<const uint16_t *>(tile + cp * 64 + 2 * tr);
                                uint32_t lo, hi;
                                i8x4_to_h2x2(v, lo, hi);
                                h[cp] = lo;
                            }
                        } else {
#pragma unroll
                            for (int cp = 0; cp < 16; ++cp) {
                                const uint32_t b = tile[cp * 32 + tr];
                                if constexpr (TYPE == QMM_Q4_0) h[cp] = q4_byte_to_h2<0>(b);
                                else if constexpr (TYPE == QMM_Q4_1) h[cp] = q4_byte_to_h2<0, 0>(b);
                                else h[cp] = lut_lane[b * kLutCopies];
                            }
                        }
                        if constexpr (TileFmt<TYPE>::kE8M0) {
                            dw = mx_half_scale(tile[SOFF + tr]);
                        } else if constexpr (P::kAff) {
                            const __half2 dm = bits_h2(*reinterpret_cast<const uint32_t *>(tile + SOFF + 4 * tr));
                            dw = __low2float(dm);
                            mw = __high2float(dm);
                        } else {
                            dw = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(tile + SOFF + 2 * tr)));
                        }
                    } else {
#pragma unroll
                        for (int cp = 0; cp < 16; ++cp) h[cp] = 0u;
                    }
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
                        *reinterpret_cast<uint4 *>(op + P::kOffA + sw128_off(c, 4 * j + ch)) =
                            make_uint4(h[4 * ch], h[4 * ch + 1], h[4 * ch + 2], h[4 * ch + 3]);
                    sc[j * 128 + c] = dw;
                    if constexpr (P::kAff) sc[512 + j * 128 + c] = mw;
                    // -- token row c of block j --
                    uint16_t da;
                    float ca = 0.0f;                       // Q4_1: d_a * sum(a_q) of the block
                    if constexpr (P::kPrep) {
                        da = *reinterpret_cast<const uint16_t *>(raw + P::kWTiles + 2 * (j * BN + c));
                        if constexpr (P::kAff) ca = *reinterpret_cast<const float *>(raw + P::kWTiles + 2 * BN * 2 + 4 * (j * BN + c));
                    } else {
                        da = da_cur[2 * u + j];
                        const uint4 v0 = *reinterpret_cast<const uint4 *>(raw + P::kWTiles + c * 64 + 32 * j);
                        const uint4 v1 = *reinterpret_cast<const uint4 *>(raw + P::kWTiles + c * 64 + 32 * j + 16);
                        const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            uint32_t a0, a1, a2, a3;
                            i8x4_to_h2x2(wv[2 * ch], a0, a1);
                            i8x4_to_h2x2(wv[2 * ch + 1], a2, a3);
                            *reinterpret_cast<uint4 *>(op + P::kOffB + sw128_off(c, 4 * j + ch)) =
                                make_uint4(a0, a1, a2, a3);
                        }
                        if constexpr (P::kAff) {
                            int asum = 0;
#pragma unroll
                            for (int wi = 0; wi < 8; ++wi) asum = __dp4a((int)wv[wi], 0x01010101, asum);
                            ca = __fmul_rn(__half2float(__ushort_as_half(da)), (float)asum);   // exact (23 bits)
                        }
                    }
                    sc[256 + j * 128 + c] = __half2float(__ushort_as_half(da));
                    if constexpr (P::kAff) sc[768 + j * 128 + c] = ca;
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&op_full[os]));
                mbar_arrive(smem_u32(&w_empty[ws]));
                if (++ws == WS) { ws = 0; wph ^= 1u; }
                if (++os == OS) { os = 0; oph ^= 1u; }
            }
            if (!P::kPrep) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    da_cur[u] = da_nxt[u];
                    const int kn = 2 * pg + 16 + u;
                    da_nxt[u] = (tok_ok && kn < nkt32) ? p.a_d[(m0 + c) * nkt + kt0 + kn] : (uint16_t)0;
                }
            }
        }
    } else {
        // ================================ rescale ================================
        // y[m] += (S_b[n][m] * d_a[m]) * d_w[n] for this thread's weight row n and 64 token columns.
        const int rw = warp - kRescaleWarp0;
        const int qd = warp & 3;                     // TMEM lane quadrant this warp may access
        const int half = rw >> 2;                    // token columns 64*half .. 64*half+63
        const int row = 32 * qd + lane;              // weight row within the tile (= TMEM lane)
        float2 y2[32];                               // token columns (2i, 2i + 1)
#pragma unroll
        for (int i = 0; i < 32; ++i) y2[i] = make_float2(0.0f, 0.0f);
        bool ok = true;
        int ts = 0, os = 0;
        uint32_t tph = 0, oph = 0;
        for (int kt = 0; kt < nkt32; ++kt) {
            const int j = kt & 1;
            if (!wait_warp(smem_u32(&tm_full[ts]), tph, abort)) { ok = false; break; }
            // the pair's scales were written before op_full completed (already complete here)
            if (j == 0 && !wait_warp(smem_u32(&op_full[os]), oph, abort)) { ok = false; break; }
            tc_fence_after();
            const float *sc = reinterpret_cast<const float *>(op_s + os * P::kOpStage + P::kOffScale);
            const float dw = sc[j * 128 + row];
            const float2 dw2 = make_float2(dw, dw);
            const float4 *da4 = reinterpret_cast<const float4 *>(sc + 256 + j * 128 + 64 * half);
            const uint32_t t_s = tmem_base + ((uint32_t)(32 * qd) << 16) + (uint32_t)(ts * BN + 64 * half);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t sv[16];
                tmem_ld16(t_s + 16 * cc, sv);
                float4 da[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) da[e] = da4[4 * cc + e];
                tmem_wait_ld(sv);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 t0 = __fmul2_rn(make_float2(__uint_as_float(sv[4 * e]), __uint_as_float(sv[4 * e + 1])),
                                                 make_float2(da[e].x, da[e].y));
                    const float2 t1 = __fmul2_rn(make_float2(__uint_as_float(sv[4 * e + 2]), __uint_as_float(sv[4 * e + 3])),
                                                 make_float2(da[e].z, da[e].w));
                    y2[8 * cc + 2 * e] = __ffma2_rn(t0, dw2, y2[8 * cc + 2 * e]);
                    y2[8 * cc + 2 * e + 1] = __ffma2_rn(t1, dw2, y2[8 * cc + 2 * e + 1]);
                }
                if constexpr (P::kAff) {
                    // + m_w * (d_a * sum(a_q)) of the block, per token column
                    const float4 *ca4 = reinterpret_cast<const float4 *>(sc + 768 + j * 128 + 64 * half);
                    const float2 mw2 = make_float2(sc[512 + j * 128 + row], sc[512 + j * 128 + row]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 ca = ca4[4 * cc + e];
                        y2[8 * cc + 2 * e] = __ffma2_rn(make_float2(ca.x, ca.y), mw2, y2[8 * cc + 2 * e]);
                        y2[8 * cc + 2 * e + 1] = __ffma2_rn(make_float2(ca.z, ca.w), mw2, y2[8 * cc + 2 * e + 1]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tm_empty[ts]));
            if (++ts == kTmemStages) { ts = 0; tph ^= 1u; }
            if (j == 1 || kt + 1 == nkt32) {
                // both blocks of the pair applied: the operand stage (A, B and the scales) is free
                mbar_arrive(smem_u32(&op_empty[os]));
                if (++os == OS) { os = 0; oph ^= 1u; }
            }
        }
        if (ok) {
            const int64_t n = (ct0 * 32) + row;
            if (n < p.N) {
                if (!p.accumulate) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int64_t m = m0 + 64 * half + i;
                        if (m < p.M) p.y[m * p.ldy + n] = (i & 1) ? y2[i >> 1].y : y2[i >> 1].x;
                    }
                } else {
                    // a later K pass adds its partial sums into y
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int64_t m = m0 + 64 * half + i;
                        if (m < p.M) p.y[m * p.ldy + n] = __fadd_rn(p.y[m * p.ldy + n], (i & 1) ? y2[i >> 1].y : y2[i >> 1].x);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
    }
}

// Prepares the token operand for kActPrepared: a_h[m][k] = fp16(a_q[m][k]) (exact),
// a_dT[kt][m] = a_d[m][kt] for m < M_pad (zero for m >= M) and, if cA is given (Q4_1),
// cA[kt][m] = fp32(a_d[m][kt]) * sum_j a_q[m][32kt + j] (exact: at most 23 significant bits).
__global__ void __launch_bounds__(256) prepare_act_kernel(const int8_t *__restrict__ a_q, const uint16_t *__restrict__ a_d,
                                                          int64_t M, int64_t K, int64_t M_pad, __half *__restrict__ a_h,
                                                          uint16_t *__restrict__ a_dT, float *__restrict__ cA) {
    const int64_t nkt = K / 32;
    const int64_t quads = M * K / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < quads; i += stride) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(a_q) + i);
        uint32_t lo, hi;
        const uint32_t x = w ^ 0x80808080u;
        const __half2 bias = __halves2half2(__float2half_rn(1152.0f), __float2half_rn(1152.0f));
        lo = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x4140u)), bias));
        hi = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x4342u)), bias));
        reinterpret_cast<uint2 *>(a_h)[i] = make_uint2(lo, hi);
    }
    const int64_t nd = nkt * M_pad;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nd; i += stride) {
        const int64_t kt = i / M_pad, m = i - kt * M_pad;
        a_dT[i] = (m < M) ? a_d[m * nkt + kt] : (uint16_t)0;
        if (cA) {
            float v = 0.0f;
            if (m < M) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a_q + m * K + kt * 32);
                const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
                int asum = 0;
                asum = __dp4a((int)v0.x, 0x01010101, asum); asum = __dp4a((int)v0.y, 0x01010101, asum);
                asum = __dp4a((int)v0.z, 0x01010101, asum); asum = __dp4a((int)v0.w, 0x01010101, asum);
                asum = __dp4a((int)v1.x, 0x01010101, asum); asum = __dp4a((int)v1.y, 0x01010101, asum);
                asum = __dp4a((int)v1.z, 0x01010101, asum); asum = __dp4a((int)v1.w, 0x01010101, asum);
                v = __fmul_rn(__half2float(__ushort_as_half(a_d[m * nkt + kt])), (float)asum);
            }
            cA[i] = v;
        }
    }
}

}  // namespace

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (thread-safe static initialization).
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return nullptr;
    }();
    return fn;
}

// 2-D tensor map: rows of `inner` elements (row stride `row_bytes`), box {box_inner, box_rows}.
cudaError_t make_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D tensor map of the tiled weight viewed as [n_col_tiles][n_k_tiles][tile bytes / 8] of 8-byte
// words: one box = the 4 column tiles x 2 K tiles of a block pair (column tiles past the end read
// as zeros).
cudaError_t make_weight_map(CUtensorMap *map, const uint8_t *tiled, int tile_bytes, int64_t nkt, int64_t nct) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)(tile_bytes / 8), (cuuint64_t)nkt, (cuuint64_t)nct};
    const cuuint64_t strides[2] = {(cuuint64_t)tile_bytes, (cuuint64_t)nkt * (cuuint64_t)tile_bytes};
    const cuuint32_t box[3] = {(cuuint32_t)(tile_bytes / 8), 2, 4};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t *>(tiled), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

template <int TYPE, int ACT>
cudaError_t launch_typed(const GemmParams &p, const CUtensorMap &act_map, const CUtensorMap &da_map, const CUtensorMap &ca_map,
                         cudaStream_t s) {
    using P = GemmPlan<TYPE, ACT>;
    static_assert(P::kSmem <= 227 * 1024, "shared memory plan too large");
    auto kern = gemm_kernel<TYPE, ACT>;
    static int attr_done[4] = {0, 0, 0, 0};
    cudaError_t e = ensure_smem_limit(kern, P::kSmem, attr_done);
    if (e != cudaSuccess) return e;
    alignas(64) CUtensorMap w_map;
    e = make_weight_map(&w_map, p.tiled, P::TS, p.nkt, p.n_col_tiles);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((p.n_col_tiles + 3) / 4), (unsigned)((p.M + BN - 1) / BN), 1);
    // K in passes of at most kGemmChunkBlocks blocks, each adding into y in order (the error bound)
    for (int kt0 = 0; kt0 < (int)p.nkt; kt0 += kGemmChunkBlocks) {
        GemmParams q = p;
        q.kt0 = kt0;
        q.nkc = (int)p.nkt - kt0 < kGemmChunkBlocks ? (int)p.nkt - kt0 : kGemmChunkBlocks;
        q.accumulate = kt0 > 0;
        kern<<<grid, kThreads, P::kSmem, s>>>(q, w_map, act_map, da_map, ca_map);
        const cudaError_t le = cudaGetLastError();
        if (le != cudaSuccess) return le;
    }
    return cudaSuccess;
}

template <int ACT>
cudaError_t dispatch(qmm_type t, const GemmParams &p, const CUtensorMap &am, const CUtensorMap &dm, const CUtensorMap &cm,
                     cudaStream_t s) {
    switch (t) {
        case QMM_Q4_0: return launch_typed<QMM_Q4_0, ACT>(p, am, dm, cm, s);
        case QMM_IQ4_NL: return launch_typed<QMM_IQ4_NL, ACT>(p, am, dm, cm, s);
        case QMM_MXFP4: return launch_typed<QMM_MXFP4, ACT>(p, am, dm, cm, s);
        case QMM_Q4_1: return launch_typed<QMM_Q4_1, ACT>(p, am, dm, cm, s);
        default: return launch_typed<QMM_Q8_0, ACT>(p, am, dm, cm, s);
    }
}

GemmParams make_params(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                       int64_t M, float *y, int64_t ldy) {
    GemmParams p;
    p.tiled = tiled;
    p.a_q = a_q;
    p.a_d = a_d;
    p.y = y;
    p.K = K;
    p.nkt = K / 32;
    p.N = N;
    p.M = M;
    p.ldy = ldy;
    p.n_col_tiles = (N + 31) / 32;
    p.kt0 = 0;
    p.nkc = (int)p.nkt;
    p.accumulate = 0;
    p.lut = lut_for(t);
    return p;
}

}  // namespace

cudaError_t launch_gemm(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                        int64_t M, float *y, int64_t ldy, cudaStream_t s) {
    if ((M + BN - 1) / BN > 65535) return cudaErrorInvalidValue;
    const GemmParams p = make_params(t, tiled, K, N, a_q, a_d, M, y, ldy);
    alignas(64) CUtensorMap am, dm;
    cudaError_t e = make_map_2d(&am, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_q, (uint64_t)K, (uint64_t)M, (uint64_t)K, 64, BN,
                                CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    dm = am;   // unused by this variant
    return dispatch<kActInt8>(t, p, am, dm, am, s);
}

size_t gemm_workspace_bytes(int64_t M, int64_t K) { return gemm_ws_layout(M, K).total; }

cudaError_t launch_gemm_ws(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                           const uint16_t *a_d, int64_t M, float *y, int64_t ldy, void *ws, cudaStream_t s) {
    if ((M + BN - 1) / BN > 65535) return cudaErrorInvalidValue;
    const int64_t nkt = K / 32, m_pad = (M + 7) / 8 * 8;
    const GemmWsLayout L = gemm_ws_layout(M, K);
    __half *a_h = reinterpret_cast<__half *>(static_cast<uint8_t *>(ws) + L.hi);
    uint16_t *a_dT = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + L.dT);
    float *cA = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + L.cA);
    const bool need_ca = t == QMM_Q4_1;
    {
        const int64_t work = M * K / 4 > nkt * m_pad ? M * K / 4 : nkt * m_pad;
        int64_t grid = (work + 255) / 256;
        if (grid > 152 * 8) grid = 152 * 8;
        prepare_act_kernel<<<(unsigned)grid, 256, 0, s>>>(a_q, a_d, M, K, m_pad, a_h, a_dT, need_ca ? cA : nullptr);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const GemmParams p = make_params(t, tiled, K, N, a_q, a_d, M, y, ldy);
    alignas(64) CUtensorMap am, dm;
    cudaError_t e = make_map_2d(&am, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a_h, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64,
                                BN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = make_map_2d(&dm, CU_TENSOR_MAP_DATA_TYPE_UINT16, a_dT, (uint64_t)m_pad, (uint64_t)nkt, (uint64_t)m_pad * 2, BN, 2,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    alignas(64) CUtensorMap cm = dm;
    if (need_ca) {
        e = make_map_2d(&cm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cA, (uint64_t)m_pad, (uint64_t)nkt, (uint64_t)m_pad * 4, BN, 2,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
        if (e != cudaSuccess) return e;
    }
    return dispatch<kActPrepared>(t, p, am, dm, cm, s);
}

// ---------------------------------------------------------------------------------------------
// No-allocation variant of the workspace path.
// Some callers cannot allocate device memory: code running under a custom allocator or memory pool
// that must not see foreign allocations, inference runtimes that pre-plan every byte of device
// memory, or programs that must not touch the CUDA allocator in a latency-critical section.  For
// them the workspace lives in this fixed, file-scope device array instead of a caller buffer.  The
// array exists once per device for as long as the library stays loaded; its contents persist from
// call to call, and calls that overlap on the GPU share (and race on) it.
// ---------------------------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context.  The host-side symbol is only a
// stand-in for the device variable, and the module (with the array) is loaded again after a device
// reset, so the address is looked up on every call rather than cached.
cudaError_t noalloc_scratch(void **out) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = ptr;
    return cudaSuccess;
}

cudaError_t launch_selftest_wait_gemm(unsigned long long limit_ns, int *out, cudaStream_t s) {
    selftest_wait_kernel<<<1, 64, 0, s>>>(limit_ns, out);
    return cudaGetLastError();
}

cudaError_t read_and_clear_device_status(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_device_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

QMM_DCHECK_READER(read_dcheck_gemm)

}  // namespace qmm

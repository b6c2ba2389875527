// gemm_fold.cu -- prefill-shaped matmul over 32-row weight tiles with the block scales folded into the
// tensor-core operands (sm_103a, tcgen05).
//
// What it computes ("Hexagon backend developer details", "Tiled Weight Formats"):
//   Y[m, n] = sum_k a[m, k] * w[n, k],  a = d_a * q_a (the Q8_0 activation),  w = d_w * w_int,
// with the pages' dequantized weight w_int = q - 8 (Q4_0), q (Q8_0) or table[q] (IQ4_NL).  This is the
// block formula sum_b d_w d_a S_b summed element by element instead of block by block.  The pages'
// prefill path also dequantizes to FP16 and contracts on the matrix unit, but rounds d*q to FP16 once.
// Here no operand value is rounded:
//   * an fp16 scale times an integer code of at most 8 bits has at most 19 significant bits and is a
//     multiple of 2^-24, so it splits exactly into two fp16 numbers v = hi + lo, hi = fp16(v) and
//     lo = fma(d, q, -hi) (the fma is exact because v - hi is representable);
//   * Y = sum a_hi w_hi + a_hi w_lo + a_lo w_hi: three fp16 MMAs per K step; the dropped a_lo w_lo is
//     below 2^-22 |a w|;
//   * the fp32 accumulator in tensor memory takes a chunk of kChunkPairs = 2 block pairs (128 K) at a
//     time, and the CUDA cores add the chunk sums in fp32.  A host model of this order (each MMA
//     step's product sum exact and rounded once into the accumulator, 24 steps per chunk, one rounding
//     per chunk sum) puts the error below 5e-6 of sum_k |a w| for K up to 4096.  That figure is a
//     modelled estimate: the tensor cores' internal accumulation order is not documented.  The GPU
//     parity tests on all-positive operands (the worst case for cancellation-free growth) measure it.
//   * the host launches K in passes of at most kGemmChunkBlocks blocks (K = 4096); a pass after the first
//     adds its result into y, which adds one fp32 rounding per pass to the bound.
// Compared with the exact-integer kernel (gemm_tc.cu), the tensor cores do three times the MACs but
// the per-block fp32 rescale of every output (two CUDA-core operations per output and block, which
// made that kernel issue-bound) is gone: what is left for the CUDA cores is the weight split (once
// per weight element and token tile) and one fp32 add per output and chunk.  The token operand is
// split once per call by prepare_fold_act_kernel into the caller's workspace (a_hi, a_lo, and the
// per-row power of two); the GEMM is its programmatic dependent and overlaps it with its set-up.
//
// Ranges.  hi must stay finite.  A weight row whose largest |d_w| * max|w_int| reaches 2^15 (and a
// token row whose largest |d_a| * 127 does) is scaled by a power of two 2^-t before the split, and its
// outputs by 2^t after the sum.  That is exact unless a scaled-down block scale d * 2^-t of that row
// loses bits, i.e. falls below fp16's normal range (d * 2^-t < 2^-14): with t about
// log2(max d * qmax) - 14, a row whose block scales span more than about 2^28 / qmax (2^21 for
// qmax = 127, 2^25 for Q4_0's 8).  Both sides check every scaled scale for that (the token rows when
// they are prepared, the weight rows when the workers scale them) and report a row that fails as
// QMM_ERR_RANGE through qmm_device_status, after which the caller can run the call again on the
// exact-integer kernel (qmm_matmul_path with QMM_PATH_GEMM).
//
// Tile: 128 weight rows (4 column tiles, the UMMA M) x 128 tokens (UMMA N), all of K.  K moves in
// pairs of 32-wide blocks; a chunk is two pairs.
// Warp roles (352 threads):
//   warp 0      W producer: per pair, one 3-D TMA of the 4 x 2 raw weight tiles into the W ring.
//   warp 1      TMEM owner; one thread issues the MMAs: per pair 12 (K = 16, three products, two
//               blocks) with A (weights) from tensor memory and B (tokens) from shared memory, then
//               one commit that frees the pair's weight slots and token stage (and, after the last
//               pair of a chunk, hands the accumulator to the workers).
//   warp 2      B producer: per pair, two 128-byte-swizzled TMAs of the prepared token operand (hi and
//               lo, fp16) straight into the layout the MMA reads (lane 0); lane 1 waits for each
//               copy and adds its arrival to the pair's ready barrier, so the MMA thread waits on
//               one barrier per pair.
//   warps 3-10  workers, two per tensor-memory lane quadrant (h = 0, 1): worker h of quadrant q splits
//               block h of every pair for weight rows 32q..32q+31 into hi and lo fp16 and stores both
//               into the pair's tensor-memory slot (the A operand); after the last pair of chunk c + 1
//               it adds chunk c's sums for token columns 64h..64h+63 into registers; at the end it
//               stores y.
// Tensor memory (512 columns): two accumulator slots of 128 columns (chunk c in slot c % 2), then
// eight weight-block slots of 32 columns (hi: 16, lo: 16; two fp16 K values per column), block k in
// slot k % 8.
// Every mbarrier wait is bounded in time; on expiry the kernel records QMM_ERR_TIMEOUT in its
// device status word, lets its copies and MMAs in flight land, frees TMEM and returns.
#include <cuda.h>

#include "pipeline.cuh"
#include "qmm_internal.cuh"
#include "tc_common.cuh"

namespace qmm {

namespace {

__device__ unsigned g_fold_status = 0;     // bit 0: a bounded wait gave up; bit 1: an operand row not exact
constexpr unsigned kFoldStatusRange = 2u;

constexpr int FM = 128;                    // weight rows per CTA (UMMA M)
constexpr int FN = 128;                    // tokens per CTA (UMMA N)
constexpr int kChunkPairs = 2;             // pairs of K blocks summed in tensor memory before the fp32 add
constexpr int kAccSlots = 2;
constexpr int kPairSlots = 4;              // pairs in flight: weight slots in tensor memory, token stages
constexpr int kWCol0 = kAccSlots * FN;     // first column of the weight slots
constexpr int kTmemCols = 512;
constexpr int kWorker0 = 3, kNumWorkers = 8;
constexpr int kThreads = (kWorker0 + kNumWorkers) * 32;
constexpr int kWorkerThreads = kNumWorkers * 32;
constexpr int kTokBytes = FN * 128;        // one fp16 token operand of a block pair: 128 rows x 128 B
constexpr int kBStageBytes = 2 * kTokBytes;   // hi, then lo
constexpr int kLutCopies = 32;             // byte-indexed table copies (one per lane)
constexpr uint32_t kIdescF = tc::idesc_f16(FM, FN);
static_assert(kWCol0 + 2 * 32 * kPairSlots == kTmemCols, "tensor-memory plan");

using namespace pipe;
using namespace tc;

struct FoldParams {
    const uint8_t *tiled;
    const float *tscale;                   // per token: 2^s, the power of two its row was scaled by
    float *y;
    int64_t N, M, ldy, n_col_tiles;
    int nkt;            // K blocks of the whole row (stride of the weight tiles)
    int kt0, nkc;       // K blocks of this pass: [kt0, kt0 + nkc)
    int accumulate;     // 0: y = result, 1: y += result (passes after the first)
    Lut16 lut;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort) {
    return wait_bounded_on(bar, parity, abort, &g_fold_status, kWaitLimitNs);
}
// Warp-uniform bounded wait: the warp gives up together, so the .sync.aligned tcgen05 instructions
// that follow are always executed by the full warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = wait_bounded(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Runs this file's bounded wait out on purpose (the failure-detection test): warp 0 waits, with
// limit_ns, for a barrier phase that nothing completes; warp 1 waits for the same phase with the
// normal limit and must give up once warp 0 has raised the abort flag.  out[w] = 1 if warp w's wait
// returned true (neither should); the status word is set as by any timed-out wait of this kernel.
__global__ void __launch_bounds__(64) selftest_wait_fold_kernel(unsigned long long limit_ns, int *out) {
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
    const bool ok = wait_bounded_on(smem_u32(&bar), 0u, abort, &g_fold_status, warp == 0 ? limit_ns : kWaitLimitNs);
    if ((threadIdx.x & 31) == 0) out[warp] = ok ? 1 : 0;
}

// 2^k as an exact fp32 (k within the normal exponent range).
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }

// Power-of-two shift t >= 0 with v * 2^-t < 2^15 (v >= 0 finite): 0 unless v >= 2^15.
__device__ __forceinline__ int range_shift(float v) {
    if (!(v >= 32768.0f)) return 0;
    const int e = (int)((__float_as_uint(v) >> 23) & 0xFFu) - 127;   // floor(log2 v), v normal
    return e - 14;
}

// hi and lo of d * v for the two fp16 lanes of v (exact split, see the file header).
__device__ __forceinline__ void split2(uint32_t v, __half2 d2, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __hmul2_rn(bits_h2(v), d2);
    hi = h2_bits(h);
    lo = h2_bits(__hfma2(bits_h2(v), d2, __hneg2(h)));
}

// Range of weight row 32 * q + lane (q = warp % 4): the largest |d_w| over all of K.  The two workers
// of a lane quadrant each scan every other K tile (up to 64 loads in flight per thread), combine by an
// atomic max in shared memory and meet at named barrier 1 (all workers).  Once a thread's first loads
// are issued it arrives on `issued`: the producers hold their first copies until then, so these few
// loads are not queued behind the CTA's opening burst of tile copies.  Returns the row's
// power-of-two shift t (0 unless |d_w| * max|w_int| reaches 2^15).
template <int TYPE>
__device__ __forceinline__ int weight_row_shift(const FoldParams &p, unsigned *row_max, int64_t ct0, int qd, int part,
                                                int lane, uint64_t *issued) {
    constexpr int TS = TileFmt<TYPE>::kBytes;
    constexpr float kWMax = TYPE == QMM_Q4_0 ? 8.0f : 128.0f;   // largest |w_int| (IQ4_NL's table: 127)
    const int row = 32 * qd + lane;
    const int64_t ct = ct0 + qd;
    const int nkt = p.nkc;
    bool signalled = false;
    if (ct < p.n_col_tiles) {
        const uint8_t *sp = p.tiled + ((size_t)ct * (size_t)p.nkt + (size_t)p.kt0) * TS + TileFmt<TYPE>::kScaleOff + 2 * lane;
        float dmax = 0.0f;
        for (int k0 = part; k0 < nkt; k0 += 2 * 64) {
            unsigned short v[64];
#pragma unroll
            for (int u = 0; u < 64; ++u) {
                const int kt = k0 + 2 * u;
                v[u] = kt < nkt ? __ldg(reinterpret_cast<const unsigned short *>(sp + (size_t)kt * TS)) : (unsigned short)0;
            }
            if (!signalled) {
                mbar_arrive(smem_u32(issued));               // ordered after the loads above ("memory")
                signalled = true;
            }
#pragma unroll
            for (int u = 0; u < 64; ++u) dmax = fmaxf(dmax, fabsf(__half2float(__ushort_as_half(v[u]))));
        }
        atomicMax(&row_max[row], __float_as_uint(dmax));     // non-negative floats order as their bits
    }
    if (!signalled) mbar_arrive(smem_u32(issued));
    asm volatile("bar.sync 1, %0;" ::"r"(kWorkerThreads) : "memory");
    return range_shift(__uint_as_float(row_max[row]) * kWMax);
}

// Shared-memory plan (1024-aligned base):
//   B ring   B producer -> MMA: the pair's token operand, hi then lo, 128 rows x 128 B each (SW128);
//   W ring   W producer -> workers: the raw weight tiles [4 column tiles][2 blocks];
//   table    IQ4_NL byte -> half2 table, one copy per lane;
//   the weight rows' largest |d_w| (fp32 bits), then the mbarriers.
template <int TYPE>
struct FoldPlan {
    static constexpr int TS = TileFmt<TYPE>::kBytes;
    static constexpr int kWTiles = 8 * TS;
    static constexpr int kWStageBytes = (kWTiles + 127) / 128 * 128;
    static constexpr int kLutBytes = TileFmt<TYPE>::kLut ? 256 * kLutCopies * 4 : 0;
    static constexpr int kB = 0;
    static constexpr int kW = kB + kPairSlots * kBStageBytes;
    static constexpr int kFixed = kW + kLutBytes + 1024 + 2048;
    static constexpr int kWStagesFit = (227 * 1024 - kFixed) / kWStageBytes;
    static constexpr int kWStages = kWStagesFit > 8 ? 8 : kWStagesFit;
    static constexpr int kLut = kW + kWStages * kWStageBytes;
    static constexpr int kRowMax = kLut + kLutBytes;
    static constexpr int kBars = kRowMax + FM * 4;
    static constexpr int kNumBars = 2 * kWStages + 3 * kPairSlots + kAccSlots + 2;
    static constexpr int kEnd = kBars + kNumBars * 8 + 16;
    static constexpr size_t kSmem = 1024 + (size_t)kEnd;
    static_assert(kWStages >= 4, "W ring too shallow");
};

template <int TYPE>
__global__ void __launch_bounds__(kThreads, 1)
gemm_fold_kernel(const FoldParams p, const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap ah_map,
                 const __grid_constant__ CUtensorMap al_map) {
    using P = FoldPlan<TYPE>;
    constexpr int TS = P::TS;
    constexpr int SOFF = TileFmt<TYPE>::kScaleOff;
    constexpr int WS = P::kWStages;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base_u32 & 1023u)) & 1023u);
    uint8_t *b_s = smem + P::kB;
    uint8_t *w_s = smem + P::kW;
    uint32_t *lut_s = reinterpret_cast<uint32_t *>(smem + P::kLut);
    unsigned *row_max = reinterpret_cast<unsigned *>(smem + P::kRowMax);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::kBars);
    uint64_t *w_full = bars, *w_empty = bars + WS;
    uint64_t *b_full = bars + 2 * WS;                  // token stage of pair p landed (TMA)
    uint64_t *pair_ready = b_full + kPairSlots;        // weight blocks of pair p in tensor memory (workers)
    uint64_t *pair_done = pair_ready + kPairSlots;     // MMAs of pair p complete (commit)
    uint64_t *acc_empty = pair_done + kPairSlots;
    uint64_t *mma_done = acc_empty + kAccSlots;
    uint64_t *scan_issued = mma_done + 1;              // every worker has issued its first scale loads
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(scan_issued + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ct0 = (int64_t)blockIdx.x * 4;
    const int64_t m0 = (int64_t)blockIdx.y * FN;
    const int nkt = p.nkc;                    // blocks of this pass
    const int kt0 = p.kt0;
    const int npairs = (nkt + 1) >> 1;
    const int nchunks = (npairs + kChunkPairs - 1) / kChunkPairs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WS; ++s) { mbar_init(smem_u32(&w_full[s]), 1); mbar_init(smem_u32(&w_empty[s]), kWorkerThreads); }
        for (int s = 0; s < kPairSlots; ++s) {
            mbar_init(smem_u32(&b_full[s]), 1);
            mbar_init(smem_u32(&pair_ready[s]), kWorkerThreads + 1);
            mbar_init(smem_u32(&pair_done[s]), 1);
        }
        for (int s = 0; s < kAccSlots; ++s) mbar_init(smem_u32(&acc_empty[s]), kWorkerThreads);
        mbar_init(smem_u32(mma_done), 1);
        mbar_init(smem_u32(scan_issued), kWorkerThreads);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (TileFmt<TYPE>::kLut) {
        for (int i = threadIdx.x; i < 256 * kLutCopies; i += kThreads) {
            const int b = i / kLutCopies;
            lut_s[i] = h2_bits(__halves2half2(__int2half_rn(p.lut.v[b & 15]), __int2half_rn(p.lut.v[b >> 4])));
        }
    }
    if (threadIdx.x < FM) row_max[threadIdx.x] = 0u;
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
            int issued = 0;
            wait_bounded(smem_u32(scan_issued), 0u, abort);
            for (int pr = 0; pr < npairs; ++pr) {
                const int s = pr % WS;
                if (!wait_bounded(smem_u32(&w_empty[s]), (uint32_t)(((pr / WS) & 1) ^ 1), abort)) break;
                const uint32_t fb = smem_u32(&w_full[s]);
                if (QMM_DCHECK(s < WS && ct0 < p.n_col_tiles && kt0 + 2 * pr < p.nkt)) {
                    mbar_arrive_expect_tx(fb, (uint32_t)P::kWTiles);
                    tma_load_3d(smem_u32(w_s + s * P::kWStageBytes), &w_map, 0, kt0 + 2 * pr, (int)ct0, fb);
                } else {
                    mbar_arrive(fb);
                }
                issued = pr + 1;
            }
            for (int i = (issued > WS ? issued - WS : 0); i < issued; ++i)
                wait_drain(smem_u32(&w_full[i % WS]), (uint32_t)((i / WS) & 1));
        }
    } else if (warp == 2) {
        // ============================== B producer ==============================
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ah_map)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&al_map)) : "memory");
            // launched as a programmatic dependent of the token preparation: its output is read from here on
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int issued = 0;
            wait_bounded(smem_u32(scan_issued), 0u, abort);
            for (int pr = 0; pr < npairs; ++pr) {
                const int s = pr % kPairSlots;
                // the stage is free once the MMAs of pair pr - kPairSlots have completed
                if (!wait_bounded(smem_u32(&pair_done[s]), (uint32_t)(((pr / kPairSlots) & 1) ^ 1), abort)) break;
                const uint32_t fb = smem_u32(&b_full[s]);
                const uint32_t dst = smem_u32(b_s + s * kBStageBytes);
                if (QMM_DCHECK(s < kPairSlots && kt0 + 2 * pr < p.nkt && m0 < p.M)) {
                    mbar_arrive_expect_tx(fb, (uint32_t)kBStageBytes);
                    tma_load_2d(dst, &ah_map, 32 * kt0 + 64 * pr, (int)m0, fb);
                    tma_load_2d(dst + kTokBytes, &al_map, 32 * kt0 + 64 * pr, (int)m0, fb);
                } else {
                    mbar_arrive(fb);
                }
                issued = pr + 1;
            }
            for (int i = (issued > kPairSlots ? issued - kPairSlots : 0); i < issued; ++i)
                wait_drain(smem_u32(&b_full[i % kPairSlots]), (uint32_t)((i / kPairSlots) & 1));
        } else if (lane == 1) {
            // relay: token stage of pair pr landed -> one arrival on pair_ready (the workers add theirs)
            for (int pr = 0; pr < npairs; ++pr) {
                const int s = pr % kPairSlots;
                if (!wait_bounded(smem_u32(&b_full[s]), (uint32_t)((pr / kPairSlots) & 1), abort)) break;
                mbar_arrive(smem_u32(&pair_ready[s]));
            }
        }
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        if (lane == 0) {
            for (int pr = 0; pr < npairs; ++pr) {
                const int s = pr % kPairSlots;
                const uint32_t ph = (uint32_t)((pr / kPairSlots) & 1);
                const int c = pr / kChunkPairs, as = c % kAccSlots;
                const bool chunk_first = (pr % kChunkPairs) == 0;
                if (!wait_bounded(smem_u32(&pair_ready[s]), ph, abort)) break;
                if (chunk_first && !wait_bounded(smem_u32(&acc_empty[as]), (uint32_t)(((c / kAccSlots) & 1) ^ 1), abort))
                    break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(as * FN);
                const uint32_t bh0 = smem_u32(b_s + s * kBStageBytes);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int kt = 2 * pr + j;
                    if (kt >= nkt) break;
                    const uint32_t a_hi = tmem_base + (uint32_t)(kWCol0 + 32 * (kt % (2 * kPairSlots))), a_lo = a_hi + 16;
                    const uint32_t bh = bh0 + 64 * j, bl = bh + kTokBytes;
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        const uint32_t acc = (chunk_first && j == 0 && kh == 0) ? 0u : 1u;
                        mma_f16_ts(d, a_hi + 8 * kh, smem_desc_sw128(bh + 32 * kh), kIdescF, acc);
                        mma_f16_ts(d, a_hi + 8 * kh, smem_desc_sw128(bl + 32 * kh), kIdescF, 1u);
                        mma_f16_ts(d, a_lo + 8 * kh, smem_desc_sw128(bh + 32 * kh), kIdescF, 1u);
                    }
                }
                mma_commit(smem_u32(&pair_done[s]));
            }
            // every MMA issued has completed before tensor memory is released
            mma_commit(smem_u32(mma_done));
            wait_drain(smem_u32(mma_done), 0u);
        }
        __syncwarp();
    } else {
        // ================================== workers ==================================
        const int qd = warp & 3;                              // tensor-memory lane quadrant this warp may access
        const int h = (warp - kWorker0) >> 2;                 // block of each pair, and token-column half
        const int row = 32 * qd + lane;                       // weight row within the tile (= TMEM lane)
        const int t = weight_row_shift<TYPE>(p, row_max, ct0, qd, h, lane, scan_issued);
        const float down = exp2i(-t);
        const uint32_t *lut_lane = lut_s + lane;
        const uint32_t t_lane = tmem_base + ((uint32_t)(32 * qd) << 16);
        float2 y2[32];                                        // token columns (2i, 2i + 1) of this half
#pragma unroll
        for (int i = 0; i < 32; ++i) y2[i] = make_float2(0.0f, 0.0f);

        // adds chunk c's sums of this thread's row and 64 token columns into y2; the chunk is complete
        // once the MMAs of its last pair are (the commit of a pair covers every MMA issued before it)
        auto drain = [&](int c) -> bool {
            const int as = c % kAccSlots;
            const int last = (c + 1) * kChunkPairs - 1 < npairs - 1 ? (c + 1) * kChunkPairs - 1 : npairs - 1;
            if (!wait_warp(smem_u32(&pair_done[last % kPairSlots]), (uint32_t)((last / kPairSlots) & 1), abort)) return false;
            tc_fence_after();
            const uint32_t ta = t_lane + (uint32_t)(as * FN + 64 * h);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t sv[16];
                tmem_ld16(ta + 16 * cc, sv);
                tmem_wait_ld(sv);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    y2[8 * cc + e] = __fadd2_rn(y2[8 * cc + e], make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])));
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&acc_empty[as]));
            return true;
        };

        bool ok = true;
        int pend = -1;                                        // pair whose stores are still in flight
        int drained = 0;
        for (int pr = 0; pr < npairs && ok; ++pr) {
            const int s = pr % kPairSlots;
            if (!wait_warp(smem_u32(&w_full[pr % WS]), (uint32_t)((pr / WS) & 1), abort)) { ok = false; break; }
            // this pair's weight slots are free once the MMAs of pair pr - kPairSlots have completed
            if (!wait_warp(smem_u32(&pair_done[s]), (uint32_t)(((pr / kPairSlots) & 1) ^ 1), abort)) { ok = false; break; }
            tc_fence_after();
            const int kt = 2 * pr + h;
            uint32_t hi[16], lo[16];
            if (kt < nkt) {
                const uint8_t *tile = w_s + (pr % WS) * P::kWStageBytes + (qd * 2 + h) * TS;
                __half d = __ushort_as_half(*reinterpret_cast<const uint16_t *>(tile + SOFF + 2 * lane));
                if (t != 0) {
                    const float d0 = __half2float(d);
                    d = __float2half_rn(d0 * down);
                    // a scale that does not survive the shift exactly: this call's result is not exact
                    if (__half2float(d) * exp2i(t) != d0) atomicOr(&g_fold_status, kFoldStatusRange);
                }
                const __half2 d2 = __half2half2(d);
#pragma unroll
                for (int cp = 0; cp < 16; ++cp) {
                    uint32_t v;
                    if constexpr (TYPE == QMM_Q8_0) {
                        uint32_t vh;
                        i8x4_to_h2x2(*reinterpret_cast<const uint16_t *>(tile + cp * 64 + 2 * lane), v, vh);
                    } else if constexpr (TYPE == QMM_Q4_0) {
                        v = q4_byte_to_h2<0>(tile[cp * 32 + lane]);
                    } else {
                        v = lut_lane[tile[cp * 32 + lane] * kLutCopies];
                    }
                    split2(v, d2, hi[cp], lo[cp]);
                }
            }
            mbar_arrive(smem_u32(&w_empty[pr % WS]));
            // the previous pair's stores have landed while this block was converted: publish them
            if (pend >= 0) {
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&pair_ready[pend % kPairSlots]));
            }
            if (kt < nkt) {
                const uint32_t slot = t_lane + (uint32_t)(kWCol0 + 32 * (kt % (2 * kPairSlots)));
                tmem_st16(slot, hi);
                tmem_st16(slot + 16, lo);
            }
            pend = pr;
            // chunk c is drained once the last pair of chunk c + 1 has been converted (the MMAs of chunk
            // c + 1 then run while this warp waits for and reads chunk c); that pair is published first
            if ((pr % kChunkPairs) == kChunkPairs - 1 && pr / kChunkPairs >= 1) {
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&pair_ready[pr % kPairSlots]));
                pend = -1;
                if (!drain(drained)) { ok = false; break; }
                ++drained;
            }
        }
        tmem_wait_st();
        if (ok && pend >= 0) {
            tc_fence_before();
            mbar_arrive(smem_u32(&pair_ready[pend % kPairSlots]));
        }
        for (; ok && drained < nchunks; ++drained)
            if (!drain(drained)) ok = false;
        asm volatile("griddepcontrol.wait;" ::: "memory");   // tscale comes from the preparation grid
        if (ok) {
            const int64_t n = ct0 * 32 + row;
            const float rs = exp2i(t);
            if (n < p.N) {
                if (!p.accumulate) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int64_t m = m0 + 64 * h + i;
                        const float v = (i & 1) ? y2[i >> 1].y : y2[i >> 1].x;
                        if (m < p.M) p.y[m * p.ldy + n] = v * rs * __ldg(p.tscale + m);
                    }
                } else {
                    // a later K pass adds its partial sums into y
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int64_t m = m0 + 64 * h + i;
                        const float v = (i & 1) ? y2[i >> 1].y : y2[i >> 1].x;
                        if (m < p.M) p.y[m * p.ldy + n] = __fadd_rn(p.y[m * p.ldy + n], v * rs * __ldg(p.tscale + m));
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

// Token operand of the folded GEMM, one warp per 512-element segment of a token row m (lane c takes
// elements 16c..16c+15 of the segment): the row's shift s (so that 127 * max_b |d_a| * 2^-s < 2^15;
// every warp of the row finds the same s), tscale[m] = 2^s (written by the row's first segment), and
// for each element the exact split of d_a[m, k/32] * 2^-s * a_q[m, k] into a_hi[m, k] + a_lo[m, k]
// (fp16).  All of a lane's loads are issued before its arithmetic.
constexpr int kPrepSeg = 512;

// Every block scale of a row shifted by 2^-s must survive the shift exactly; if one does not, the call
// is reported (QMM_ERR_RANGE).  Called by one warp per shifted row (rare, so kept out of line).
inline __device__ __noinline__ void check_shifted_row(const uint16_t *dr, int64_t nkt, int s, int lane) {
    bool exact = true;
    for (int64_t kt = lane; kt < nkt; kt += 32) {
        const float d0 = __half2float(__ushort_as_half(dr[kt]));
        exact = exact && __half2float(__float2half_rn(d0 * exp2i(-s))) * exp2i(s) == d0;
    }
    if (!__all_sync(0xffffffffu, exact) && lane == 0) atomicOr(&g_fold_status, kFoldStatusRange);
}
__global__ void __launch_bounds__(256) prepare_fold_act_kernel(const int8_t *__restrict__ a_q, const uint16_t *__restrict__ a_d,
                                                               int64_t M, int64_t K, __half *__restrict__ a_hi,
                                                               __half *__restrict__ a_lo, float *__restrict__ tscale) {
    // Launched as a programmatic dependent: wait for the grid before it on the stream (which may have
    // written a_q / a_d, or still read the workspace), then let the GEMM that follows start its set-up
    // and weight streaming; the GEMM waits for this grid before it reads the prepared tokens.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t nkt = K / 32, nseg = (K + kPrepSeg - 1) / kPrepSeg;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * 8;
    for (int64_t wi = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); wi < M * nseg; wi += warps) {
        const int64_t m = wi / nseg, seg = wi - m * nseg;
        const uint16_t *dr = a_d + m * nkt;
        const int64_t c = seg * (kPrepSeg / 16) + lane;        // 16-element chunk of the row
        const bool has = c < K / 16;
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        uint16_t dq = 0;
        if (has) {
            q = __ldg(reinterpret_cast<const uint4 *>(a_q + m * K + 16 * c));
            dq = dr[c >> 1];
        }
        float dmax = 0.0f;
#pragma unroll 4
        for (int64_t kt = lane; kt < nkt; kt += 32) dmax = fmaxf(dmax, fabsf(__half2float(__ushort_as_half(dr[kt]))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
        const int s = range_shift(dmax * 127.0f);
        if (seg == 0 && lane == 0) tscale[m] = exp2i(s);
        if (s != 0 && seg == 0) check_shifted_row(dr, nkt, s, lane);
        if (!has) continue;
        __half d = __ushort_as_half(dq);
        if (s != 0) d = __float2half_rn(__half2float(d) * exp2i(-s));
        const __half2 d2 = __half2half2(d);
        uint32_t v[8], h[8], l[8];
        i8x4_to_h2x2(q.x, v[0], v[1]);
        i8x4_to_h2x2(q.y, v[2], v[3]);
        i8x4_to_h2x2(q.z, v[4], v[5]);
        i8x4_to_h2x2(q.w, v[6], v[7]);
#pragma unroll
        for (int e = 0; e < 8; ++e) split2(v[e], d2, h[e], l[e]);
        uint4 *ho = reinterpret_cast<uint4 *>(a_hi + m * K + 16 * c), *lo = reinterpret_cast<uint4 *>(a_lo + m * K + 16 * c);
        ho[0] = make_uint4(h[0], h[1], h[2], h[3]);
        ho[1] = make_uint4(h[4], h[5], h[6], h[7]);
        lo[0] = make_uint4(l[0], l[1], l[2], l[3]);
        lo[1] = make_uint4(l[4], l[5], l[6], l[7]);
    }
}

template <int TYPE>
cudaError_t launch_fold_typed(const FoldParams &p, const CUtensorMap &ah, const CUtensorMap &al, cudaStream_t s) {
    using P = FoldPlan<TYPE>;
    static_assert(P::kSmem <= 227 * 1024, "shared memory plan too large");
    auto kern = gemm_fold_kernel<TYPE>;
    static int attr_done[4] = {0, 0, 0, 0};
    cudaError_t e = ensure_smem_limit(kern, P::kSmem, attr_done);
    if (e != cudaSuccess) return e;
    alignas(64) CUtensorMap w_map;
    e = make_weight_map(&w_map, p.tiled, P::TS, p.nkt, p.n_col_tiles);
    if (e != cudaSuccess) return e;
    // programmatic dependent of the token preparation: set-up, the weight-range scan and the weight
    // stream overlap that grid's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.n_col_tiles + 3) / 4), (unsigned)((p.M + FN - 1) / FN), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = P::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // K in passes of at most kGemmChunkBlocks blocks, each adding into y in order (the error bound)
    for (int kt0 = 0; kt0 < p.nkt; kt0 += kGemmChunkBlocks) {
        FoldParams q = p;
        q.kt0 = kt0;
        q.nkc = p.nkt - kt0 < kGemmChunkBlocks ? p.nkt - kt0 : kGemmChunkBlocks;
        q.accumulate = kt0 > 0;
        e = cudaLaunchKernelEx(&cfg, kern, q, w_map, ah, al);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

bool gemm_fold_supports(qmm_type t) { return t == QMM_Q4_0 || t == QMM_Q8_0 || t == QMM_IQ4_NL; }

cudaError_t launch_gemm_fold(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                             const uint16_t *a_d, int64_t M, float *y, int64_t ldy, void *ws, cudaStream_t s) {
    if (!gemm_fold_supports(t)) return cudaErrorNotSupported;
    if ((M + FN - 1) / FN > 65535) return cudaErrorInvalidValue;
    const GemmWsLayout L = gemm_ws_layout(M, K);
    uint8_t *base = static_cast<uint8_t *>(ws);
    __half *a_hi = reinterpret_cast<__half *>(base + L.hi);
    __half *a_lo = reinterpret_cast<__half *>(base + L.lo);
    float *tscale = reinterpret_cast<float *>(base + L.ts);
    {
        const int64_t warps = M * ((K + kPrepSeg - 1) / kPrepSeg);
        int64_t grid = (warps + 7) / 8;
        if (grid > 152 * 8) grid = 152 * 8;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, prepare_fold_act_kernel, a_q, a_d, M, K, a_hi, a_lo, tscale);
        if (e != cudaSuccess) return e;
    }
    alignas(64) CUtensorMap ah, al;
    cudaError_t e = make_map_2d(&ah, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a_hi, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, FN,
                                CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = make_map_2d(&al, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a_lo, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, FN,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    FoldParams p;
    p.tiled = tiled;
    p.tscale = tscale;
    p.y = y;
    p.N = N;
    p.M = M;
    p.ldy = ldy;
    p.n_col_tiles = (N + 31) / 32;
    p.nkt = (int)(K / 32);
    p.kt0 = 0;
    p.nkc = p.nkt;
    p.accumulate = 0;
    p.lut = lut_for(t);
    switch (t) {
        case QMM_Q4_0: return launch_fold_typed<QMM_Q4_0>(p, ah, al, s);
        case QMM_Q8_0: return launch_fold_typed<QMM_Q8_0>(p, ah, al, s);
        default: return launch_fold_typed<QMM_IQ4_NL>(p, ah, al, s);
    }
}

cudaError_t launch_selftest_wait_fold(unsigned long long limit_ns, int *out, cudaStream_t s) {
    selftest_wait_fold_kernel<<<1, 64, 0, s>>>(limit_ns, out);
    return cudaGetLastError();
}

cudaError_t read_and_clear_fold_status(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fold_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_fold_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

QMM_DCHECK_READER(read_dcheck_fold)

}  // namespace qmm

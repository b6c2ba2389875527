// gemm_tc.cu -- prefill-shaped matmul over 32-row weight tiles on the sm_103a tensor cores (tcgen05).
//
// What it computes ("Hexagon backend developer details", "Tiled Weight Formats"):
//   Y[m, n] = sum_b fp32(d_w[n,b]) * fp32(d_a[m,b]) * S_b[m,n],  S_b = sum_j w_int[n,32b+j] * a_q[m,32b+j]
// The pages' prefill path dequantizes tiles to FP16 in VTCM and feeds the 32x32 HMX array (folding the
// scale into the FP16 value, which rounds).  Here the block sums stay exact:
//   * int8 tcgen05 (kind::i8) does not exist on sm_103a, so quants are expanded to fp16 holding the
//     exact integer (|w| <= 127, |a| <= 127) and contracted with tcgen05.mma.kind::f16; every partial
//     sum of a 32-element block is an integer below 2^24, so the fp32 accumulator in TMEM is exact.
//   * The per-block scale product P_b[n,m] = d_w[n,b] * d_a[m,b] is itself a (rank-1) matrix
//     product: a third MMA with d_w and d_a in column 0 of otherwise-zero fp16 operands writes it,
//     exactly, next to S_b in TMEM.  The CUDA cores then do one fp32 FMA per element and block,
//     y += S_b * P_b, using packed fma.rn.f32x2.
//
// Tile: 128 weight rows (4 column tiles, the UMMA M dimension) x 128 tokens (UMMA N), all of K.
// Warp roles (448 threads):
//   warp 0      producer: cp.async.bulk copies of the 4 raw weight tiles and the 128 activation rows of
//               block kt into a 4-stage raw ring (mbarrier complete_tx).
//   warp 1      TMEM owner and MMA issuer (one thread): 3 MMAs per block into a 2-stage TMEM ring.
//   warps 2-5   converters: raw bytes -> fp16 operands in the canonical K-major 64-byte-swizzled
//               layout (3-stage ring), plus the d_w / d_a columns of the scale-product operands.
//   warps 6-13  rescale: tcgen05.ld of S_b and P_b, y += S_b*P_b in registers, then the fp32 store.
// Every mbarrier wait is bounded in time; on expiry the kernel records QMM_ERR_TIMEOUT in a device
// status word, lets its copies and MMAs in flight land, frees TMEM and returns.
#include "qmm_internal.cuh"

namespace qmm {

namespace {

__device__ unsigned g_device_status = 0;   // non-zero once a bounded wait gave up

constexpr int BM = 128;                    // weight rows per CTA
constexpr int BN = 128;                    // tokens per CTA
constexpr int kRawStages = 4;
constexpr int kOpStages = 3;
constexpr int kTmemStages = 2;
constexpr int kTmemCols = 512;             // 2 stages x (S 128 + P 128) fp32 columns
constexpr int kConvWarp0 = 2, kNumConvWarps = 4;
constexpr int kRescaleWarp0 = 6, kNumRescaleWarps = 8;
constexpr int kThreads = (kRescaleWarp0 + kNumRescaleWarps) * 32;
constexpr int kOpBytes = BM * 64;          // one 128 x 32 fp16 operand (64-byte rows)
constexpr int kOpStageBytes = 4 * kOpBytes;    // A (weights), B (tokens), AP (d_w), BP (d_a)
constexpr int kRawWBytes = 4 * kTile8Bytes;    // 4 raw tiles (Q8_0 worst case)
constexpr int kRawABytes = BN * 32;            // 128 activation rows of one block
constexpr int kRawStageBytes = kRawWBytes + kRawABytes;
constexpr int kLutCopies = 16;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s per wait

struct GemmParams {
    const uint8_t *tiled;
    const int8_t *a_q;
    const uint16_t *a_d;
    float *y;
    int64_t K, nkt, N, M, ldy;
    int64_t n_col_tiles;
    Lut16 lut;
};

// ---------------------------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait.  Gives up (returning false) when `abort` is raised by another warp or after
// kWaitLimitNs, in which case it raises `abort` and the device status word itself.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(&g_device_status, 1u);
            return false;
        }
    }
}

// Warp-uniform bounded wait: every lane waits, and the warp gives up together if any lane did, so
// the .sync.aligned tcgen05 instructions that follow are always executed by the full warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = wait_bounded(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Wait used while draining after an abort: no abort check, shorter limit, never raises.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs / 4) return;
    }
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, rows of 64 bytes, 64-byte swizzle,
// 8-row groups 512 bytes apart (SBO), descriptor version 1 (sm_100 family).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(512 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)4 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both K-major, M = 128, N = BN.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void ffma2(float &y0, float &y1, uint32_t s0, uint32_t s1, uint32_t p0, uint32_t p1) {
    unsigned long long yv, sv, pv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(yv) : "f"(y0), "f"(y1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(sv) : "r"(s0), "r"(s1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(pv) : "r"(p0), "r"(p1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(yv) : "l"(sv), "l"(pv));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(y0), "=f"(y1) : "l"(yv));
}

// ---------------------------------------------------------------------------------------------
// fp16 helpers (exact integer values)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// int8 pairs of a word (bytes 0,1 and 2,3) -> two half2, exact.
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__float2half_rn(1152.0f), __float2half_rn(1152.0f));
    lo = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x4140u)), bias));
    hi = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x4342u)), bias));
}

// Q4_0 nibble byte (lo = even column, hi = odd column) at byte position I -> half2(lo-8, hi-8).
template <int I>
__device__ __forceinline__ uint32_t q4_byte_to_h2(uint32_t w) {
    const uint32_t y = __byte_perm(w, 0u, 0x4040u | (I << 8) | I);
    uint32_t h;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(h) : "r"(y), "r"(0x00F0000Fu), "r"(0x64006400u));
    return h2_bits(__hfma2(bits_h2(h), __halves2half2(__float2half_rn(1.0f), __float2half_rn(0.0625f)),
                           __halves2half2(__float2half_rn(-1032.0f), __float2half_rn(-72.0f))));
}

// Byte offset of (row, 16-byte chunk) in a 128 x 64-byte K-major operand with the 64-byte swizzle
// (chunk index XOR bits 1..2 of the row; 8-row groups of 512 bytes).
__device__ __forceinline__ uint32_t sw64_off(int row, int chunk) {
    return (uint32_t)((row >> 3) * 512 + (row & 7) * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// ---------------------------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------------------------
template <int TYPE>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const GemmParams p) {
    constexpr int TS = (TYPE == QMM_Q8_0) ? kTile8Bytes : kTile4Bytes;
    constexpr int SOFF = (TYPE == QMM_Q8_0) ? kScale8Off : kScale4Off;

    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the operand stages
    const uint32_t raw_base_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base_u32 & 1023u)) & 1023u);
    uint8_t *op_s = smem;                                                     // kOpStages x kOpStageBytes
    uint8_t *raw_s = op_s + kOpStages * kOpStageBytes;                        // kRawStages x kRawStageBytes
    uint32_t *lut_s = reinterpret_cast<uint32_t *>(raw_s + kRawStages * kRawStageBytes);   // IQ4_NL only
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(lut_s) +
                                                  (TYPE == QMM_IQ4_NL ? 256 * kLutCopies * 4 : 0));
    uint64_t *raw_full = bars, *raw_empty = bars + kRawStages;
    uint64_t *op_full = bars + 2 * kRawStages, *op_empty = op_full + kOpStages;
    uint64_t *tm_full = op_empty + kOpStages, *tm_empty = tm_full + kTmemStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tm_empty + kTmemStages);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ct0 = (int64_t)blockIdx.x * 4;
    const int64_t m0 = (int64_t)blockIdx.y * BN;
    const int n_tiles = (int)((p.n_col_tiles - ct0) < 4 ? (p.n_col_tiles - ct0) : 4);
    const int n_tok = (int)((p.M - m0) < BN ? (p.M - m0) : BN);
    const int64_t nkt = p.nkt;

    // ---- set-up: barriers, zeroed scale-product operands, IQ4_NL table, TMEM ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) { mbar_init(smem_u32(&raw_full[s]), 1); mbar_init(smem_u32(&raw_empty[s]), kNumConvWarps * 32); }
        for (int s = 0; s < kOpStages; ++s) { mbar_init(smem_u32(&op_full[s]), kNumConvWarps * 32); mbar_init(smem_u32(&op_empty[s]), 1); }
        for (int s = 0; s < kTmemStages; ++s) { mbar_init(smem_u32(&tm_full[s]), 1); mbar_init(smem_u32(&tm_empty[s]), kNumRescaleWarps * 32); }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int s = 0; s < kOpStages; ++s) {
        uint4 *zp = reinterpret_cast<uint4 *>(op_s + s * kOpStageBytes + 2 * kOpBytes);   // AP and BP
        for (int i = threadIdx.x; i < 2 * kOpBytes / 16; i += kThreads) zp[i] = make_uint4(0, 0, 0, 0);
    }
    if constexpr (TYPE == QMM_IQ4_NL) {
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
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ================================ producer ================================
        uint32_t issued[kRawStages] = {0, 0, 0, 0};
        for (int64_t kt = 0; kt < nkt; ++kt) {
            const int s = (int)(kt % kRawStages);
            const uint32_t ph = (uint32_t)((kt / kRawStages) & 1);
            if (!wait_warp(smem_u32(&raw_empty[s]), ph ^ 1u, abort)) break;
            const uint32_t full = smem_u32(&raw_full[s]);
            if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(n_tiles * TS + n_tok * 32));
            __syncwarp();
            const uint32_t dst_w = smem_u32(raw_s + s * kRawStageBytes);
            if (lane < n_tiles)
                bulk_g2s(dst_w + lane * TS, p.tiled + ((ct0 + lane) * nkt + kt) * TS, TS, full);
            for (int r = lane; r < n_tok; r += 32)
                bulk_g2s(dst_w + kRawWBytes + r * 32, p.a_q + (m0 + r) * p.K + kt * 32, 32, full);
            issued[s] += 1;
        }
        // let every copy issued land before the CTA can exit
        for (int s = 0; s < kRawStages; ++s)
            if (issued[s]) wait_drain(smem_u32(&raw_full[s]), (issued[s] - 1) & 1u);
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        uint32_t committed[kTmemStages] = {0, 0};
        for (int64_t kt = 0; kt < nkt; ++kt) {
            const int os = (int)(kt % kOpStages);
            const uint32_t oph = (uint32_t)((kt / kOpStages) & 1);
            const int ts = (int)(kt % kTmemStages);
            const uint32_t tph = (uint32_t)((kt / kTmemStages) & 1);
            if (!wait_warp(smem_u32(&op_full[os]), oph, abort)) break;
            if (!wait_warp(smem_u32(&tm_empty[ts]), tph ^ 1u, abort)) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t a = smem_u32(op_s + os * kOpStageBytes);
                const uint32_t b = a + kOpBytes, ap = a + 2 * kOpBytes, bp = a + 3 * kOpBytes;
                const uint32_t d_s = tmem_base + (uint32_t)(ts * 256);
                mma_f16(d_s, smem_desc_sw64(a), smem_desc_sw64(b), 0u);
                mma_f16(d_s, smem_desc_sw64(a + 32), smem_desc_sw64(b + 32), 1u);
                mma_f16(d_s + 128, smem_desc_sw64(ap), smem_desc_sw64(bp), 0u);
                mma_commit(smem_u32(&op_empty[os]));
                mma_commit(smem_u32(&tm_full[ts]));
            }
            __syncwarp();
            committed[ts] += 1;
        }
        for (int s = 0; s < kTmemStages; ++s)
            if (committed[s]) wait_drain(smem_u32(&tm_full[s]), (committed[s] - 1) & 1u);
    } else if (warp < kRescaleWarp0) {
        // ================================ converters ================================
        const int c = threadIdx.x - kConvWarp0 * 32;        // 0..127
        const int q = c >> 5;                               // local column tile of this thread's weight word
        const int j = (c & 31) >> 2;                        // rows 4j..4j+3 of that tile
        const int cq = c & 3;                               // column pairs 4cq..4cq+3 (k 8cq..8cq+7)
        const int copy = lane & (kLutCopies - 1);
        const bool tok_ok = c < n_tok;
        uint16_t da_next = tok_ok ? p.a_d[(m0 + c) * nkt + 0] : (uint16_t)0;
        for (int64_t kt = 0; kt < nkt; ++kt) {
            const int rs = (int)(kt % kRawStages);
            const uint32_t rph = (uint32_t)((kt / kRawStages) & 1);
            const int os = (int)(kt % kOpStages);
            const uint32_t oph = (uint32_t)((kt / kOpStages) & 1);
            const uint16_t da = da_next;
            if (tok_ok && kt + 1 < nkt) da_next = p.a_d[(m0 + c) * nkt + kt + 1];
            if (!wait_bounded(smem_u32(&raw_full[rs]), rph, abort)) break;
            if (!wait_bounded(smem_u32(&op_empty[os]), oph ^ 1u, abort)) break;
            const uint8_t *raw = raw_s + rs * kRawStageBytes;
            uint8_t *op = op_s + os * kOpStageBytes;
            // -- weights: 4 rows x 8 columns per thread --
            uint32_t h[4][4];                               // [row offset][column pair offset]
            if (q < n_tiles) {
                const uint8_t *tile = raw + q * TS;
                if constexpr (TYPE == QMM_Q8_0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(tile + (4 * cq + i) * 64 + 8 * j);
                        i8x4_to_h2x2(v.x, h[0][i], h[1][i]);
                        i8x4_to_h2x2(v.y, h[2][i], h[3][i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(tile + (4 * cq + i) * 32 + 4 * j);
                        if constexpr (TYPE == QMM_Q4_0) {
                            h[0][i] = q4_byte_to_h2<0>(w);
                            h[1][i] = q4_byte_to_h2<1>(w);
                            h[2][i] = q4_byte_to_h2<2>(w);
                            h[3][i] = q4_byte_to_h2<3>(w);
                        } else {
#pragma unroll
                            for (int rr = 0; rr < 4; ++rr) h[rr][i] = lut_s[((w >> (8 * rr)) & 0xFFu) * kLutCopies + copy];
                        }
                    }
                }
            } else {
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int i = 0; i < 4; ++i) h[rr][i] = 0u;
            }
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int row = 32 * q + 4 * j + rr;
                *reinterpret_cast<uint4 *>(op + sw64_off(row, cq)) = make_uint4(h[rr][0], h[rr][1], h[rr][2], h[rr][3]);
            }
            // -- d_w of weight row c into column 0 of the AP operand --
            {
                const int tq = c >> 5, tr = c & 31;
                const uint16_t dw = (tq < n_tiles) ? *reinterpret_cast<const uint16_t *>(raw + tq * TS + SOFF + 2 * tr) : (uint16_t)0;
                *reinterpret_cast<uint16_t *>(op + 2 * kOpBytes + sw64_off(c, 0)) = dw;
            }
            // -- activations: token row c, 32 int8 -> 32 fp16 --
            {
                uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
                if (tok_ok) {
                    v0 = *reinterpret_cast<const uint4 *>(raw + kRawWBytes + c * 32);
                    v1 = *reinterpret_cast<const uint4 *>(raw + kRawWBytes + c * 32 + 16);
                }
                const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t a0, a1, a2, a3;
                    i8x4_to_h2x2(wv[2 * ch], a0, a1);
                    i8x4_to_h2x2(wv[2 * ch + 1], a2, a3);
                    *reinterpret_cast<uint4 *>(op + kOpBytes + sw64_off(c, ch)) = make_uint4(a0, a1, a2, a3);
                }
                *reinterpret_cast<uint16_t *>(op + 3 * kOpBytes + sw64_off(c, 0)) = da;
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&op_full[os]));
            mbar_arrive(smem_u32(&raw_empty[rs]));
        }
    } else {
        // ================================ rescale ================================
        const int rw = warp - kRescaleWarp0;
        const int qd = warp & 3;                     // TMEM lane quadrant this warp may access
        const int half = rw >> 2;                    // token columns 64*half .. 64*half+63
        float y[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) y[i] = 0.0f;
        bool ok = true;
        for (int64_t kt = 0; kt < nkt; ++kt) {
            const int ts = (int)(kt % kTmemStages);
            const uint32_t tph = (uint32_t)((kt / kTmemStages) & 1);
            if (!wait_warp(smem_u32(&tm_full[ts]), tph, abort)) { ok = false; break; }
            tc_fence_after();
            const uint32_t t_s = tmem_base + ((uint32_t)(32 * qd) << 16) + (uint32_t)(ts * 256 + 64 * half);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t s[16], pr[16];
                tmem_ld16(t_s + 16 * cc, s);
                tmem_ld16(t_s + 128 + 16 * cc, pr);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e += 2) ffma2(y[16 * cc + e], y[16 * cc + e + 1], s[e], s[e + 1], pr[e], pr[e + 1]);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tm_empty[ts]));
        }
        if (ok) {
            const int64_t n = (ct0 * 32) + 32 * qd + lane;
            if (n < p.N) {
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int64_t m = m0 + 64 * half + i;
                    if (m < p.M) p.y[m * p.ldy + n] = y[i];
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

template <int TYPE>
size_t gemm_smem_bytes() {
    size_t b = 1024 + (size_t)kOpStages * kOpStageBytes + (size_t)kRawStages * kRawStageBytes;
    if (TYPE == QMM_IQ4_NL) b += 256 * kLutCopies * 4;
    b += (2 * kRawStages + 2 * kOpStages + 2 * kTmemStages) * 8 + 16;
    return b;
}

template <int TYPE>
cudaError_t launch_typed(const GemmParams &p, cudaStream_t s) {
    auto kern = gemm_kernel<TYPE>;
    const size_t smem = gemm_smem_bytes<TYPE>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((p.n_col_tiles + 3) / 4), (unsigned)((p.M + BN - 1) / BN), 1);
    kern<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d,
                        int64_t M, float *y, int64_t ldy, cudaStream_t s) {
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
    p.lut = iq4nl_lut();
    if ((M + BN - 1) / BN > 65535) return cudaErrorInvalidValue;
    switch (t) {
        case QMM_Q4_0: return launch_typed<QMM_Q4_0>(p, s);
        case QMM_IQ4_NL: return launch_typed<QMM_IQ4_NL>(p, s);
        default: return launch_typed<QMM_Q8_0>(p, s);
    }
}

cudaError_t read_and_clear_device_status(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_device_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

}  // namespace qmm

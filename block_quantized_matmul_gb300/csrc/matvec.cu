// matvec.cu -- decode-shaped matmul (M <= 16 activation rows per pass) over 32-row weight tiles.
//
// What it computes ("Hexagon backend developer details", "Tiled Weight Formats"):
//   Y[m, n] = sum_b fp32(d_w[n,b]) * fp32(d_a[m,b]) * S_b[m,n],  S_b = sum_j w_int[n,32b+j] * a_q[m,32b+j]
// with w_int = q-8 (Q4_0), q (Q8_0), table[q] (IQ4_NL) read from the tile layouts of "Block-32
// Quantized Formats".  The pages' decode kernel is an HVX 32x1 / 32x2 vector dot product fed by a
// DDR -> DMA -> VTCM multi-buffered pipeline ("DDR -> DMA -> VTCM Execution Pipeline"); this is the
// GB300 counterpart of both.
//
// GB300 design:
//   * Persistent CTAs (one wide or two narrow per SM) each own a set of column tiles.  The K tiles of a column
//     tile are contiguous in memory (tile_idx = ct*n_k_tiles + kt), so one producer warp streams them
//     with 1-D cp.async.bulk copies of one stage (2 tiles per consumer warp) into a deep ring (mbarrier
//     complete_tx / consumer release) -- the pipelined multi-buffering of the pages, with the TMA
//     engine as the DMA queue.
//   * 8 or 16 consumer warps take two tiles each of every stage (two independent chains per warp).  Quants become fp16 holding exact integers
//     (biased: 1024+q or 1152+q, see decode_*), activations are staged once per CTA as fp16 in the
//     mma fragment order, and mma.sync.m16n8k16 (fp32 accumulate) yields block sums that are exact
//     integers; subtracting the exact per-(token, block) bias gives S_b.  fp16 mma.sync runs at ~4x
//     the int8 mma.sync rate on sm_103a, where int8 tcgen05 does not exist.
//   * Per block the fp32 result is rescaled by d_w*d_a with packed f32x2 arithmetic and accumulated.
//   * Launched as a programmatic dependent: weight streaming overlaps the end of the preceding grid
//     (the activation quantizer), and only the activation staging waits for it.
//   * No atomics and no scratch memory: each column tile is reduced across the warps in a fixed
//     order; if the staged activations would not fit, K is processed in passes that add into y.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kTilesPerWarp = 2;                        // independent tiles per warp per stage (ILP)
constexpr int kLutCopies = 16;
constexpr int kActBudget = 64 * 1024;                   // bytes of staged activations per CTA
constexpr int kSmemLimit = 227 * 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

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
};

__device__ unsigned g_mv_status = 0;   // set when a bounded wait gave up (reported with the GEMM's word)

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
// kWaitLimitNs, in which case it raises `abort` and the device status word itself.  The fast path
// (phase already complete) is inline; the timer is read only every 64 polls of the slow path.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(&g_mv_status, 1u);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort);
}
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
template <int CW>
__device__ __forceinline__ void consumer_sync() {      // named barrier over the consumer warps
    asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
    unsigned long long v;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(a), "f"(b));
    return v;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fmul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

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
            if constexpr (TYPE == QMM_Q4_0) {
                H[q][0] = q4_biased<0>(w);
                H[q][1] = q4_biased<1>(w);
                H[q][2] = q4_biased<2>(w);
                H[q][3] = q4_biased<3>(w);
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) H[q][r] = lut_lane[((w >> (8 * r)) & 0xFFu) * kLutCopies];
            }
        }
    }
}

// Token stride of the staged activations in uint4 units: an odd multiple of 4, so the 8 lanes of a
// quarter-warp (2 tokens x 4 column groups) read 8 distinct 16-byte bank groups.
__host__ __device__ inline int act_tok_stride(int nkc) { return nkc * 4 + ((nkc & 1) ? 0 : 4); }

// Shared-memory layout (offsets in bytes from a 128-byte aligned base).
struct MvLayout {
    int ring, bars, act, da, corr, red, lut, total;
};
template <int TYPE, int NF, int CW>
__host__ __device__ inline MvLayout mv_layout(int M, int nkc, int stages) {
    constexpr int TS = (TYPE == QMM_Q8_0) ? kTile8Bytes : kTile4Bytes;
    constexpr int kTilesPerStage = CW * kTilesPerWarp;
    MvLayout L;
    int off = 0;
    L.ring = off;  off += stages * kTilesPerStage * TS;
    off = (off + 15) & ~15;
    L.bars = off;  off += 2 * stages * 8 + 16;
    off = (off + 15) & ~15;
    L.act = off;   off += M * act_tok_stride(nkc) * 16;     // [M][stride] uint4 (16 half2 per block)
    L.da = off;    off += nkc * 8 * NF * 4;                 // [nkc][8*NF] float
    L.corr = off;  off += nkc * 8 * NF * 4;                 // [nkc][8*NF] float
    L.red = off;   off += CW * 2 * NF * 4 * 32 * 4;
    L.lut = off;   off += (TYPE == QMM_IQ4_NL) ? 256 * kLutCopies * 4 : 0;
    L.total = off;
    return L;
}

// CW consumer warps per CTA: 8 (two CTAs per SM) for grids with many column tiles, 16 (one wide CTA
// per SM) for small ones.
template <int TYPE, int NF, int CW>
__global__ void __launch_bounds__(32 * (1 + CW), 16 / CW) matvec_kernel(const MvParams p) {
    constexpr int kConsumerWarps = CW;
    constexpr int kTilesPerStage = CW * kTilesPerWarp;
    constexpr int TS = (TYPE == QMM_Q8_0) ? kTile8Bytes : kTile4Bytes;
    constexpr int SOFF = (TYPE == QMM_Q8_0) ? kScale8Off : kScale4Off;
    constexpr int TOK = 8 * NF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const MvLayout L = mv_layout<TYPE, NF, CW>(p.M, p.nkc, p.stages);
    uint8_t *ring = smem + L.ring;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + p.stages;
    volatile int *abort = reinterpret_cast<volatile int *>(empty + p.stages);
    uint4 *act_s = reinterpret_cast<uint4 *>(smem + L.act);      // [M][act_tok_stride] uint4
    const int tok_stride = act_tok_stride(p.nkc);
    float *da_s = reinterpret_cast<float *>(smem + L.da);         // [nkc][TOK]
    float *corr_s = reinterpret_cast<float *>(smem + L.corr);     // [nkc][TOK]
    float *red_s = reinterpret_cast<float *>(smem + L.red);
    uint32_t *lut_s = reinterpret_cast<uint32_t *>(smem + L.lut);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stages = p.stages;
    const int nkc = p.nkc;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        // ============================== producer ==============================
        uint32_t it = 0;
        bool ok = true;
        for (int64_t ct = blockIdx.x; ct < p.n_col_tiles && ok; ct += gridDim.x) {
            const uint8_t *src = p.tiled + (ct * p.nkt + p.kt0) * TS;
            for (int j0 = 0; j0 < nkc; j0 += kTilesPerStage, ++it) {
                const int s = (int)(it % (uint32_t)stages);
                const uint32_t ph = (it / (uint32_t)stages) & 1u;
                if (!wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort)) { ok = false; break; }
                if (lane == 0) {
                    const int nt = (nkc - j0) < kTilesPerStage ? (nkc - j0) : kTilesPerStage;
                    const uint32_t bytes = (uint32_t)(nt * TS);
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s(smem_u32(ring + s * kTilesPerStage * TS), src + (int64_t)j0 * TS, bytes, fb);
                }
                __syncwarp();
            }
        }
        // copies in flight land before the CTA may exit
        if (lane == 0 && it > 0) {
            const uint32_t last = it - 1;
            for (uint32_t k = 0; k < (uint32_t)stages && k <= last; ++k) {
                const uint32_t i = last - k;
                wait_drain(smem_u32(&full[i % stages]), (i / stages) & 1u);
            }
        }
        return;
    }

    // ============================== consumers ==============================
    const int cw = warp - 1;                  // consumer warp 0..7
    const int ctid = threadIdx.x - 32;        // 0..255
    const int g = lane >> 2, t = lane & 3;

    // The weights never depend on the kernel launched just before on the stream, so the producer
    // starts streaming at once; the activations may, so the consumers wait for that grid first
    // (a no-op unless this grid was launched as its programmatic dependent).
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- stage activations once: per (token, block) 16 half2 in fragment order, plus the
    //      per-block scale and the exact bias of the biased weight decode ----
    if constexpr (TYPE == QMM_IQ4_NL) {
        for (int i = ctid; i < 256 * kLutCopies; i += kConsumerWarps * 32) {
            const int b = i / kLutCopies;
            lut_s[i] = h2_bits(__halves2half2(__int2half_rn(p.lut.v[b & 15]), __int2half_rn(p.lut.v[b >> 4])));
        }
    }
    for (int i = ctid; i < TOK * nkc; i += kConsumerWarps * 32) {
        const int j = i / TOK, tok = i - j * TOK;
        float d = 0.0f, corr = 0.0f;
        if (tok < p.M) {
            const int64_t kt = p.kt0 + j;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.a_q + (int64_t)tok * p.K + kt * 32);
            const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
            const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            int sum_even = 0, sum_odd = 0;
            uint32_t hp[16];                 // half2 of column pair cp, in cp order
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int a0 = (int)(int8_t)((wv[wi] >> (16 * h)) & 0xFF);
                    const int a1 = (int)(int8_t)((wv[wi] >> (16 * h + 8)) & 0xFF);
                    sum_even += a0;
                    sum_odd += a1;
                    const float f1 = (TYPE == QMM_Q4_0) ? (float)a1 * 0.0625f : (float)a1;   // exact
                    hp[2 * wi + h] = h2_bits(__halves2half2(__float2half_rn((float)a0), __float2half_rn(f1)));
                }
            }
            // fragment order: position 4t + q holds column pair t + 4q
            uint4 *dst = act_s + tok * tok_stride + j * 4;
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) dst[tt] = make_uint4(hp[tt], hp[tt + 4], hp[tt + 8], hp[tt + 12]);
            d = __half2float(__ushort_as_half(p.a_d[(int64_t)tok * p.nkt + kt]));
            if (TYPE == QMM_Q4_0) corr = 1032.0f * (float)sum_even + 72.0f * (float)sum_odd;
            else if (TYPE == QMM_Q8_0) corr = 1152.0f * (float)(sum_even + sum_odd);
        }
        da_s[j * TOK + tok] = d;
        corr_s[j * TOK + tok] = corr;
    }
    consumer_sync<CW>();

    // After a timed-out wait a warp stops waiting and computing but keeps the loop structure, so
    // every consumer warp still reaches the same named barriers.
    const uint32_t *lut_lane = lut_s + (lane & (kLutCopies - 1));
    uint32_t it = 0;
    bool ok = true;
    for (int64_t ct = blockIdx.x; ct < p.n_col_tiles; ct += gridDim.x) {
        unsigned long long acc[2][NF][2];     // [rb][nf][row pair half]: (tok 2t, 2t+1) of rows 4g+2rb(+1)
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int nf = 0; nf < NF; ++nf) acc[rb][nf][0] = acc[rb][nf][1] = 0ull;

        for (int j0 = 0; j0 < nkc; j0 += kTilesPerStage, ++it) {
            const int s = (int)(it % (uint32_t)stages);
            const uint32_t ph = (it / (uint32_t)stages) & 1u;
            if (ok) ok = __all_sync(0xffffffffu, wait_bounded(smem_u32(&full[s]), ph, abort));
            if (ok) {
                // tiles cw and cw + 8 of this stage, decoded and contracted side by side
                uint32_t H[kTilesPerWarp][4][4];
                float dwr[kTilesPerWarp][4];
                bool live[kTilesPerWarp];
#pragma unroll
                for (int u = 0; u < kTilesPerWarp; ++u) {
                    const int jt = j0 + cw + kConsumerWarps * u;
                    live[u] = jt < nkc;
                    const uint8_t *tile = ring + (s * kTilesPerStage + cw + kConsumerWarps * u) * TS;
                    if (live[u]) {
                        decode_tile<TYPE>(tile, g, t, H[u], lut_lane);
                        const uint2 sc = *reinterpret_cast<const uint2 *>(tile + SOFF + 8 * g);
                        const float2 dw01 = __half22float2(bits_h2(sc.x));      // rows 4g, 4g+1
                        const float2 dw23 = __half22float2(bits_h2(sc.y));      // rows 4g+2, 4g+3
                        dwr[u][0] = dw01.x; dwr[u][1] = dw01.y; dwr[u][2] = dw23.x; dwr[u][3] = dw23.y;
                    }
                }
#pragma unroll
                for (int u = 0; u < kTilesPerWarp; ++u) {
                    if (!live[u]) continue;
                    const int j = j0 + cw + kConsumerWarps * u;
#pragma unroll
                    for (int nf = 0; nf < NF; ++nf) {
                        const int tok = 8 * nf + g;
                        uint4 b = make_uint4(0, 0, 0, 0);
                        if (tok < p.M) b = act_s[tok * tok_stride + j * 4 + t];
                        const float2 da = *reinterpret_cast<const float2 *>(da_s + j * TOK + 8 * nf + 2 * t);
                        const float2 cr = *reinterpret_cast<const float2 *>(corr_s + j * TOK + 8 * nf + 2 * t);
                        const unsigned long long ncorr = pack2(-cr.x, -cr.y);
                        const unsigned long long da2 = pack2(da.x, da.y);
#pragma unroll
                        for (int rb = 0; rb < 2; ++rb) {
                            float c[4] = {0.f, 0.f, 0.f, 0.f};
                            mma16816(c, H[u][0][2 * rb], H[u][0][2 * rb + 1], H[u][1][2 * rb], H[u][1][2 * rb + 1], b.x, b.y);
                            mma16816(c, H[u][2][2 * rb], H[u][2][2 * rb + 1], H[u][3][2 * rb], H[u][3][2 * rb + 1], b.z, b.w);
                            // c0,c1: row 4g+2rb, tokens 2t,2t+1;  c2,c3: row 4g+2rb+1
                            const unsigned long long s01 = fadd2(pack2(c[0], c[1]), ncorr);
                            const unsigned long long s23 = fadd2(pack2(c[2], c[3]), ncorr);
                            const unsigned long long p01 = fmul2(pack2(dwr[u][2 * rb], dwr[u][2 * rb]), da2);
                            const unsigned long long p23 = fmul2(pack2(dwr[u][2 * rb + 1], dwr[u][2 * rb + 1]), da2);
                            acc[rb][nf][0] = ffma2(s01, p01, acc[rb][nf][0]);
                            acc[rb][nf][1] = ffma2(s23, p23, acc[rb][nf][1]);
                        }
                    }
                }
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

struct Plan {
    int nf, nkc, stages, ctas_per_sm;
    size_t smem;
};

template <int TYPE, int NF, int CW>
Plan plan_for(int M, int64_t nkt) {
    constexpr int TS = (TYPE == QMM_Q8_0) ? kTile8Bytes : kTile4Bytes;
    constexpr int kTilesPerStage = CW * kTilesPerWarp;
    Plan pl;
    pl.nf = NF;
    int64_t nkc = kActBudget / (64 * (int64_t)M);
    if (nkc > nkt) nkc = nkt;
    if (nkc < 1) nkc = 1;
    pl.nkc = (int)nkc;
    const int fixed = mv_layout<TYPE, NF, CW>(M, pl.nkc, 0).total + 128;
    const int stage_bytes = kTilesPerStage * TS + 16;
    // CW = 16: one wide CTA per SM (all of shared memory); CW = 8: two CTAs per SM (half each)
    const int budget = (CW == 16) ? kSmemLimit : kSmemLimit / 2;
    int st = (budget - 1024 - fixed) / stage_bytes;
    pl.stages = st > 12 ? 12 : st;
    pl.ctas_per_sm = 16 / CW;
    if (pl.stages < 2) pl.stages = 2;
    pl.smem = (size_t)mv_layout<TYPE, NF, CW>(M, pl.nkc, pl.stages).total + 128;
    return pl;
}

int num_sms() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 152;
    }
    return sms;
}

template <int TYPE, int NF, int CW>
cudaError_t run_cw(const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d, int M, float *y,
                   int64_t ldy, cudaStream_t s) {
    const int64_t nkt = K / 32, nct = (N + 31) / 32;
    const Plan pl = plan_for<TYPE, NF, CW>(M, nkt);
    auto kern = matvec_kernel<TYPE, NF, CW>;
    static int attr_done[4] = {0, 0, 0, 0};
    cudaError_t e = ensure_smem_limit(kern, kSmemLimit, attr_done);
    if (e != cudaSuccess) return e;
    int64_t grid = (int64_t)num_sms() * pl.ctas_per_sm;
    if (grid > nct) grid = nct;
    for (int64_t kt0 = 0; kt0 < nkt; kt0 += pl.nkc) {
        MvParams p;
        p.tiled = tiled;
        p.a_q = a_q;
        p.a_d = a_d;
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
        p.lut = iq4nl_lut();
        // programmatic dependent launch: may start while the previous grid on the stream is still
        // running (only if that grid allows it); the kernel waits before it reads activations or y
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(32 * (1 + CW), 1, 1);
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, p);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Many column tiles: two narrow CTAs per SM hide latency best; few: one wide CTA per SM streams each
// column tile twice as fast, which keeps the rounds of a small grid short and balanced.
template <int TYPE, int NF>
cudaError_t run(const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q, const uint16_t *a_d, int M, float *y,
                int64_t ldy, cudaStream_t s) {
    const int64_t nct = (N + 31) / 32;
    if (nct >= (int64_t)num_sms() * 8) return run_cw<TYPE, NF, 8>(tiled, K, N, a_q, a_d, M, y, ldy, s);
    return run_cw<TYPE, NF, 16>(tiled, K, N, a_q, a_d, M, y, ldy, s);
}

}  // namespace

cudaError_t launch_matvec(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                          const uint16_t *a_d, int64_t M, float *y, int64_t ldy, cudaStream_t s) {
    const int64_t nkt = K / 32;
    for (int64_t m0 = 0; m0 < M; m0 += kDecodeMaxM) {
        const int mm = (int)((M - m0) < kDecodeMaxM ? (M - m0) : kDecodeMaxM);
        const int8_t *aq = a_q + m0 * K;
        const uint16_t *ad = a_d + m0 * nkt;
        float *yy = y + m0 * ldy;
        cudaError_t e;
        const bool two = mm > 8;
        switch (t) {
            case QMM_Q4_0: e = two ? run<QMM_Q4_0, 2>(tiled, K, N, aq, ad, mm, yy, ldy, s) : run<QMM_Q4_0, 1>(tiled, K, N, aq, ad, mm, yy, ldy, s); break;
            case QMM_IQ4_NL: e = two ? run<QMM_IQ4_NL, 2>(tiled, K, N, aq, ad, mm, yy, ldy, s) : run<QMM_IQ4_NL, 1>(tiled, K, N, aq, ad, mm, yy, ldy, s); break;
            default: e = two ? run<QMM_Q8_0, 2>(tiled, K, N, aq, ad, mm, yy, ldy, s) : run<QMM_Q8_0, 1>(tiled, K, N, aq, ad, mm, yy, ldy, s); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t read_and_clear_matvec_status(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_mv_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_mv_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

}  // namespace qmm

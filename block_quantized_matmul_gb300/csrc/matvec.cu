// matvec.cu -- decode-shaped matmul (M <= 16 activation rows) over 32-row weight tiles.
//
// What it computes ("Hexagon backend developer details", "Tiled Weight Formats"):
//   Y[m, n] = sum_b fp32(d_w[n,b]) * fp32(d_a[m,b]) * S_b[m,n],  S_b = sum_j w_int[n,32b+j] * a_q[m,32b+j]
// with w_int = q-8 (Q4_0), q (Q8_0), table[q] (IQ4_NL) read from the tile layouts of "Block-32
// Quantized Formats".  The pages' own decode kernel is an HVX 32x1 / 32x2 vector dot product against
// Q8_0 activation tiles; on GB300 the block dot products run on the tensor cores instead.
//
// GB300 design:
//   * Weight bytes are streamed once from HBM with 4/8-byte vector loads straight into registers;
//     each warp owns one column tile (32 rows) and a strided subset of its K tiles.
//   * Quants are decoded to fp16 holding the exact integer value (|v| <= 127), activations are the
//     int8 quants as fp16, and `mma.sync.m16n8k16` with fp32 accumulation produces the exact integer
//     block sums S_b (every partial sum is an integer below 2^24).  fp16 mma runs at ~4x the rate of
//     the int8 mma.sync path on sm_103a, and int8 tcgen05 does not exist there.
//   * Dot products within a block do not depend on the order of k, nor on which logical mma row a
//     weight row occupies: each thread takes the 4 tile rows 4g..4g+3 of one 4-byte word and the
//     column pairs cp = t, t+4, t+8, t+12, so every load is a whole word of the tile.
//   * Per block, the fp32 result is rescaled by d_w*d_a in registers and accumulated in fp32.
//   * Split-K across the CTAs of a thread-block cluster; partial sums are added in a fixed order
//     through distributed shared memory, so results are bit-reproducible (no atomics).
#include <cooperative_groups.h>

#include "qmm_internal.cuh"

namespace cg = cooperative_groups;

namespace qmm {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kChunkTiles = 32;          // K tiles of activations staged in shared memory at a time
constexpr int kActPad = 8;               // halfs of padding per staged activation row (bank spread)
constexpr int kLutCopies = 16;           // IQ4_NL byte->half2 table copies (spreads banks)
constexpr int kUnroll = 4;               // tiles loaded ahead per warp

struct MatvecParams {
    const uint8_t *tiled;
    const int8_t *a_q;
    const uint16_t *a_d;
    float *y;
    int64_t nkt;          // K / 32
    int64_t N;
    int64_t ldy;
    int M;                // activation rows in this launch (<= 8 * NF)
    int kt_per_cta;       // K tiles handled by one CTA of the split
    int ksplit;           // CTAs per column tile (= cluster size along y)
    Lut16 lut;
};

__device__ __forceinline__ uint32_t ldg_u32(const uint8_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_u64(const uint8_t *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Q4_0 byte i of a tile word -> half2(lo - 8, hi - 8), exact.  The byte is copied into both 16-bit
// halves; the low nibble becomes the mantissa of 1024 + lo, the high nibble that of 1024 + 16*hi,
// and one fp16 fma removes the offsets.
template <int I>
__device__ __forceinline__ uint32_t q4_pair(uint32_t w) {
    const uint32_t y = __byte_perm(w, 0u, 0x4040u | (I << 8) | I);
    uint32_t h;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(h) : "r"(y), "r"(0x00F0000Fu), "r"(0x64006400u));  // (y & b) | c
    const __half2 r = __hfma2(bits_h2(h), __halves2half2(__float2half_rn(1.0f), __float2half_rn(0.0625f)),
                              __halves2half2(__float2half_rn(-1032.0f), __float2half_rn(-72.0f)));
    return h2_bits(r);
}

// Q8_0: two int8 of one row (bytes I, I+1 of w) -> half2, exact: (b ^ 0x80) is b + 128 as an
// unsigned byte, placed in the mantissa of 1024; subtracting 1152 leaves b.
template <int SEL>
__device__ __forceinline__ uint32_t q8_pair(uint32_t w_xor) {
    const uint32_t h = __byte_perm(w_xor, 0x64646464u, SEL);
    const __half2 r = __hsub2(bits_h2(h), __halves2half2(__float2half_rn(1152.0f), __float2half_rn(1152.0f)));
    return h2_bits(r);
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Raw bytes of one tile held by one thread.
template <int TYPE>
struct TileRegs;
template <>
struct TileRegs<QMM_Q8_0> {
    uint2 q[4];
    uint2 sc;
};
template <int TYPE>
struct TileRegs {
    uint32_t q[4];
    uint2 sc;
};

template <int TYPE>
__device__ __forceinline__ void load_tile(TileRegs<TYPE> &r, const uint8_t *tp, int g, int t) {
    if constexpr (TYPE == QMM_Q8_0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) r.q[q] = ldg_u64(tp + (t + 4 * q) * 64 + 8 * g);
        r.sc = ldg_u64(tp + kScale8Off + 8 * g);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) r.q[q] = ldg_u32(tp + (t + 4 * q) * 32 + 4 * g);
        r.sc = ldg_u64(tp + kScale4Off + 8 * g);
    }
}

// Decode to H[q][i]: half2 of (column 2cp, 2cp+1) for tile row 4g+i, column pair cp = t + 4q.
template <int TYPE>
__device__ __forceinline__ void decode_tile(const TileRegs<TYPE> &r, uint32_t (&H)[4][4], const uint32_t *lut_s,
                                            int copy) {
    if constexpr (TYPE == QMM_Q8_0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t x = r.q[q].x ^ 0x80808080u, z = r.q[q].y ^ 0x80808080u;
            H[q][0] = q8_pair<0x4140>(x);
            H[q][1] = q8_pair<0x4342>(x);
            H[q][2] = q8_pair<0x4140>(z);
            H[q][3] = q8_pair<0x4342>(z);
        }
    } else if constexpr (TYPE == QMM_Q4_0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            H[q][0] = q4_pair<0>(r.q[q]);
            H[q][1] = q4_pair<1>(r.q[q]);
            H[q][2] = q4_pair<2>(r.q[q]);
            H[q][3] = q4_pair<3>(r.q[q]);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t b = (r.q[q] >> (8 * i)) & 0xFFu;
                H[q][i] = lut_s[b * kLutCopies + copy];
            }
        }
    }
}

template <int TYPE, int NF>
__global__ void __launch_bounds__(kThreads) matvec_kernel(const MatvecParams p) {
    constexpr int TS = (TYPE == QMM_Q8_0) ? kTile8Bytes : kTile4Bytes;
    constexpr int TOK = 8 * NF;
    constexpr int ROW_H = kChunkTiles * 32 + kActPad;       // staged activation row stride (halfs)

    extern __shared__ __align__(16) uint8_t smem[];
    __half *act_s = reinterpret_cast<__half *>(smem);                                   // [TOK][ROW_H]
    float *da_s = reinterpret_cast<float *>(smem + TOK * ROW_H * 2);                     // [TOK][kChunkTiles]
    float *red_s = da_s + TOK * kChunkTiles;                                             // [kWarps][2][NF][4][32]
    uint32_t *lut_s = reinterpret_cast<uint32_t *>(red_s + kWarps * 2 * NF * 4 * 32);     // [256][kLutCopies]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t ct = blockIdx.x;
    const int64_t kt_begin = (int64_t)blockIdx.y * p.kt_per_cta;
    const int64_t kt_end = (kt_begin + p.kt_per_cta < p.nkt) ? kt_begin + p.kt_per_cta : p.nkt;

    if constexpr (TYPE == QMM_IQ4_NL) {
        for (int i = threadIdx.x; i < 256 * kLutCopies; i += kThreads) {
            const int b = i / kLutCopies;
            const __half2 v = __halves2half2(__int2half_rn(p.lut.v[b & 15]), __int2half_rn(p.lut.v[b >> 4]));
            lut_s[i] = h2_bits(v);
        }
    }

    float acc[2][NF][4];
#pragma unroll
    for (int rb = 0; rb < 2; ++rb)
#pragma unroll
        for (int nf = 0; nf < NF; ++nf)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[rb][nf][c] = 0.0f;

    const uint8_t *col_base = p.tiled + (size_t)ct * p.nkt * TS;

    for (int64_t c0 = kt_begin; c0 < kt_end; c0 += kChunkTiles) {
        const int nt = (int)((kt_end - c0) < kChunkTiles ? (kt_end - c0) : kChunkTiles);
        // ---- stage activations of this chunk: int8 -> fp16 (exact), rows >= M zero ----
        __syncthreads();
        {
            const int words_per_row = nt * 8;                  // 4 int8 per word
            for (int i = threadIdx.x; i < TOK * words_per_row; i += kThreads) {
                const int tok = i / words_per_row, wi = i - tok * words_per_row;
                uint32_t v = 0;
                if (tok < p.M) v = __ldg(reinterpret_cast<const uint32_t *>(p.a_q + (int64_t)tok * p.nkt * 32 + c0 * 32) + wi);
                const __half2 lo = __halves2half2(__int2half_rn((int8_t)(v & 0xFF)), __int2half_rn((int8_t)((v >> 8) & 0xFF)));
                const __half2 hi = __halves2half2(__int2half_rn((int8_t)((v >> 16) & 0xFF)), __int2half_rn((int8_t)(v >> 24)));
                uint2 st;
                st.x = h2_bits(lo);
                st.y = h2_bits(hi);
                *reinterpret_cast<uint2 *>(act_s + tok * ROW_H + wi * 4) = st;
            }
            for (int i = threadIdx.x; i < TOK * nt; i += kThreads) {
                const int tok = i / nt, j = i - tok * nt;
                float d = 0.0f;
                if (tok < p.M) d = __half2float(__ushort_as_half(p.a_d[(int64_t)tok * p.nkt + c0 + j]));
                da_s[tok * kChunkTiles + j] = d;
            }
        }
        __syncthreads();

        // ---- each warp takes tiles j = warp, warp + kWarps, ... of the chunk, kUnroll at a time ----
        for (int j0 = warp * kUnroll; j0 < nt; j0 += kWarps * kUnroll) {
            TileRegs<TYPE> regs[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (j0 + u < nt) load_tile<TYPE>(regs[u], col_base + (size_t)(c0 + j0 + u) * TS, g, t);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u;
                if (j >= nt) break;
                uint32_t H[4][4];
                decode_tile<TYPE>(regs[u], H, lut_s, lane & (kLutCopies - 1));
                const float dw[4] = {__half2float(__ushort_as_half((uint16_t)(regs[u].sc.x & 0xFFFF))),
                                     __half2float(__ushort_as_half((uint16_t)(regs[u].sc.x >> 16))),
                                     __half2float(__ushort_as_half((uint16_t)(regs[u].sc.y & 0xFFFF))),
                                     __half2float(__ushort_as_half((uint16_t)(regs[u].sc.y >> 16)))};
#pragma unroll
                for (int nf = 0; nf < NF; ++nf) {
                    const __half *arow = act_s + (8 * nf + g) * ROW_H + j * 32;
                    // b registers: column pair cp = t + 4q -> halfs 2cp, 2cp+1 of the block
                    const uint32_t b00 = *reinterpret_cast<const uint32_t *>(arow + 2 * t);
                    const uint32_t b01 = *reinterpret_cast<const uint32_t *>(arow + 2 * (t + 4));
                    const uint32_t b10 = *reinterpret_cast<const uint32_t *>(arow + 2 * (t + 8));
                    const uint32_t b11 = *reinterpret_cast<const uint32_t *>(arow + 2 * (t + 12));
                    const float da0 = da_s[(8 * nf + 2 * t) * kChunkTiles + j];
                    const float da1 = da_s[(8 * nf + 2 * t + 1) * kChunkTiles + j];
#pragma unroll
                    for (int rb = 0; rb < 2; ++rb) {
                        float c[4] = {0.f, 0.f, 0.f, 0.f};
                        const uint32_t a0[4] = {H[0][2 * rb], H[0][2 * rb + 1], H[1][2 * rb], H[1][2 * rb + 1]};
                        const uint32_t a1[4] = {H[2][2 * rb], H[2][2 * rb + 1], H[3][2 * rb], H[3][2 * rb + 1]};
                        mma16816(c, a0, b00, b01);
                        mma16816(c, a1, b10, b11);
                        // c0: (row 4g+2rb, tok 2t) c1: (row 4g+2rb, tok 2t+1) c2/c3: row 4g+2rb+1
                        acc[rb][nf][0] = fmaf(c[0], dw[2 * rb] * da0, acc[rb][nf][0]);
                        acc[rb][nf][1] = fmaf(c[1], dw[2 * rb] * da1, acc[rb][nf][1]);
                        acc[rb][nf][2] = fmaf(c[2], dw[2 * rb + 1] * da0, acc[rb][nf][2]);
                        acc[rb][nf][3] = fmaf(c[3], dw[2 * rb + 1] * da1, acc[rb][nf][3]);
                    }
                }
            }
        }
    }

    // ---- reduce the warps of this CTA in a fixed order ----
#pragma unroll
    for (int rb = 0; rb < 2; ++rb)
#pragma unroll
        for (int nf = 0; nf < NF; ++nf)
#pragma unroll
            for (int c = 0; c < 4; ++c) red_s[(((warp * 2 + rb) * NF + nf) * 4 + c) * 32 + lane] = acc[rb][nf][c];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int nf = 0; nf < NF; ++nf)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float s = red_s[(((0 * 2 + rb) * NF + nf) * 4 + c) * 32 + lane];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) s += red_s[(((w * 2 + rb) * NF + nf) * 4 + c) * 32 + lane];
                    red_s[(((0 * 2 + rb) * NF + nf) * 4 + c) * 32 + lane] = s;   // CTA partial in slot 0
                    acc[rb][nf][c] = s;
                }
    }

    if (p.ksplit > 1) {
        // ---- add the partials of the cluster's CTAs (rank order) through distributed smem ----
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (cluster.block_rank() == 0 && warp == 0) {
            for (int rk = 1; rk < p.ksplit; ++rk) {
                const float *peer = cluster.map_shared_rank(red_s, rk);
#pragma unroll
                for (int rb = 0; rb < 2; ++rb)
#pragma unroll
                    for (int nf = 0; nf < NF; ++nf)
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[rb][nf][c] += peer[((rb * NF + nf) * 4 + c) * 32 + lane];
            }
        }
        cluster.sync();
        if (cluster.block_rank() != 0) return;
    }

    if (warp == 0) {
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
            for (int nf = 0; nf < NF; ++nf)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int row = 4 * g + 2 * rb + (c >> 1);
                    const int tok = 8 * nf + 2 * t + (c & 1);
                    const int64_t n = ct * 32 + row;
                    if (tok < p.M && n < p.N) p.y[(int64_t)tok * p.ldy + n] = acc[rb][nf][c];
                }
    }
}

template <int TYPE, int NF>
size_t smem_bytes() {
    constexpr int TOK = 8 * NF;
    size_t b = (size_t)TOK * (kChunkTiles * 32 + kActPad) * 2 + (size_t)TOK * kChunkTiles * 4 +
               (size_t)kWarps * 2 * NF * 4 * 32 * 4;
    if (TYPE == QMM_IQ4_NL) b += 256 * kLutCopies * 4;
    return b;
}

template <int TYPE, int NF>
cudaError_t launch_typed(const MatvecParams &p0, int64_t n_col_tiles, cudaStream_t s) {
    MatvecParams p = p0;
    auto kern = matvec_kernel<TYPE, NF>;
    const size_t smem = smem_bytes<TYPE, NF>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_col_tiles, (unsigned)p.ksplit, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.ksplit;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_matvec(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, const int8_t *a_q,
                          const uint16_t *a_d, int64_t M, float *y, int64_t ldy, cudaStream_t s) {
    const int64_t nkt = K / 32, nct = (N + 31) / 32;
    // Split K over up to 8 CTAs (one cluster) so that the grid holds several CTAs per SM.
    const int64_t target_ctas = 152 * 8;
    int ksplit = 1;
    while (ksplit < 8 && nct * ksplit < target_ctas && nkt / (ksplit * 2) >= kUnroll) ksplit *= 2;
    const int kpc = (int)((nkt + ksplit - 1) / ksplit);
    ksplit = (int)((nkt + kpc - 1) / kpc);      // no empty CTAs
    for (int64_t m0 = 0; m0 < M; m0 += kDecodeMaxM) {
        const int mm = (int)((M - m0) < kDecodeMaxM ? (M - m0) : kDecodeMaxM);
        MatvecParams p;
        p.tiled = tiled;
        p.a_q = a_q + m0 * K;
        p.a_d = a_d + m0 * nkt;
        p.y = y + m0 * ldy;
        p.nkt = nkt;
        p.N = N;
        p.ldy = ldy;
        p.M = mm;
        p.kt_per_cta = kpc;
        p.ksplit = ksplit;
        p.lut = iq4nl_lut();
        cudaError_t e;
        const bool two = mm > 8;
        switch (t) {
            case QMM_Q4_0: e = two ? launch_typed<QMM_Q4_0, 2>(p, nct, s) : launch_typed<QMM_Q4_0, 1>(p, nct, s); break;
            case QMM_IQ4_NL: e = two ? launch_typed<QMM_IQ4_NL, 2>(p, nct, s) : launch_typed<QMM_IQ4_NL, 1>(p, nct, s); break;
            default: e = two ? launch_typed<QMM_Q8_0, 2>(p, nct, s) : launch_typed<QMM_Q8_0, 1>(p, nct, s); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace qmm

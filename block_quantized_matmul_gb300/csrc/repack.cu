// repack.cu -- flat GGML rows <-> 32-row tiles ("Tiled Weight Formats": "Tile Dimensions and Grid
// Layout", "Block-32 Quantized Formats").  Load-time kernels: read and write the weight once.
//
// Thread mapping: one thread per (tile, tile row).  A warp covers the 32 rows of one tile, so each
// per-column-pair store of the warp is one contiguous run (32 bytes for 4-bit tiles, 64 for Q8_0).
// Q4_K super-blocks ("K-Quants Formats") are split into the 8 Q4_1-layout tiles of their 32-wide
// sub-blocks, the row pair becoming (fp16(d*sc), fp16(-dmin*m)); that direction only (the products
// cannot be split back).
#include "qmm_internal.cuh"

namespace qmm {
namespace {

__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

template <int TYPE>
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *__restrict__ flat, int64_t n_k_tiles, int64_t N,
                                                     int64_t n_tiles, uint8_t *__restrict__ tiled) {
    constexpr bool k8 = (TYPE == QMM_Q8_0);
    constexpr bool mx = (TYPE == QMM_MXFP4);            // 17-byte blocks: byte access only
    constexpr bool q41 = (TYPE == QMM_Q4_1);            // 20-byte blocks: (d, m) then the nibbles
    constexpr int bb = k8 ? kBlock8Bytes : (mx ? kBlockMxBytes : (q41 ? kBlock41Bytes : kBlock4Bytes));
    constexpr int head = mx ? 1 : (q41 ? 4 : 2);        // bytes before the quants
    constexpr int ts = TileFmt<TYPE>::kBytes;
    constexpr int soff = TileFmt<TYPE>::kScaleOff;
    const int64_t total = n_tiles * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i >> 5;
        const int r = (int)(i & 31);
        const int64_t ct = tile / n_k_tiles, kt = tile - ct * n_k_tiles;
        const int64_t n = ct * 32 + r;
        // tile index < n_col_tiles * n_k_tiles, block index kt < K / 32
        if (!QMM_DCHECK(tile < n_tiles && kt < n_k_tiles)) continue;
        uint8_t *t = tiled + tile * ts;
        if (n >= N) {                                   // padding row: all zero
            if (k8) {
#pragma unroll
                for (int cp = 0; cp < 16; ++cp) *reinterpret_cast<uint16_t *>(t + cp * 64 + 2 * r) = 0;
            } else {
#pragma unroll
                for (int cp = 0; cp < 16; ++cp) t[cp * 32 + r] = 0;
            }
            if (mx) t[soff + r] = 0;
            else if (q41) *reinterpret_cast<uint32_t *>(t + soff + 4 * r) = 0u;
            else *reinterpret_cast<uint16_t *>(t + soff + 2 * r) = 0;
            continue;
        }
        const uint8_t *blk = flat + (n * n_k_tiles + kt) * bb;
        if (k8) {
            // element pair (2cp, 2cp+1) is already adjacent in the flat block
#pragma unroll
            for (int cp = 0; cp < 16; ++cp)
                *reinterpret_cast<uint16_t *>(t + cp * 64 + 2 * r) = (uint16_t)ld_u16(blk + 2 + 2 * cp);
        } else {
            uint32_t qs[8];                             // 16 nibble bytes as 8 halfwords
#pragma unroll
            for (int h = 0; h < 8; ++h)
                qs[h] = mx ? ((uint32_t)blk[1 + 2 * h] | ((uint32_t)blk[2 + 2 * h] << 8)) : ld_u16(blk + head + 2 * h);
#pragma unroll
            for (int cp = 0; cp < 16; ++cp) {
                // element e: byte e&15 of the block, low nibble for e < 16, high nibble otherwise
                const int e0 = 2 * cp, e1 = 2 * cp + 1;
                const uint32_t b0 = (qs[(e0 & 15) >> 1] >> (8 * (e0 & 1))) & 0xFF;
                const uint32_t b1 = (qs[(e1 & 15) >> 1] >> (8 * (e1 & 1))) & 0xFF;
                const uint32_t c0 = (e0 < 16) ? (b0 & 15) : (b0 >> 4);
                const uint32_t c1 = (e1 < 16) ? (b1 & 15) : (b1 >> 4);
                t[cp * 32 + r] = (uint8_t)(c0 | (c1 << 4));
            }
        }
        if (mx) t[soff + r] = blk[0];                   // the row's E8M0 exponent
        else if (q41) *reinterpret_cast<uint32_t *>(t + soff + 4 * r) = *reinterpret_cast<const uint32_t *>(blk);   // d, m
        else *reinterpret_cast<uint16_t *>(t + soff + 2 * r) = (uint16_t)ld_u16(blk);
    }
    // The decode matmul streams tiles before it waits for the kernel before it on the stream, so the
    // tiles must be visible device-wide by the time this grid's blocks have exited.
    __threadfence();
}

// Q4_K super-blocks -> Q4_1-layout tiles ("K-Quants Formats"): tile kt of row n holds sub-block
// j = kt % 8 of super-block kt / 8, its codes in the Q4_0 nibble layout and the row pair
// (fp16(d*sc_j), fp16(-dmin*m_j)).  One thread per (tile, tile row), as above.
__global__ void __launch_bounds__(256) repack_q4k_kernel(const uint8_t *__restrict__ flat, int64_t n_k_tiles, int64_t N,
                                                         int64_t n_tiles, uint8_t *__restrict__ tiled) {
    const int64_t total = n_tiles * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i >> 5;
        const int r = (int)(i & 31);
        const int64_t ct = tile / n_k_tiles, kt = tile - ct * n_k_tiles;
        const int64_t n = ct * 32 + r;
        uint8_t *t = tiled + tile * kTile41Bytes;
        if (n >= N) {
#pragma unroll
            for (int cp = 0; cp < 16; ++cp) t[cp * 32 + r] = 0;
            *reinterpret_cast<uint32_t *>(t + kScale4Off + 4 * r) = 0u;
            continue;
        }
        // the row is n_k_tiles * 18 bytes; super-block kt / 8 starts 144 * (kt / 8) bytes in
        const uint32_t *sb = reinterpret_cast<const uint32_t *>(flat + (n * n_k_tiles + (kt & ~7)) * kQ4KBytesPer32);
        const int j = (int)(kt & 7), jj = j & 3;
        const uint32_t head = sb[0];
        const uint32_t b0 = (sb[1] >> (8 * jj)) & 0xFF, b1 = (sb[2] >> (8 * jj)) & 0xFF, b2 = (sb[3] >> (8 * jj)) & 0xFF;
        const uint32_t sc = j < 4 ? (b0 & 63) : ((b2 & 15) | ((b0 >> 6) << 4));
        const uint32_t m = j < 4 ? (b1 & 63) : ((b2 >> 4) | ((b1 >> 6) << 4));
        const uint32_t *qs = sb + 4 + 8 * (j >> 1);            // 32 bytes, nibble j & 1
        const int sh = 4 * (j & 1);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t c = (qs[k] >> sh) & 0x0F0F0F0Fu;    // elements 4k..4k+3, one per byte
            t[(2 * k) * 32 + r] = (uint8_t)((c & 15) | ((c >> 4) & 0xF0));
            t[(2 * k + 1) * 32 + r] = (uint8_t)(((c >> 16) & 15) | ((c >> 20) & 0xF0));
        }
        const float d = __half2float(__ushort_as_half((unsigned short)(head & 0xFFFF)));
        const float dmin = __half2float(__ushort_as_half((unsigned short)(head >> 16)));
        const uint32_t dp = __half_as_ushort(__float2half_rn(__fmul_rn(d, (float)sc)));
        const uint32_t mp = __half_as_ushort(__float2half_rn(-__fmul_rn(dmin, (float)m)));
        *reinterpret_cast<uint32_t *>(t + kScale4Off + 4 * r) = dp | (mp << 16);
    }
    __threadfence();
}

template <int TYPE>
__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t *__restrict__ tiled, int64_t n_k_tiles, int64_t N,
                                                     uint8_t *__restrict__ flat) {
    constexpr bool k8 = (TYPE == QMM_Q8_0);
    constexpr bool mx = (TYPE == QMM_MXFP4);
    constexpr bool q41 = (TYPE == QMM_Q4_1);
    constexpr int bb = k8 ? kBlock8Bytes : (mx ? kBlockMxBytes : (q41 ? kBlock41Bytes : kBlock4Bytes));
    constexpr int ts = TileFmt<TYPE>::kBytes;
    constexpr int soff = TileFmt<TYPE>::kScaleOff;
    const int64_t total = N * n_k_tiles;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / n_k_tiles, kt = i - n * n_k_tiles;
        const int64_t ct = n >> 5;
        const int r = (int)(n & 31);
        if (!QMM_DCHECK(n < N && kt < n_k_tiles)) continue;
        const uint8_t *t = tiled + (ct * n_k_tiles + kt) * ts;
        if (mx) {
            uint8_t *b8 = flat + i * bb;
            b8[0] = t[soff + r];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                // element j is the low nibble of byte j, element j + 16 its high nibble
                const uint32_t lo = (t[(j >> 1) * 32 + r] >> (4 * (j & 1))) & 15;
                const uint32_t hi = (t[((j + 16) >> 1) * 32 + r] >> (4 * (j & 1))) & 15;
                b8[1 + j] = (uint8_t)(lo | (hi << 4));
            }
            continue;
        }
        uint16_t *blk = reinterpret_cast<uint16_t *>(flat + i * bb);
        if (q41) {
            *reinterpret_cast<uint32_t *>(blk) = *reinterpret_cast<const uint32_t *>(t + soff + 4 * r);   // d, m
            blk += 1;                                   // the quants follow 4 bytes in, as for 2 below
        } else {
            blk[0] = (uint16_t)ld_u16(t + soff + 2 * r);
        }
        if (k8) {
#pragma unroll
            for (int cp = 0; cp < 16; ++cp) blk[1 + cp] = (uint16_t)ld_u16(t + cp * 64 + 2 * r);
        } else {
            uint32_t codes[32];
#pragma unroll
            for (int cp = 0; cp < 16; ++cp) {
                const uint32_t b = t[cp * 32 + r];
                codes[2 * cp] = b & 15;
                codes[2 * cp + 1] = b >> 4;
            }
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const uint32_t lo = codes[j] | (codes[j + 16] << 4);
                const uint32_t hi = codes[j + 1] | (codes[j + 17] << 4);
                blk[1 + j / 2] = (uint16_t)(lo | (hi << 8));
            }
        }
    }
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    if (g > 152 * 16) g = 152 * 16;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace

cudaError_t launch_repack(qmm_type t, const uint8_t *flat, int64_t K, int64_t N, uint8_t *tiled, cudaStream_t s) {
    const int64_t nkt = K / 32, nct = (N + 31) / 32;
    const int64_t n_tiles = nkt * nct;
    const int threads = 256;
    const int grid = grid_for(n_tiles * 32, threads);
    switch (t) {
        case QMM_Q4_0: repack_kernel<QMM_Q4_0><<<grid, threads, 0, s>>>(flat, nkt, N, n_tiles, tiled); break;
        case QMM_IQ4_NL: repack_kernel<QMM_IQ4_NL><<<grid, threads, 0, s>>>(flat, nkt, N, n_tiles, tiled); break;
        case QMM_MXFP4: repack_kernel<QMM_MXFP4><<<grid, threads, 0, s>>>(flat, nkt, N, n_tiles, tiled); break;
        case QMM_Q4_1: repack_kernel<QMM_Q4_1><<<grid, threads, 0, s>>>(flat, nkt, N, n_tiles, tiled); break;
        case QMM_Q4_K: repack_q4k_kernel<<<grid, threads, 0, s>>>(flat, nkt, N, n_tiles, tiled); break;
        default: repack_kernel<QMM_Q8_0><<<grid, threads, 0, s>>>(flat, nkt, N, n_tiles, tiled); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_unpack(qmm_type t, const uint8_t *tiled, int64_t K, int64_t N, uint8_t *flat, cudaStream_t s) {
    const int64_t nkt = K / 32;
    const int threads = 256;
    const int grid = grid_for(N * nkt, threads);
    switch (t) {
        case QMM_Q4_0: unpack_kernel<QMM_Q4_0><<<grid, threads, 0, s>>>(tiled, nkt, N, flat); break;
        case QMM_IQ4_NL: unpack_kernel<QMM_IQ4_NL><<<grid, threads, 0, s>>>(tiled, nkt, N, flat); break;
        case QMM_MXFP4: unpack_kernel<QMM_MXFP4><<<grid, threads, 0, s>>>(tiled, nkt, N, flat); break;
        case QMM_Q4_1: unpack_kernel<QMM_Q4_1><<<grid, threads, 0, s>>>(tiled, nkt, N, flat); break;
        case QMM_Q4_K: return cudaErrorNotSupported;           // tiles hold rounded products
        default: unpack_kernel<QMM_Q8_0><<<grid, threads, 0, s>>>(tiled, nkt, N, flat); break;
    }
    return cudaGetLastError();
}

QMM_DCHECK_READER(read_dcheck_repack)

}  // namespace qmm

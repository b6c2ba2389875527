// quant.cu -- activation quantization (hot path) and weight quantization (model-load helper).
//
// Activation rule (dynamic Q8_0, per 32 elements): amax = max|x|, d = amax/127, id = d ? 1/d : 0,
// q = round-half-away(x*id) clamped to [-127,127] (NaN product -> 0), stored scale fp16(d).
// Every operation is an IEEE-rounded fp32 intrinsic (__fdiv_rn, __frcp_rn-free 1/d via __fdiv_rn,
// __fmul_rn, __fadd_rn), so nvcc cannot contract or reassociate them.
// Weight rules (test data and load time; stated with qmm_quantize_weight in qmm.h): Q4_0, Q8_0,
// IQ4_NL, MXFP4 and Q4_1 per 32-element block (one thread per block), Q4_K per 256-element
// super-block (one warp per super-block).
#include "qmm_internal.cuh"

namespace qmm {
namespace {

// 8 threads per 32-element block, 4 consecutive elements per thread.  Grid-stride over all
// M*K/4 element quads.  `vec` selects float4 loads (x 16-byte aligned, ldx % 4 == 0).
template <bool vec>
__global__ void __launch_bounds__(256) quantize_act_kernel(const float *__restrict__ x, int64_t M, int64_t K,
                                                           int64_t ldx, int8_t *__restrict__ a_q,
                                                           uint16_t *__restrict__ a_d) {
    // This grid is launched as a programmatic dependent: x may be written by the grid before it on
    // the stream (and a_q / a_d still read by it), so wait for that grid to complete first.  Only
    // then let the dependent matmul start streaming weights: anything the earlier grids wrote, the
    // weights included, is visible by now.  The matmul still waits for this grid before it reads
    // a_q / a_d.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t quads_per_row = K / 4;
    const int64_t total = M * quads_per_row;
    const unsigned lane = threadIdx.x & 31u;
    // All 32 lanes of a warp stay in the loop together (total is a multiple of 8, and the
    // stride is a multiple of 32), so the group-of-8 shuffles below are always complete.
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < total; base += stride) {
        const int64_t i = base + lane;
        const bool active = i < total;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        int64_t m = 0, kq = 0;
        if (active && QMM_DCHECK(i / quads_per_row < M)) {
            m = i / quads_per_row;
            kq = (i - m * quads_per_row) * 4;
            const float *p = x + m * ldx + kq;
            if (vec) {
                v = __ldg(reinterpret_cast<const float4 *>(p));
            } else {
                v.x = __ldg(p); v.y = __ldg(p + 1); v.z = __ldg(p + 2); v.w = __ldg(p + 3);
            }
        }
        float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        if (active) {
            const float d = q8_scale(amax);
            const float id = inv_or_zero(d);
            const uint32_t packed = (uint32_t)(q8_code(v.x, id) & 0xFF) | ((uint32_t)(q8_code(v.y, id) & 0xFF) << 8) |
                                    ((uint32_t)(q8_code(v.z, id) & 0xFF) << 16) |
                                    ((uint32_t)(q8_code(v.w, id) & 0xFF) << 24);
            // block kq / 32 < K / 32 of row m < M
            if (QMM_DCHECK(m < M && kq + 4 <= K)) {
                *reinterpret_cast<uint32_t *>(a_q + m * K + kq) = packed;
                if ((lane & 7u) == 0) a_d[m * (K / 32) + kq / 32] = __half_as_ushort(__float2half_rn(d));
            }
        }
    }
}

// One thread per flat output block (32 input elements).  Model-load helper: simple, not tuned.
__global__ void __launch_bounds__(128) quantize_weight_kernel(int type, const float *__restrict__ w, int64_t N,
                                                              int64_t K, int64_t ldw, uint8_t *__restrict__ flat,
                                                              Lut16 lut) {
    const int64_t nb = K / 32;
    const int64_t total = N * nb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / nb, b = i - n * nb;
        const float *x = w + n * ldw + b * 32;
        float xs[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 v = __ldg(reinterpret_cast<const float4 *>(x + j));
            xs[j] = v.x; xs[j + 1] = v.y; xs[j + 2] = v.z; xs[j + 3] = v.w;
        }
        float amax = 0.0f, m = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (fabsf(xs[j]) > amax) { amax = fabsf(xs[j]); m = xs[j]; }
        }
        if (type == QMM_MXFP4) {
            // e = floor(log2 amax) - 2 + 127 (0 for an all-zero block, at most 254); each code the
            // nearest level s * fp4(code) under the dequantizing fp16 scale s, lowest code on ties
            int e = 0;
            if (amax > 0.0f) {
                int ex;
                (void)frexpf(amax, &ex);
                e = (ex - 1) - 2 + 127;
                e = e < 0 ? 0 : (e > 254 ? 254 : e);
            }
            const float s = 2.0f * mx_half_scale((uint32_t)e);                 // exact power of two (or 0)
            uint8_t *blk = flat + i * kBlockMxBytes;
            int codes[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                int best = 0;
                float best_err = INFINITY;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float level = __fmul_rn(s, __fmul_rn(0.5f, (float)lut.v[q]));   // lut: doubled FP4 values
                    const float err = fabsf(__fsub_rn(xs[j], level));
                    if (err < best_err) { best_err = err; best = q; }
                }
                codes[j] = best;
            }
            blk[0] = (uint8_t)e;
#pragma unroll
            for (int j = 0; j < 16; ++j) blk[1 + j] = (uint8_t)((codes[j] & 15) | ((codes[j + 16] & 15) << 4));
            continue;
        }
        if (type == QMM_Q4_1) {
            // d = (max - min)/15, q = min(15, trunc((x - min)*(1/d) + 0.5)), m = min
            float mn = xs[0], mx = xs[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) {
                mn = xs[j] < mn ? xs[j] : mn;
                mx = xs[j] > mx ? xs[j] : mx;
            }
            const float d = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
            const float id = inv_or_zero(d);
            int codes[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float v = __fadd_rn(__fmul_rn(__fsub_rn(xs[j], mn), id), 0.5f);
                int c;
                if (!(v >= 0.0f)) c = 0;                 // NaN
                else if (v >= 15.0f) c = 15;
                else c = __float2int_rz(v);
                codes[j] = c;
            }
            uint16_t *out = reinterpret_cast<uint16_t *>(flat + i * kBlock41Bytes);   // 4-byte aligned
            out[0] = __half_as_ushort(__float2half_rn(d));
            out[1] = __half_as_ushort(__float2half_rn(mn));
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const uint32_t b0 = (uint32_t)(codes[j] & 15) | ((uint32_t)(codes[j + 16] & 15) << 4);
                const uint32_t b1 = (uint32_t)(codes[j + 1] & 15) | ((uint32_t)(codes[j + 17] & 15) << 4);
                out[2 + j / 2] = (uint16_t)(b0 | (b1 << 8));
            }
            continue;
        }
        const int bb = (type == QMM_Q8_0) ? kBlock8Bytes : kBlock4Bytes;
        uint16_t *out = reinterpret_cast<uint16_t *>(flat + i * bb);   // 2-byte aligned
        int codes[32];
        float d;
        if (type == QMM_Q8_0) {
            d = q8_scale(amax);
            const float id = inv_or_zero(d);
#pragma unroll
            for (int j = 0; j < 32; ++j) codes[j] = q8_code(xs[j], id);
            out[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
            for (int j = 0; j < 32; j += 2) out[1 + j / 2] = (uint16_t)((codes[j] & 0xFF) | ((codes[j + 1] & 0xFF) << 8));
            continue;
        }
        if (type == QMM_Q4_0) {
            d = __fdiv_rn(m, -8.0f);
            const float id = inv_or_zero(d);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float v = __fadd_rn(__fmul_rn(xs[j], id), 8.5f);
                int c;
                if (!(v >= 0.0f)) c = 0;                 // NaN or negative
                else if (v >= 15.0f) c = 15;
                else c = __float2int_rz(v);              // truncation toward zero
                codes[j] = c;
            }
            out[0] = __half_as_ushort(__float2half_rn(d));
        } else {
            d = __fdiv_rn(m, (float)lut.v[0]);
            const __half d16 = __float2half_rn(d);
            const float ds = __half2float(d16);
            float levels[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) levels[q] = __fmul_rn(ds, (float)lut.v[q]);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                int best = 0;
                float best_err = INFINITY;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float e = fabsf(__fsub_rn(xs[j], levels[q]));
                    if (e < best_err) { best_err = e; best = q; }
                }
                codes[j] = best;
            }
            out[0] = __half_as_ushort(d16);
        }
        // nibble byte j holds element j (low) and element j+16 (high)
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            const uint32_t b0 = (uint32_t)(codes[j] & 15) | ((uint32_t)(codes[j + 16] & 15) << 4);
            const uint32_t b1 = (uint32_t)(codes[j + 1] & 15) | ((uint32_t)(codes[j + 17] & 15) << 4);
            out[1 + j / 2] = (uint16_t)(b0 | (b1 << 8));
        }
    }
}

// Q4_K super-blocks (the rule stated with qmm_quantize_weight): one warp per 256 weights, lane l
// holding element l of each of the 8 sub-blocks.  Sub-block minima and maxima come from warp
// reductions (min and max do not depend on the order; the range is taken as +0 when it is not
// positive, so the sign of a zero maximum cannot matter); everything after that is the same fp32
// arithmetic in every lane, in the order of the rule.
__global__ void __launch_bounds__(128) quantize_q4k_kernel(const float *__restrict__ w, int64_t N, int64_t K, int64_t ldw,
                                                           uint8_t *__restrict__ flat) {
    const int64_t nsb = K / 256, total = N * nsb;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < total; i += nwarps) {
        const int64_t n = i / nsb, sbi = i - n * nsb;
        const float *x = w + n * ldw + sbi * 256;
        uint8_t *sb = flat + i * kSuperQ4KBytes;            // row n, super-block sbi
        float xv[8], scale[8], mins[8];
        float max_scale = 0.0f, max_min = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            xv[j] = x[32 * j + lane];
            float mn = xv[j] < 0.0f ? xv[j] : 0.0f, mx = xv[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float a = __shfl_xor_sync(0xffffffffu, mn, o), b = __shfl_xor_sync(0xffffffffu, mx, o);
                mn = a < mn ? a : mn;
                mx = b > mx ? b : mx;
            }
            float range = __fsub_rn(mx, mn);
            if (!(range > 0.0f)) range = 0.0f;
            scale[j] = __fdiv_rn(range, 15.0f);
            mins[j] = __fsub_rn(0.0f, mn);
            if (scale[j] > max_scale) max_scale = scale[j];
            if (mins[j] > max_min) max_min = mins[j];
        }
        const float isc = max_scale > 0.0f ? __fdiv_rn(63.0f, max_scale) : 0.0f;
        const float imn = max_min > 0.0f ? __fdiv_rn(63.0f, max_min) : 0.0f;
        const __half d16 = __float2half_rn(__fdiv_rn(max_scale, 63.0f));
        const __half dmin16 = __float2half_rn(__fdiv_rn(max_min, 63.0f));
        int sc[8], m[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float vs = __fadd_rn(__fmul_rn(scale[j], isc), 0.5f), vm = __fadd_rn(__fmul_rn(mins[j], imn), 0.5f);
            sc[j] = !(vs >= 0.0f) ? 0 : (vs >= 63.0f ? 63 : __float2int_rz(vs));
            m[j] = !(vm >= 0.0f) ? 0 : (vm >= 63.0f ? 63 : __float2int_rz(vm));
        }
        const float d = __half2float(d16), dmin = __half2float(dmin16);
        int codes[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float D = __fmul_rn(d, (float)sc[j]), Mj = __fmul_rn(dmin, (float)m[j]);
            const float v = __fadd_rn(__fmul_rn(__fadd_rn(xv[j], Mj), inv_or_zero(D)), 0.5f);
            codes[j] = !(v >= 0.0f) ? 0 : (v >= 15.0f ? 15 : __float2int_rz(v));
        }
        // quant byte 32g + l: sub-block 2g in the low nibble, 2g + 1 in the high nibble
#pragma unroll
        for (int g = 0; g < 4; ++g) sb[16 + 32 * g + lane] = (uint8_t)(codes[2 * g] | (codes[2 * g + 1] << 4));
        if (lane == 0) {
            uint32_t s0 = 0, s1 = 0, s2 = 0;                 // scale bytes 0..3, 4..7, 8..11
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                s0 |= (uint32_t)((sc[q] & 63) | ((sc[q + 4] >> 4) << 6)) << (8 * q);
                s1 |= (uint32_t)((m[q] & 63) | ((m[q + 4] >> 4) << 6)) << (8 * q);
                s2 |= (uint32_t)((sc[q + 4] & 15) | ((m[q + 4] & 15) << 4)) << (8 * q);
            }
            uint32_t *h = reinterpret_cast<uint32_t *>(sb);   // 4-byte aligned
            h[0] = (uint32_t)__half_as_ushort(d16) | ((uint32_t)__half_as_ushort(dmin16) << 16);
            h[1] = s0;
            h[2] = s1;
            h[3] = s2;
        }
    }
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    if (g > 152 * 32) g = 152 * 32;
    if (g < 1) g = 1;
    return (int)g;
}

// Copies M fp32 rows (row stride ldx) from page-locked host memory into the dense device buffer
// dst [M][K]: each byte crosses NVLink-C2C once (a kernel reading host rows from every CTA pays the
// link once per CTA).  Launched as a programmatic dependent.  It lets the dependent decode kernel
// launch at once, so that the decode's CTAs take the SMs as the grid before this one leaves them
// and start streaming weights (the decode waits for this grid before it reads dst or writes y);
// then it waits for the grid before it before it reads x or writes dst.
template <bool vec>
__global__ void __launch_bounds__(256) stage_rows_kernel(const float *__restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                         float *__restrict__ dst) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t quads_per_row = K / 4;
    const int64_t total = M * quads_per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / quads_per_row, k = (i - m * quads_per_row) * 4;
        if (!QMM_DCHECK(m < M && k + 4 <= K)) continue;
        const float *src = x + m * ldx + k;
        float4 v;
        if constexpr (vec) {
            v = *reinterpret_cast<const float4 *>(src);
        } else {
            v = make_float4(src[0], src[1], src[2], src[3]);
        }
        *reinterpret_cast<float4 *>(dst + m * K + k) = v;
    }
}

}  // namespace

cudaError_t launch_stage_rows(const float *x, int64_t M, int64_t K, int64_t ldx, float *dst, cudaStream_t s) {
    const int threads = 256;
    const int grid = grid_for(M * (K / 4), threads);
    const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) && (ldx % 4 == 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec) return cudaLaunchKernelEx(&cfg, stage_rows_kernel<true>, x, M, K, ldx, dst);
    return cudaLaunchKernelEx(&cfg, stage_rows_kernel<false>, x, M, K, ldx, dst);
}

cudaError_t launch_quantize_act(const float *x, int64_t M, int64_t K, int64_t ldx, int8_t *a_q, uint16_t *a_d,
                                cudaStream_t s) {
    const int threads = 256;
    const int64_t quads = M * (K / 4);
    const int grid = grid_for(quads, threads);
    const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) && (ldx % 4 == 0);
    // programmatic dependent launch: the launch overlaps the tail of the grid before it on the stream
    // (if that grid allows it); the kernel waits for that grid before touching memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec) return cudaLaunchKernelEx(&cfg, quantize_act_kernel<true>, x, M, K, ldx, a_q, a_d);
    return cudaLaunchKernelEx(&cfg, quantize_act_kernel<false>, x, M, K, ldx, a_q, a_d);
}

cudaError_t launch_quantize_weight(qmm_type t, const float *w, int64_t N, int64_t K, int64_t ldw, uint8_t *flat,
                                   cudaStream_t s) {
    const int threads = 128;
    if (t == QMM_Q4_K) {
        quantize_q4k_kernel<<<grid_for(N * (K / 256) * 32, threads), threads, 0, s>>>(w, N, K, ldw, flat);
        return cudaGetLastError();
    }
    const int grid = grid_for(N * (K / 32), threads);
    quantize_weight_kernel<<<grid, threads, 0, s>>>((int)t, w, N, K, ldw, flat, lut_for(t));
    return cudaGetLastError();
}

QMM_DCHECK_READER(read_dcheck_quant)

}  // namespace qmm

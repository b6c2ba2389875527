// gemm_tc.cu -- prefill-shaped matmul on tcgen05 tensor cores (placeholder until the kernel lands).
#include "qmm_internal.cuh"

namespace qmm {

namespace {
__device__ unsigned g_device_status = 0;   // set by pipelined kernels when a bounded wait gives up
}

cudaError_t launch_gemm(qmm_type, const uint8_t *, int64_t, int64_t, const int8_t *, const uint16_t *, int64_t,
                        float *, int64_t, cudaStream_t) {
    return cudaErrorNotSupported;
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

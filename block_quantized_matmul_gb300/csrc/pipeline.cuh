// pipeline.cuh -- shared-memory pipeline primitives used by the decode kernels and the GEMM:
// mbarrier set-up, arrivals and bounded waits, and the bulk / tensor copies that complete on them.
//
// Every wait is bounded: it gives up after a time limit (or as soon as another warp of the CTA has
// given up), records that in the calling kernel family's device status word and lets the kernel
// finish, so a broken pipeline surfaces as QMM_ERR_TIMEOUT on the host instead of a hung GPU.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace qmm {
namespace pipe {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s per wait

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

// Slow path of a bounded wait: polls until the phase completes (true), or until `abort` is raised by
// another warp or limit_ns has passed (false); on its own time-out it raises `abort` and sets bit 0
// of *status.  The timer and the flag are read only every 64 polls.
inline __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort, unsigned *status,
                                              unsigned long long limit_ns) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort = 1;
                atomicOr(status, 1u);
                return false;
            }
        }
    }
}
// The fast path (phase already complete) inline, the rest in wait_slow.
__device__ __forceinline__ bool wait_bounded_on(uint32_t bar, uint32_t parity, volatile int *abort, unsigned *status,
                                                unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort, status, limit_ns);
}

// Wait used while draining after an abort: no abort check, a quarter of the limit, never raises.
inline __device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs / 4) return;
    }
}

// ---- thread-block clusters: rank, peer shared-memory addresses, remote arrivals ----
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}
// The shared::cluster address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(rank));
    return a;
}
__device__ __forceinline__ void st_peer_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// Arrival on a barrier of a CTA of this cluster, releasing this thread's prior writes (and those it
// has synchronised with) at cluster scope.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for a phase completed by arrivals from other CTAs of the cluster (acquire at cluster
// scope); gives up as wait_slow does.
inline __device__ __noinline__ bool wait_cluster_bounded(uint32_t bar, uint32_t parity, volatile int *abort, unsigned *status,
                                                         unsigned long long limit_ns) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort = 1;
                atomicOr(status, 1u);
                return false;
            }
        }
    }
}

// 1-D bulk copy global -> shared, completing `bytes` on the mbarrier (addresses and size 16-byte
// multiples).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// 2-D tensor copy of one box of `map` at element coordinates (x, y) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

}  // namespace pipe
}  // namespace qmm

// Tensor-memory-accelerator (TMA) staging of the scan kernels' tiles: 3-D
// tensor maps over the [B, L, D] and [B, L, N] tensors, bulk copies into
// shared memory issued by one thread, completion on an mbarrier, and a
// time-limited wait that reports instead of hanging.
//
// A TMA copy moves a tile without any of the block's threads touching it, so
// the copies take neither issue slots nor the shared-memory data pipe of the
// SM (unlike per-thread asynchronous copies); out-of-range rows and channels
// of a box are filled with zeros.
#pragma once

#include <cuda.h>  // CUtensorMap (the type only; maps are encoded on the host)
#include <stdint.h>

namespace ss {

// Tensor maps a scan kernel loads its tiles through (passed by value as a
// __grid_constant__ parameter).  The forward uses delta, u, z, B, C; the
// backward also dy and the forward's pre-gate readout y0.
enum { kMapDelta = 0, kMapU, kMapZ, kMapDy, kMapY0, kMapB, kMapC, kMaps };
struct TmaMaps {
    CUtensorMap m[kMaps];
};

// Bits a kernel sets in the library's device status word (ss_device_status
// reads and clears it): it gave up waiting for a copy ...
constexpr int kDevWaitTimeout = 1;
// ... or found its TMA buffers off the 128-byte alignment the copies need (it
// staged with per-thread copies instead; its results are intact).
constexpr int kDevMisaligned = 2;

// Limit of every wait on a copy: a tile arrives within microseconds, so a wait
// that outlasts two seconds has failed.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Destination of a TMA box: 128-byte aligned shared memory.
__device__ __forceinline__ bool smem_aligned128(const void* p) { return (smem_addr(p) & 127u) == 0; }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make initialized barriers (generic-proxy writes) visible to the TMA unit.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Arrive on the barrier and add `bytes` to the bytes it waits for.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// One box of a 3-D tensor map at coordinates (x, y, z) into shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// A contiguous run of `bytes` (a multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the barrier's phase `phase` completes, at most limit_ns; false
// when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, phase)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, phase)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

}  // namespace ss

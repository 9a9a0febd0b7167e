// flag_ops.cuh -- memory operations of the Data-as-Flag kernels (sp.cu, tff.cu)
// and of the split small-batch dispatch (fused.cu): flags stored with release
// and loaded with acquire at GPU scope, a bounded warp-wide wait on a flag, and
// coherent 16-byte loads of data another CTA may still be writing.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace ep {
namespace {

__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits, by the whole warp, until *flag is non-zero: every lane polls with an
// acquire load (so each lane's later loads are ordered after the flag's
// release), sleeping briefly between polls. Bounded: false after max_polls
// polls without seeing the flag set.
__device__ __forceinline__ bool warp_wait_flag(const unsigned *flag, uint32_t max_polls) {
    bool seen = false;
    for (uint32_t polls = 0; polls <= max_polls; ++polls) {
        if (ld_acquire_u32(flag) != 0u) {
            seen = true;
            break;
        }
        __nanosleep(32);
    }
    return __all_sync(0xffffffffu, seen);
}

// Relaxed (coherent, GPU-scope) 16-byte load: sees a concurrent writer's data.
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint4 *p) {
    uint4 r;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}

}  // namespace
}  // namespace ep

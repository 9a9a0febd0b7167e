// ep_internal.cuh -- shared declarations of the CUDA side of the C ABI.
//
// Kernels live in route.cu, layout.cu, dispatch.cu and combine.cu; each file
// exposes one host launcher declared here. The C entry points in ep_api.cu
// validate arguments, then call the launchers.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/ep.h"

namespace ep {

constexpr int kFullMask = -1;  // all 32 lanes (as unsigned in shuffles)

// Layout tiling: a layout CTA owns kLayoutTokens consecutive tokens, 32 per warp.
constexpr int kLayoutWarps = 8;
constexpr int kLayoutTokens = 32 * kLayoutWarps;

constexpr int kMaxDevices_ = 64;  // device ordinals with cached attributes

// Largest shapes the kernels are built for.
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxGroups = 32;

inline int64_t layout_blocks(int64_t T) { return (T + kLayoutTokens - 1) / kLayoutTokens; }

// Workspace carve-up for ep_layout (all offsets 256-byte aligned).
struct LayoutWorkspace {
    size_t block_counts_off;  // int32 [E][nb]: per-CTA expert histograms, then their exclusive scan
    size_t bytes;
};
LayoutWorkspace layout_workspace(int64_t T, int32_t E);

// Cached device properties (per device ordinal).
int sm_count(int device);
int current_device_sm_count();
// Resident CTAs per SM for a kernel (cached per kernel, device and launch shape).
int max_blocks_per_sm(const void *fn, int threads, size_t smem);

cudaError_t launch_route(const ep_config &c, const float *logits, int32_t *idx, float *w, cudaStream_t s);

cudaError_t launch_layout(const ep_config &c, int32_t W, const int32_t *idx, int32_t *expert_count,
                          int32_t *expert_offset, int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                          ep_chunk *chunks, int32_t *n_chunks, int32_t *worker_begin, void *workspace,
                          cudaStream_t s);

cudaError_t launch_dispatch(const ep_config &c, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send,
                            int32_t *meta, cudaStream_t s);

cudaError_t launch_combine(const ep_config &c, const ep_bf16 *y, const int32_t *slot, const float *w,
                           ep_bf16 *out, cudaStream_t s);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// 16-byte streaming load that does not allocate in L1 (data read once).
__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(uint4 *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

}  // namespace ep

// ep_internal.cuh -- shared declarations of the CUDA side of the C ABI.
//
// Kernels live in route.cu, layout.cu, dispatch.cu, combine.cu, fused.cu,
// gather.cu, sp.cu and tff.cu; each file exposes its host launchers, declared
// here. The C entry points in ep_api.cu validate arguments, then call the
// launchers.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ep.h"

namespace ep {

// The hop tiers the chunk schedule classes ranks by (ep_config fields).
struct HopTiers {
    int32_t ranks_per_node, ranks_per_pod, self_rank;
};
inline HopTiers hop_tiers(const ep_config &c) { return HopTiers{c.ranks_per_node, c.ranks_per_pod, c.self_rank}; }
inline int hop_classes(const ep_config &c) { return c.ranks_per_pod > 0 ? 3 : 2; }

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

// Workspace carve-up for ep_layout. The single-kernel layout uses a [CTA][E]
// count table of table_words 32-bit words at block_counts_off, which must be
// zero when it starts; the fallback path uses [E][ceil(T/256)] counts there.
struct LayoutWorkspace {
    size_t block_counts_off;
    size_t table_words;
    size_t bytes;
};
LayoutWorkspace layout_workspace(const ep_config &c);

// The current device's ordinal, checked against the per-device caches
// (cudaErrorInvalidDevice beyond them).
inline cudaError_t current_device(int *dev) {
    const cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    return (*dev < 0 || *dev >= kMaxDevices_) ? cudaErrorInvalidDevice : cudaSuccess;
}

// Cached device properties (per device ordinal).
int sm_count(int device);
int current_device_sm_count();
// Resident CTAs per SM for a kernel (cached per kernel, device and launch shape).
int max_blocks_per_sm(const void *fn, int threads, size_t smem);

// za / zb: optional words (na / nb of them) the route kernel sets to zero for
// kernels that follow it in the same call sequence (za spread over all its
// CTAs, zb by its first CTA: nb <= 256).
// zc: optional int32 word the route kernel also sets to zero.
cudaError_t launch_route(const ep_config &c, const float *logits, int32_t *idx, float *w, cudaStream_t s,
                         unsigned *za = nullptr, int na = 0, unsigned *zb = nullptr, int nb = 0,
                         int32_t *zc = nullptr);

// Whether every CTA of the route kernel for c is resident at once on the current device.
bool route_one_wave(const ep_config &c);

// table_zeroed: the caller already zeroed the single-kernel layout's count
// table (layout_workspace(c).table_words words at the workspace's start), so
// no memset is enqueued.
// defer_schedule: when the layout runs as the single cooperative kernel, leave
// the chunk schedule to the caller (*deferred = true; chunks, n_chunks and
// worker_begin are then not written, except n_chunks = -1 on failure).
// after_route: the single-kernel layout follows the route kernel in the same
// stream and is launched as its programmatic dependent.
// zero_ctr: a word the single-kernel layout zeroes before a dependent grid
// can start (the bulk dispatch's token counter).
cudaError_t launch_layout(const ep_config &c, int32_t W, const int32_t *idx, int32_t *expert_count,
                          int32_t *expert_offset, int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                          ep_chunk *chunks, int32_t *n_chunks, int32_t *worker_begin, void *workspace,
                          cudaStream_t s, bool table_zeroed = false, bool defer_schedule = false,
                          bool *deferred = nullptr, bool after_route = false, unsigned *zero_ctr = nullptr);

// Runs two CTAs into a grid barrier that expects three (a third arrives only
// after one gave up), one CTA into a wait on a flag nothing sets, and two
// through a count-table exchange whose second row is published only after the
// reader gave up; *gave_up counts the CTAs that stopped waiting after
// max_polls polls or learnt they came too late (5 when the bounds work), or is
// -1 if a late CTA missed the failure.
cudaError_t launch_bounded_wait_check(uint32_t max_polls, int32_t *gave_up, cudaStream_t s);

// Kernels launch_layout enqueues for c on the current device (1 fused, or 3).
int layout_kernel_count(const ep_config &c);

// ctr: optional device counter (4 bytes) for dynamic token assignment, zeroed
// here unless ctr_zeroed.
// after_layout: the launch follows the layout kernel in the same stream and may
// start while it runs (programmatic dependent launch; the kernel loads x rows
// first and reads the slots only after griddepcontrol.wait).
// A chunk schedule for one extra CTA of the bulk dispatch to build from
// rank_offset (after the layout grid it depends on), unless *n_chunks is -1.
struct ScheduleTask {
    const int32_t *rank_offset;
    ep_chunk *chunks;
    int32_t *n_chunks;
    int32_t *worker_begin;
    int32_t R, W;
    HopTiers tiers;
};
// sched: build that schedule in the dispatch kernel (bulk path only; see
// dispatch_uses_bulk).
cudaError_t launch_dispatch(const ep_config &c, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send,
                            int32_t *meta, cudaStream_t s, unsigned *ctr = nullptr, bool ctr_zeroed = false,
                            bool after_layout = false, const ScheduleTask *sched = nullptr);
bool dispatch_uses_bulk(const ep_config &c, const int32_t *slot);

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

// ---------------------------------------------------------------------------
// Bulk async copies (TMA, non-tensor form) and mbarriers, sm_90+ PTX.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Programmatic dependent launch. griddepcontrol.wait returns once the grids
// this one depends on have completed and their memory is visible (at once when
// there are none); launch_dependents lets the dependent grid start early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` as a programmatic dependent of the previous work in stream s
// (it must call grid_dependency_wait() before it touches memory the earlier
// kernels write or read).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Bounded wait on one mbarrier phase: false if it did not complete in time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t max_polls) {
    for (uint32_t i = 0; i < max_polls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        __nanosleep(32);
    }
    return false;
}

// global -> shared bulk copy completing on an mbarrier (dst, src, bytes 16-B aligned).
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 cache policies for the bulk copies' cache hints: keep (lines likely to be
// read again soon) or evict first (lines written once and not read back soon).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_g2s with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// bulk_s2g (below) with an L2 cache policy for the destination lines.
__device__ __forceinline__ void bulk_s2g_hint(void *dst, const void *src_smem, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(smem_u32(src_smem)), "r"(bytes), "l"(policy)
                 : "memory");
}

// shared -> global bulk copy, tracked by this thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src_smem)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Device-side error flags (bit values), one word per translation unit that
// can set them; ep_device_error() collects and clears them.
constexpr int32_t kErrDispatchWait = 1;  // a dispatch CTA gave up waiting for a bulk copy
constexpr int32_t kErrFusedWait = 2;     // a fused-dispatch CTA gave up waiting (barrier or bulk copy)
constexpr int32_t kErrSpWait = 4;        // a sentinel-polling CTA gave up waiting
constexpr int32_t kErrGatherWait = 8;    // a schedule-driven dispatch CTA gave up waiting (or a bad table)
cudaError_t dispatch_error_word(int32_t **addr);
cudaError_t fused_error_word(int32_t **addr);
cudaError_t sp_error_word(int32_t **addr);

// Schedule-driven dispatch (gather.cu).
int64_t gather_ctas(const ep_config &c, int32_t W);
cudaError_t launch_dispatch_scheduled(const ep_config &c, int32_t W, const ep_bf16 *x, const int32_t *slot,
                                      const ep_chunk *chunks, const int32_t *n_chunks, const int32_t *worker_begin,
                                      ep_bf16 *send, int32_t *meta, int64_t *cta_ns, cudaStream_t s);

// Data-as-Flag by Token-Flag Fusion: the 512-byte block codec (tff.cu).
int64_t tff_blocks_per_row(const ep_config &c);
cudaError_t launch_tff_encode(const ep_config &c, const ep_bf16 *rows, void *framed, unsigned epoch,
                              cudaStream_t s);
cudaError_t launch_tff_decode(const ep_config &c, const void *framed, unsigned epoch, ep_bf16 *rows,
                              unsigned *bad, cudaStream_t s);

// Data-as-Flag by sentinel polling (sp.cu).
cudaError_t launch_sentinel_arm(const ep_config &c, ep_bf16 *send, cudaStream_t s);
cudaError_t launch_expert_scale(const ep_config &c, const ep_bf16 *send, const int32_t *expert_offset,
                                const float *scale, ep_bf16 *y, cudaStream_t s);
cudaError_t launch_dispatch_expert_sp(const ep_config &c, int32_t W, const ep_bf16 *x, const int32_t *slot,
                                      const int32_t *expert_offset, const float *scale, const ep_chunk *chunks,
                                      const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send,
                                      int32_t *meta, ep_bf16 *y, cudaStream_t s);
cudaError_t launch_dispatch_expert_sw(const ep_config &c, int32_t W, const ep_bf16 *x, const int32_t *slot,
                                      const int32_t *expert_offset, const float *scale, const ep_chunk *chunks,
                                      const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send,
                                      int32_t *meta, ep_bf16 *y, unsigned *row_flag, unsigned epoch,
                                      cudaStream_t s);

// Fused route + layout + dispatch (fused.cu).
size_t fused_workspace_bytes(const ep_config &c);
// Kernels one ep_dispatch_fused call enqueues on the current device.
int fused_call_kernels(const ep_config &c);
cudaError_t launch_dispatch_fused(const ep_config &c, int32_t W, const float *logits, const ep_bf16 *x,
                                  int32_t *topk_idx, float *topk_w, int32_t *expert_count, int32_t *expert_offset,
                                  int32_t *rank_count, int32_t *rank_offset, int32_t *slot, ep_chunk *chunks,
                                  int32_t *n_chunks, int32_t *worker_begin, ep_bf16 *send, int32_t *meta,
                                  void *workspace, cudaStream_t s);

}  // namespace ep

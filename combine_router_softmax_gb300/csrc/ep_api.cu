// ep_api.cu -- the extern "C" entry points declared in include/ep.h.
//
// Every entry point checks its arguments on the host and returns a status
// before anything is enqueued; only then does it call the launcher of its
// kernels. Nothing here allocates device memory or synchronises.
#include <mutex>

#include "ep_internal.cuh"

namespace ep {

namespace {
constexpr int kMaxDevices = kMaxDevices_;
std::atomic<int> g_sm_count[kMaxDevices];  // zero-initialised: not yet queried

struct OccEntry {
    const void *fn;
    int dev;
    int threads;
    size_t smem;
    int blocks;
};
std::mutex g_occ_mu;
OccEntry g_occ[64];
int g_occ_n = 0;
}  // namespace

int sm_count(int device) {
    if (device < 0 || device >= kMaxDevices) return 0;
    int v = g_sm_count[device].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
        g_sm_count[device].store(v, std::memory_order_relaxed);
    }
    return v;
}

int current_device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return sm_count(dev);
}

int max_blocks_per_sm(const void *fn, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(g_occ_mu);
    for (int i = 0; i < g_occ_n; ++i)
        if (g_occ[i].fn == fn && g_occ[i].dev == dev && g_occ[i].threads == threads && g_occ[i].smem == smem)
            return g_occ[i].blocks;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem) != cudaSuccess || b <= 0) {
        cudaGetLastError();
        b = 1;
    }
    if (g_occ_n < 64) g_occ[g_occ_n++] = OccEntry{fn, dev, threads, smem, b};
    return b;
}

}  // namespace ep

namespace {

using ep::kMaxE;
using ep::kMaxGroups;
using ep::kMaxK;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by all entry points.
ep_status check_config(const ep_config *c) {
    if (!c) return EP_ERR_INVALID_ARG;
    if (c->T < 0 || c->E <= 0 || c->R <= 0 || c->k <= 0 || c->n_groups <= 0 || c->topk_groups <= 0)
        return EP_ERR_INVALID_ARG;
    if (c->E % c->R != 0 || c->k > c->E || c->E % c->n_groups != 0 || c->topk_groups > c->n_groups)
        return EP_ERR_INVALID_ARG;
    if ((int64_t)c->topk_groups * (c->E / c->n_groups) < c->k) return EP_ERR_INVALID_ARG;
    if (c->renormalize != 0 && c->renormalize != 1) return EP_ERR_INVALID_ARG;
    if ((int64_t)c->T * c->k > INT32_MAX) return EP_ERR_INVALID_ARG;
    if (c->E > kMaxE || c->k > kMaxK || c->n_groups > kMaxGroups) return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

ep_status check_rows(const ep_config *c) {
    if (c->H <= 0) return EP_ERR_INVALID_ARG;
    if (c->H % 8 != 0) return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

ep_status check_schedule(const ep_config *c) {
    if (c->ranks_per_node <= 0 || c->self_rank < 0 || c->self_rank >= c->R || c->num_workers < 0)
        return EP_ERR_INVALID_ARG;
    if (c->ranks_per_pod < 0 || (c->ranks_per_pod > 0 && c->ranks_per_pod % c->ranks_per_node != 0))
        return EP_ERR_INVALID_ARG;
    return EP_OK;
}

ep_status resolve_workers(const ep_config *c, int32_t *W) {
    if (c->num_workers > 0) {
        *W = c->num_workers;
        return EP_OK;
    }
    const int sms = ep::current_device_sm_count();
    if (sms <= 0) return EP_ERR_CUDA;
    *W = sms;
    return EP_OK;
}

ep_status from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

}  // namespace

extern "C" {

const char *ep_status_string(int status) {
    switch (status) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG: bad argument (null pointer, size or alignment)";
        case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED: shape outside the built kernels";
        case EP_ERR_CUDA: return "EP_ERR_CUDA: CUDA launch or query failed";
        case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY: output table or workspace too small";
        default: return "EP_ERR_UNKNOWN";
    }
}

int ep_version(void) { return 100; }

ep_status ep_device_error(int32_t *flags) {
    if (!flags) return EP_ERR_INVALID_ARG;
    int32_t *words[3] = {nullptr, nullptr, nullptr};
    if (ep::dispatch_error_word(&words[0]) != cudaSuccess) return EP_ERR_CUDA;
    if (ep::fused_error_word(&words[1]) != cudaSuccess) return EP_ERR_CUDA;
    if (ep::sp_error_word(&words[2]) != cudaSuccess) return EP_ERR_CUDA;
    int32_t all = 0;
    for (int32_t *word : words) {
        int32_t v = 0;
        if (cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return EP_ERR_CUDA;
        if (v != 0 && cudaMemset(word, 0, sizeof v) != cudaSuccess) return EP_ERR_CUDA;
        all |= v;
    }
    *flags = all;
    return EP_OK;
}

ep_status ep_check_bounded_wait(int32_t max_polls, int32_t *gave_up, cudaStream_t stream) {
    if (max_polls <= 0 || !gave_up) return EP_ERR_INVALID_ARG;
    return from_cuda(ep::launch_bounded_wait_check((uint32_t)max_polls, gave_up, stream));
}

ep_status ep_dispatch_fused_workspace_size(const ep_config *cfg, size_t *bytes) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if (!bytes) return EP_ERR_INVALID_ARG;
    *bytes = ep::fused_workspace_bytes(*cfg);
    return EP_OK;
}

ep_status ep_layout_workspace_size(const ep_config *cfg, size_t *bytes) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if (!bytes) return EP_ERR_INVALID_ARG;
    *bytes = ep::layout_workspace(*cfg).bytes;
    return EP_OK;
}

ep_status ep_schedule_capacity(const ep_config *cfg, int32_t *capacity) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if (!capacity) return EP_ERR_INVALID_ARG;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    const int64_t cap = (int64_t)ep::hop_classes(*cfg) * W + cfg->R;
    if (cap > INT32_MAX) return EP_ERR_INVALID_ARG;
    *capacity = (int32_t)cap;
    return EP_OK;
}

ep_status ep_step_kernel_count(const ep_config *cfg, int32_t *kernels) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if (!kernels) return EP_ERR_INVALID_ARG;
    if (cfg->T == 0) {
        *kernels = 1;  // the layout's scan still runs
        return EP_OK;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    *kernels = 3 + ep::layout_kernel_count(*cfg);
    return EP_OK;
}

ep_status ep_fused_step_kernel_count(const ep_config *cfg, int32_t *kernels) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if (!kernels) return EP_ERR_INVALID_ARG;
    if (cfg->T == 0) {
        *kernels = 1;
        return EP_OK;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    *kernels = ep::fused_call_kernels(*cfg) + 1;  // + combine
    return EP_OK;
}

ep_status ep_route(const ep_config *cfg, const float *logits, int32_t *topk_idx, float *topk_w,
                   cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!logits || !topk_idx || !topk_w) return EP_ERR_INVALID_ARG;
    return from_cuda(ep::launch_route(*cfg, logits, topk_idx, topk_w, stream));
}

ep_status ep_layout(const ep_config *cfg, const int32_t *topk_idx, int32_t *expert_count, int32_t *expert_offset,
                    int32_t *rank_count, int32_t *rank_offset, int32_t *slot, ep_chunk *chunks,
                    int32_t chunk_capacity, int32_t *n_chunks, int32_t *worker_begin, void *workspace,
                    size_t workspace_bytes, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if (!expert_count || !expert_offset || !rank_count || !rank_offset || !chunks || !n_chunks || !worker_begin)
        return EP_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!topk_idx || !slot)) return EP_ERR_INVALID_ARG;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    if ((int64_t)chunk_capacity < (int64_t)ep::hop_classes(*cfg) * W + cfg->R) return EP_ERR_CAPACITY;
    const size_t need = ep::layout_workspace(*cfg).bytes;
    if (need > 0) {
        if (!workspace) return EP_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EP_ERR_INVALID_ARG;
        if (workspace_bytes < need) return EP_ERR_CAPACITY;
    }
    return from_cuda(ep::launch_layout(*cfg, W, topk_idx, expert_count, expert_offset, rank_count, rank_offset,
                                       slot, chunks, n_chunks, worker_begin, workspace, stream));
}

ep_status ep_dispatch_fused(const ep_config *cfg, const float *logits, const ep_bf16 *x, int32_t *topk_idx,
                            float *topk_w, int32_t *expert_count, int32_t *expert_offset, int32_t *rank_count,
                            int32_t *rank_offset, int32_t *slot, ep_chunk *chunks, int32_t chunk_capacity,
                            int32_t *n_chunks, int32_t *worker_begin, ep_bf16 *send, int32_t *slot_meta,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (!expert_count || !expert_offset || !rank_count || !rank_offset || !chunks || !n_chunks || !worker_begin)
        return EP_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!logits || !x || !topk_idx || !topk_w || !slot || !send || !slot_meta))
        return EP_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!aligned16(x) || !aligned16(send))) return EP_ERR_INVALID_ARG;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    if ((int64_t)chunk_capacity < (int64_t)ep::hop_classes(*cfg) * W + cfg->R) return EP_ERR_CAPACITY;
    const size_t need = ep::fused_workspace_bytes(*cfg);
    if (need > 0) {
        if (!workspace) return EP_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EP_ERR_INVALID_ARG;
        if (workspace_bytes < need) return EP_ERR_CAPACITY;
    }
    if (cfg->T == 0)
        return from_cuda(ep::launch_layout(*cfg, W, topk_idx, expert_count, expert_offset, rank_count, rank_offset,
                                           slot, chunks, n_chunks, worker_begin, workspace, stream));
    return from_cuda(ep::launch_dispatch_fused(*cfg, W, logits, x, topk_idx, topk_w, expert_count, expert_offset,
                                               rank_count, rank_offset, slot, chunks, n_chunks, worker_begin, send,
                                               slot_meta, workspace, stream));
}

ep_status ep_dispatch_scheduled_ctas(const ep_config *cfg, int32_t *ctas) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if (!ctas) return EP_ERR_INVALID_ARG;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    const int64_t n = ep::gather_ctas(*cfg, W);
    if (n > INT32_MAX) return EP_ERR_INVALID_ARG;
    *ctas = (int32_t)n;
    return EP_OK;
}

ep_status ep_dispatch_scheduled(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot, const ep_chunk *chunks,
                                const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send,
                                int32_t *slot_meta, int64_t *cta_ns, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!x || !slot || !chunks || !n_chunks || !worker_begin || !send || !slot_meta) return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(send) || (reinterpret_cast<uintptr_t>(cta_ns) & 7u)) return EP_ERR_INVALID_ARG;
    if (cfg->H * 2 > 48 * 1024) return EP_ERR_UNSUPPORTED;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    const cudaError_t e = ep::launch_dispatch_scheduled(*cfg, W, x, slot, chunks, n_chunks, worker_begin, send,
                                                        slot_meta, cta_ns, stream);
    if (e == cudaErrorNotSupported) return EP_ERR_UNSUPPORTED;
    return from_cuda(e);
}

ep_status ep_tff_framed_bytes(const ep_config *cfg, size_t *bytes) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (!bytes) return EP_ERR_INVALID_ARG;
    *bytes = (size_t)cfg->T * (size_t)cfg->k * (size_t)ep::tff_blocks_per_row(*cfg) * EP_TFF_BLOCK_BYTES;
    return EP_OK;
}

ep_status ep_tff_encode(const ep_config *cfg, const ep_bf16 *rows, void *framed, uint32_t epoch,
                        cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!rows || !framed || !aligned16(rows) || !aligned16(framed)) return EP_ERR_INVALID_ARG;
    if ((int64_t)cfg->T * cfg->k * ep::tff_blocks_per_row(*cfg) > INT32_MAX) return EP_ERR_UNSUPPORTED;
    return from_cuda(ep::launch_tff_encode(*cfg, rows, framed, epoch, stream));
}

ep_status ep_tff_decode(const ep_config *cfg, const void *framed, uint32_t epoch, ep_bf16 *rows,
                        uint32_t *bad_blocks, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!rows || !framed || !bad_blocks || !aligned16(rows) || !aligned16(framed) ||
        (reinterpret_cast<uintptr_t>(bad_blocks) & 3u))
        return EP_ERR_INVALID_ARG;
    if ((int64_t)cfg->T * cfg->k * ep::tff_blocks_per_row(*cfg) > INT32_MAX) return EP_ERR_UNSUPPORTED;
    return from_cuda(ep::launch_tff_decode(*cfg, framed, epoch, rows, bad_blocks, stream));
}

ep_status ep_sentinel_arm(const ep_config *cfg, ep_bf16 *send, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!send || !aligned16(send)) return EP_ERR_INVALID_ARG;
    return from_cuda(ep::launch_sentinel_arm(*cfg, send, stream));
}

ep_status ep_expert_scale(const ep_config *cfg, const ep_bf16 *send, const int32_t *expert_offset,
                          const float *expert_scale, ep_bf16 *y, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!send || !expert_offset || !expert_scale || !y) return EP_ERR_INVALID_ARG;
    if (!aligned16(send) || !aligned16(y)) return EP_ERR_INVALID_ARG;
    return from_cuda(ep::launch_expert_scale(*cfg, send, expert_offset, expert_scale, y, stream));
}

ep_status ep_dispatch_expert_sp(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot,
                                const int32_t *expert_offset, const float *expert_scale, const ep_chunk *chunks,
                                const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send,
                                int32_t *slot_meta, ep_bf16 *y, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!x || !slot || !expert_offset || !expert_scale || !chunks || !n_chunks || !worker_begin || !send ||
        !slot_meta || !y)
        return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(send) || !aligned16(y) || (reinterpret_cast<uintptr_t>(slot) & 15u))
        return EP_ERR_INVALID_ARG;
    if (cfg->k % 4 != 0 || cfg->H * 2 < 1024 || cfg->H * 2 > 48 * 1024) return EP_ERR_UNSUPPORTED;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    const cudaError_t e = ep::launch_dispatch_expert_sp(*cfg, W, x, slot, expert_offset, expert_scale, chunks,
                                                        n_chunks, worker_begin, send, slot_meta, y, stream);
    if (e == cudaErrorNotSupported) return EP_ERR_UNSUPPORTED;
    return from_cuda(e);
}

ep_status ep_dispatch_expert_sw(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot,
                                const int32_t *expert_offset, const float *expert_scale, const ep_chunk *chunks,
                                const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send,
                                int32_t *slot_meta, ep_bf16 *y, uint32_t *row_flag, uint32_t epoch,
                                cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!x || !slot || !expert_offset || !expert_scale || !chunks || !n_chunks || !worker_begin || !send ||
        !slot_meta || !y || !row_flag)
        return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(send) || !aligned16(y) || (reinterpret_cast<uintptr_t>(slot) & 15u) ||
        (reinterpret_cast<uintptr_t>(row_flag) & 3u))
        return EP_ERR_INVALID_ARG;
    if (cfg->k % 4 != 0 || cfg->H * 2 < 1024 || cfg->H * 2 > 48 * 1024) return EP_ERR_UNSUPPORTED;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    const cudaError_t e = ep::launch_dispatch_expert_sw(*cfg, W, x, slot, expert_offset, expert_scale, chunks,
                                                        n_chunks, worker_begin, send, slot_meta, y, row_flag, epoch,
                                                        stream);
    if (e == cudaErrorNotSupported) return EP_ERR_UNSUPPORTED;
    return from_cuda(e);
}

ep_status ep_dispatch(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send,
                      int32_t *slot_meta, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!x || !slot || !send || !slot_meta) return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(send)) return EP_ERR_INVALID_ARG;
    return from_cuda(ep::launch_dispatch(*cfg, x, slot, send, slot_meta, stream));
}

ep_status ep_combine(const ep_config *cfg, const ep_bf16 *y, const int32_t *slot, const float *topk_w,
                     ep_bf16 *out, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_rows(cfg)) != EP_OK) return st;
    if (cfg->T == 0) return EP_OK;
    if (!y || !slot || !topk_w || !out) return EP_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out)) return EP_ERR_INVALID_ARG;
    return from_cuda(ep::launch_combine(*cfg, y, slot, topk_w, out, stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// ep_layout_static: ep_layout with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory at call time and so cannot
// supply ep_layout's workspace -- e.g. an engine that hands the library only
// the input and output buffers it owns and has no allocator to lend (its
// memory is carved up once at start-up), or code running where a device
// allocation is not allowed. The scratch is a file-scope __device__ array of
// EP_LAYOUT_STATIC_SCRATCH_BYTES that every GPU which loads this library
// keeps until the process exits. Its device address is looked up once per
// device, on the first call made with that device current.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_layout_static_scratch[EP_LAYOUT_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void *g_static_addr[ep::kMaxDevices_] = {nullptr};

// Device address of g_layout_static_scratch on the current device (set-up on first use).
ep_status static_scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= ep::kMaxDevices_) return EP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_static_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        g_static_addr[dev] = p;
    }
    *addr = g_static_addr[dev];
    return EP_OK;
}

}  // namespace

extern "C" ep_status ep_layout_static(const ep_config *cfg, const int32_t *topk_idx, int32_t *expert_count,
                                      int32_t *expert_offset, int32_t *rank_count, int32_t *rank_offset,
                                      int32_t *slot, ep_chunk *chunks, int32_t chunk_capacity, int32_t *n_chunks,
                                      int32_t *worker_begin, cudaStream_t stream) {
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;
    if ((st = check_schedule(cfg)) != EP_OK) return st;
    if (!expert_count || !expert_offset || !rank_count || !rank_offset || !chunks || !n_chunks || !worker_begin)
        return EP_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!topk_idx || !slot)) return EP_ERR_INVALID_ARG;
    if (ep::layout_workspace(*cfg).bytes > (size_t)EP_LAYOUT_STATIC_SCRATCH_BYTES) return EP_ERR_CAPACITY;
    int32_t W = 0;
    if ((st = resolve_workers(cfg, &W)) != EP_OK) return st;
    if ((int64_t)chunk_capacity < (int64_t)ep::hop_classes(*cfg) * W + cfg->R) return EP_ERR_CAPACITY;
    void *scratch = nullptr;
    if ((st = static_scratch_address(&scratch)) != EP_OK) return st;
    return from_cuda(ep::launch_layout(*cfg, W, topk_idx, expert_count, expert_offset, rank_count, rank_offset,
                                       slot, chunks, n_chunks, worker_begin, scratch, stream));
}

// gather.cu -- schedule-driven dispatch (ep_dispatch_scheduled).
//
// The UBEP article ("Hierarchical Token-Level Scheduling") hands each worker
// (an AIV core there, a CTA here) a list of chunks of the send buffer and lets
// it move exactly those rows. Here the rows are pulled: a first kernel inverts
// the slot map (slot_meta[slot[t, j]] = t k + j, the same slot_meta
// ep_dispatch writes), then CTA c serves worker c mod W of the chunk table and
// copies, for every row s of its share, x[slot_meta[s] / k] into send[s] with
// TMA bulk copies (global -> shared -> global) through a ring of stages. The
// result equals ep_dispatch's for any table that tiles the rows once.
//
// Each x row is read k times (once per slot) instead of once; those reads hit
// L2 whenever x fits in it. Optionally every CTA stamps %globaltimer at entry
// and after its last store has landed, for per-worker timing.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kGatherBatch = 256;          // rows whose sources are staged at once
constexpr int kGatherMaxStages = 8;
constexpr uint32_t kGatherMaxPolls = 1u << 20;
constexpr size_t kGatherStageBudget = 100 * 1024;

__global__ void __launch_bounds__(256) slot_inverse_kernel(const int32_t *__restrict__ slot, int64_t pairs,
                                                           int32_t *__restrict__ meta) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const int32_t s = slot[i];
        if (s >= 0 && (int64_t)s < pairs) meta[s] = (int32_t)i;
    }
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

struct GatherArgs {
    const char *x;
    const int32_t *meta;
    const ep_chunk *chunks;
    const int32_t *n_chunks;
    const int32_t *worker_begin;
    char *send;
    int64_t *cta_ns;  // optional [gridDim.x][2]
    int32_t *err;
    int32_t T, k, W, parts, row_bytes, row_pad, stages;
};

// One warp per CTA. Lane 0 drives the copy engine; the warp stages the
// sources of up to kGatherBatch rows at a time in shared memory.
__global__ void __launch_bounds__(32) dispatch_gather_kernel(GatherArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const uint64_t t_start = globaltimer();
    const int lane = threadIdx.x;
    const int w = (int)(blockIdx.x % (unsigned)a.W);
    const int part = (int)(blockIdx.x / (unsigned)a.W);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + (size_t)a.stages * a.row_pad);
    int32_t *s_row = reinterpret_cast<int32_t *>(bar + kGatherMaxStages);  // [kGatherBatch] send row
    int32_t *s_src = s_row + kGatherBatch;                                // [kGatherBatch] x row
    if (lane == 0) {
        for (int s = 0; s < a.stages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int64_t rows = (int64_t)a.T * a.k;
    const int nc = __ldg(a.n_chunks);
    int c0 = __ldg(a.worker_begin + w), c1 = __ldg(a.worker_begin + w + 1);
    bool ok = true;
    if (c0 < 0 || c1 > nc || c0 > c1) {
        ok = false;
        c1 = c0;
    }
    uint32_t used = 0;  // stage uses so far: item g goes to stage g % stages, phase (g / stages) & 1
    for (int ci = c0; ci < c1 && ok; ++ci) {
        const int64_t rb = __ldg(&a.chunks[ci].row_begin), rn = __ldg(&a.chunks[ci].row_count);
        if (rb < 0 || rn < 0 || rb + rn > rows) {
            ok = false;
            break;
        }
        // this CTA's contiguous part of the chunk
        const int64_t lo = rb + rn * part / a.parts, hi = rb + rn * (part + 1) / a.parts;
        for (int64_t b0 = lo; b0 < hi && ok; b0 += kGatherBatch) {
            const int nb = (int)(hi - b0 < kGatherBatch ? hi - b0 : kGatherBatch);
            int n = 0;  // rows of this batch with a valid source
            for (int i0 = 0; i0 < nb; i0 += 32) {
                const int i = i0 + lane;
                int32_t src = -1;
                if (i < nb) {
                    const int32_t m = __ldg(a.meta + b0 + i);
                    if (m >= 0 && (int64_t)m < rows) src = m / a.k;
                }
                const unsigned valid = __ballot_sync(0xffffffffu, src >= 0);
                if (src >= 0) {
                    const int at = n + __popc(valid & ((1u << lane) - 1u));
                    s_row[at] = (int32_t)(b0 + i);
                    s_src[at] = src;
                }
                n += __popc(valid);
            }
            __syncwarp();
            if (lane == 0) {
                // x rows are read k times: ask L2 to keep them; send rows are
                // written once: let them go first
                const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
                auto load = [&](int i) {
                    const uint32_t g = used + (uint32_t)i;
                    const int st = (int)(g % (uint32_t)a.stages);
                    mbar_arrive_expect_tx(&bar[st], (uint32_t)a.row_bytes);
                    bulk_g2s_hint(smem + (size_t)st * a.row_pad, a.x + (int64_t)s_src[i] * a.row_bytes,
                                  (uint32_t)a.row_bytes, &bar[st], keep);
                };
                const int pre = n < a.stages ? n : a.stages;
                for (int i = 0; i < pre; ++i) load(i);
                int i = 0;
                for (; i < n; ++i) {
                    const uint32_t g = used + (uint32_t)i;
                    const int st = (int)(g % (uint32_t)a.stages);
                    if (!mbar_wait_bounded(&bar[st], (g / (uint32_t)a.stages) & 1u, kGatherMaxPolls)) {
                        ok = false;
                        break;
                    }
                    bulk_s2g_hint(a.send + (int64_t)s_row[i] * a.row_bytes, smem + (size_t)st * a.row_pad,
                                  (uint32_t)a.row_bytes, drop);
                    bulk_commit();
                    // the stage of row i - 1 is free once its store has read it
                    if (i >= 1 && i - 1 + a.stages < n) {
                        bulk_wait_read<1>();
                        load(i - 1 + a.stages);
                    }
                }
                if (!ok) {
                    // loads still in flight: rows i .. min(n, i + stages) - 1 were issued
                    // (row i + stages - 1 only if i >= 1 issued it; waiting on a phase
                    // that never completes just runs out)
                    const int last = (i == 0 ? pre : (i + a.stages - 1 < n ? i + a.stages - 1 : n));
                    for (int j = i; j < last; ++j) {
                        const uint32_t g = used + (uint32_t)j;
                        mbar_wait_bounded(&bar[g % (uint32_t)a.stages], (g / (uint32_t)a.stages) & 1u,
                                          kGatherMaxPolls);
                    }
                }
                bulk_wait_read<0>();
                used += (uint32_t)n;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            used = __shfl_sync(0xffffffffu, used, 0);
            __syncwarp();
        }
    }
    if (lane == 0) {
        bulk_wait<0>();
        if (!ok) atomicOr(a.err, kErrGatherWait);
        if (a.cta_ns) {
            a.cta_ns[2 * (int64_t)blockIdx.x] = (int64_t)t_start;
            a.cta_ns[2 * (int64_t)blockIdx.x + 1] = (int64_t)globaltimer();
        }
    }
}

struct GatherPlan {
    int parts, stages, row_pad;
    size_t smem;
};

GatherPlan plan_gather(const ep_config &c, int32_t W) {
    GatherPlan p;
    const int row_bytes = c.H * 2;
    p.row_pad = (row_bytes + 127) & ~127;
    int st = (int)(kGatherStageBudget / (size_t)p.row_pad);
    p.stages = st > kGatherMaxStages ? kGatherMaxStages : st;
    p.smem = (size_t)p.stages * p.row_pad + kGatherMaxStages * sizeof(uint64_t) + 2 * kGatherBatch * sizeof(int32_t);
    const int sms = current_device_sm_count();
    const int per_worker = W > 0 ? 2 * sms / W : 1;  // two CTAs per SM when there are few workers
    p.parts = per_worker > 1 ? per_worker : 1;
    return p;
}

}  // namespace

int64_t gather_ctas(const ep_config &c, int32_t W) {
    return (int64_t)W * plan_gather(c, W).parts;
}

cudaError_t launch_dispatch_scheduled(const ep_config &c, int32_t W, const ep_bf16 *x, const int32_t *slot,
                                      const ep_chunk *chunks, const int32_t *n_chunks, const int32_t *worker_begin,
                                      ep_bf16 *send, int32_t *meta, int64_t *cta_ns, cudaStream_t s) {
    const int64_t pairs = (int64_t)c.T * c.k;
    if (pairs == 0) return cudaSuccess;
    if (c.H * 2 > 48 * 1024) return cudaErrorNotSupported;
    int64_t g = (pairs + 255) / 256;
    const int64_t cap = (int64_t)current_device_sm_count() * 8;
    if (g > cap) g = cap;
    slot_inverse_kernel<<<(unsigned)g, 256, 0, s>>>(slot, pairs, meta);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    const GatherPlan p = plan_gather(c, W);
    int dev = 0;
    if ((e = current_device(&dev)) != cudaSuccess) return e;
    static std::atomic<bool> attr_set[kMaxDevices_];  // zero-initialised: false
    if (!attr_set[dev]) {
        if ((e = cudaFuncSetAttribute(dispatch_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)(kGatherStageBudget + 4096))) != cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    GatherArgs a;
    a.x = reinterpret_cast<const char *>(x);
    a.meta = meta;
    a.chunks = chunks;
    a.n_chunks = n_chunks;
    a.worker_begin = worker_begin;
    a.send = reinterpret_cast<char *>(send);
    a.cta_ns = cta_ns;
    if ((e = dispatch_error_word(&a.err)) != cudaSuccess) return e;
    a.T = c.T;
    a.k = c.k;
    a.W = W;
    a.parts = p.parts;
    a.row_bytes = c.H * 2;
    a.row_pad = p.row_pad;
    a.stages = p.stages;
    dispatch_gather_kernel<<<(unsigned)((int64_t)W * p.parts), 32, p.smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ep

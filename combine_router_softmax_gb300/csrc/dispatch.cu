// dispatch.cu -- row scatter into the rank-partitioned send buffer (ep_dispatch).
//
// send[slot[t, j], :] = x[t, :] and slot_meta[slot[t, j]] = t k + j: each token
// row goes to the send-buffer row of every selected expert (the UBEP article,
// opening section: a token has to reach the device that holds each expert
// chosen for it). This is the data-movement half of the article's kernel
// decomposition; on one GPU it is a pure HBM copy: read x once, write k rows.
//
// Work unit = (token, segment of 32 * U 16-byte vectors). A warp loads its U
// vectors per lane once (non-allocating streaming loads) and stores them to
// the k destination rows, so each x byte is read once and each send byte
// written once. Units are spread over a grid sized to the resident capacity
// of the GPU, which keeps the load balanced when T is small relative to the
// SM count and rows are long (H = 7168: 7 segments per row).
#include "block_common.cuh"

namespace ep {
namespace {

constexpr int kDispatchThreads = 256;
constexpr int kDispatchU = 4;  // vectors per lane per unit: 4 x 16 B in flight

template <int K>
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ slot, uint4 *__restrict__ send,
                int32_t *__restrict__ meta, int32_t k_rt, int32_t hv, int32_t segs, int64_t units,
                int64_t rows) {
    const int k = K > 0 ? K : k_rt;
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;

    for (int64_t u = gwarp; u < units; u += nwarp) {
        const int64_t t = u / segs;
        const int seg = (int)(u - t * segs);

        int my_slot = -1;
        if (lane < k) {
            const int s = __ldg(slot + t * k + lane);
            my_slot = (s >= 0 && (int64_t)s < rows) ? s : -1;
            if (seg == 0 && my_slot >= 0) meta[my_slot] = (int32_t)(t * k + lane);
        }

        const int v0 = seg * (32 * kDispatchU) + lane;
        const uint4 *src = x + t * hv;
        uint4 val[kDispatchU];
#pragma unroll
        for (int q = 0; q < kDispatchU; ++q) {
            const int v = v0 + 32 * q;
            if (v < hv) val[q] = ld_stream_v4(src + v);
        }
        if (K > 0) {
#pragma unroll
            for (int j = 0; j < (K > 0 ? K : 1); ++j) {
                const int s = __shfl_sync(0xffffffffu, my_slot, j);
                if (s < 0) continue;
                uint4 *dst = send + (int64_t)s * hv;
#pragma unroll
                for (int q = 0; q < kDispatchU; ++q) {
                    const int v = v0 + 32 * q;
                    if (v < hv) st_v4(dst + v, val[q]);
                }
            }
        } else {
            for (int j = 0; j < k; ++j) {
                const int s = __shfl_sync(0xffffffffu, my_slot, j);
                if (s < 0) continue;
                uint4 *dst = send + (int64_t)s * hv;
#pragma unroll
                for (int q = 0; q < kDispatchU; ++q) {
                    const int v = v0 + 32 * q;
                    if (v < hv) st_v4(dst + v, val[q]);
                }
            }
        }
    }
}

template <int K>
cudaError_t launch_k(const ep_config &c, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send, int32_t *meta,
                     cudaStream_t s) {
    const int32_t hv = c.H / 8;
    const int32_t segs = (hv + 32 * kDispatchU - 1) / (32 * kDispatchU);
    const int64_t units = (int64_t)c.T * segs;
    const int64_t rows = (int64_t)c.T * c.k;
    const int occ = max_blocks_per_sm(reinterpret_cast<const void *>(dispatch_kernel<K>), kDispatchThreads, 0);
    const int64_t want = (units * 32 + kDispatchThreads - 1) / kDispatchThreads;
    // 0 if the device query failed: the launch then reports the error
    const int64_t cap = (int64_t)current_device_sm_count() * occ;
    const int64_t grid = want < cap ? want : cap;
    dispatch_kernel<K><<<(unsigned)grid, kDispatchThreads, 0, s>>>(
        reinterpret_cast<const uint4 *>(x), slot, reinterpret_cast<uint4 *>(send), meta, c.k, hv, segs, units,
        rows);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bulk-copy path (k % 4 == 0, rows of >= 1 KiB): one warp per CTA, several
// CTAs per SM. Tokens go to CTAs in a fixed stride, or -- when the caller
// provides a counter in device memory -- are grabbed one at a time from it,
// so CTAs that happen to get more bandwidth take more rows (measured: with a
// fixed stride the last CTA ends ~20 % after the median one). Lane 0 streams
// token rows (and their k slots) into NS shared memory stages with TMA bulk
// loads completing on per-stage mbarriers; once a stage lands, lanes j < k
// each issue one bulk store of the row to send row slot[t, j] and write its
// slot_meta. The stage is refilled with the token NS places later as soon as
// those stores have finished reading it. The copy engine moves whole rows, so
// the SM issues ~10 instructions per 14 KB row instead of 900 vector
// loads/stores.
//
// Launched right after the layout (in ep_dispatch_fused) the kernel is a
// programmatic dependent of it: the first rounds' x rows are requested before
// griddepcontrol.wait, the slots only after. There it may also carry the
// chunk schedule the layout left undone: CTA 0 then builds the schedule from
// the rank offsets instead of moving rows.
// ---------------------------------------------------------------------------

static __device__ int32_t g_dispatch_error;

constexpr int kBulkMaxStages = 8;
constexpr uint32_t kBulkMaxPolls = 1u << 22;  // ~0.2 s of polling before giving up

__global__ void __launch_bounds__(32)
dispatch_bulk_kernel(const char *__restrict__ x, const int32_t *__restrict__ slot, char *__restrict__ send,
                     int32_t *__restrict__ meta, int32_t T, int32_t k, int32_t row_bytes, int32_t row_pad,
                     int32_t stage_bytes, int32_t NS, int64_t rows, int32_t *__restrict__ err,
                     unsigned *__restrict__ ctr, ScheduleTask st, int32_t sched_on) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x;
    if (sched_on && blockIdx.x == 0) {
        // The extra CTA: the chunk schedule the layout left to this kernel,
        // built from the layout's rank offsets while the other CTAs move rows.
        __shared__ int s_warp32[32];
        grid_dependency_wait();
        if (*reinterpret_cast<volatile int32_t *>(st.n_chunks) == -1) return;  // the layout gave up
        int32_t *s_roff = reinterpret_cast<int32_t *>(smem);
        int32_t *s_P = s_roff + st.R + 1;
        for (int r = lane; r <= st.R; r += 32) s_roff[r] = st.rank_offset[r];
        __syncthreads();
        cta_build_schedule(s_roff, st.R, st.W, st.tiers, st.chunks, st.n_chunks, st.worker_begin, s_warp32, s_P,
                           whole_cta());
        return;
    }
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + (size_t)NS * stage_bytes);
    int64_t *s_tok = reinterpret_cast<int64_t *>(bar + kBulkMaxStages);  // token of each stage, -1 = none
    const int64_t G = gridDim.x - sched_on;
    const int64_t first = blockIdx.x - sched_on;
    const int64_t n = first < T ? (T - first + G - 1) / G : 0;  // static order: tokens first + i G
    const bool dyn = ctr != nullptr;

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    auto load_row = [&](int s, int64_t t) {
        mbar_arrive_expect_tx(&bar[s], (uint32_t)row_bytes + 4u * (uint32_t)k);
        bulk_g2s(smem + (size_t)s * stage_bytes, x + t * row_bytes, (uint32_t)row_bytes, &bar[s]);
    };
    auto load_slots = [&](int s, int64_t t) {
        bulk_g2s(smem + (size_t)s * stage_bytes + row_pad, slot + t * k, 4u * (uint32_t)k, &bar[s]);
    };
    auto load = [&](int s, int64_t t) {
        load_row(s, t);
        load_slots(s, t);
    };

    // Tokens per round: static stride, or grabbed from the shared counter
    // (NS at once for the first rounds, then one per refill, one refill ahead).
    // The first rounds' x rows are requested before waiting for the grid that
    // writes the slots (the layout, when launched right after it); their
    // slots after.
    unsigned nxt = 0;
    if (lane == 0) {
        const int64_t c0 = dyn ? (int64_t)atomicAdd(ctr, (unsigned)NS) : 0;
        for (int s = 0; s < NS; ++s) {
            const int64_t t = dyn ? c0 + s : (s < n ? first + s * G : T);
            s_tok[s] = t < T ? t : -1;
            if (t < T) load_row(s, t);
        }
        if (dyn) nxt = atomicAdd(ctr, 1u);
    }
    grid_dependency_wait();
    if (lane == 0)
        for (int s = 0; s < NS; ++s)
            if (s_tok[s] >= 0) load_slots(s, s_tok[s]);
    __syncwarp();

    bool ok = true;
    int64_t i = 0;
    for (;; ++i) {
        const int s = (int)(i % NS);
        const int64_t t = s_tok[s];
        if (t < 0) break;
        if (!mbar_wait_bounded(&bar[s], (uint32_t)((i / NS) & 1), kBulkMaxPolls)) {
            ok = false;
            break;
        }
        const unsigned char *st = smem + (size_t)s * stage_bytes;
        if (lane < k) {
            const int sv = reinterpret_cast<const int32_t *>(st + row_pad)[lane];
            if (sv >= 0 && (int64_t)sv < rows) {
                bulk_s2g(send + (int64_t)sv * row_bytes, st, (uint32_t)row_bytes);
                meta[sv] = (int32_t)(t * k + lane);
            }
            bulk_commit();
        }
        // Refill the stage of round i - 1 (with round i - 1 + NS) once its stores have read it.
        if (i >= 1) {
            if (lane < k) bulk_wait_read<1>();
            __syncwarp();
            if (lane == 0) {
                const int sp = (int)((i - 1) % NS);
                int64_t tn;
                if (dyn) {
                    tn = (int64_t)nxt < T ? (int64_t)nxt : -1;
                    if (tn >= 0) nxt = atomicAdd(ctr, 1u);
                } else {
                    tn = (i - 1 + NS < n) ? first + (i - 1 + NS) * G : -1;
                }
                s_tok[sp] = tn;
                if (tn >= 0) load(sp, tn);
            }
            __syncwarp();
        }
    }
    if (!ok) {
        // Record the failure, then let every load already issued land before
        // the CTA (and its shared memory) goes away.
        if (lane == 0) atomicOr(err, kErrDispatchWait);
        for (int64_t j = i; j < i + NS - 1; ++j)
            if (s_tok[j % NS] >= 0) mbar_wait_bounded(&bar[j % NS], (uint32_t)((j / NS) & 1), kBulkMaxPolls);
    }
    if (lane < k) bulk_wait<0>();
}

int bulk_stages(int32_t row_bytes) {
    // Aim for ~112 KB of stages per CTA (7 stages of 14 KB rows; measured best of 28/56/112 KB).
    int ns = (112 * 1024) / (row_bytes + 256);
    if (ns < 2) ns = 2;
    if (ns > kBulkMaxStages) ns = kBulkMaxStages;
    return ns;
}

cudaError_t launch_bulk(const ep_config &c, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send, int32_t *meta,
                        cudaStream_t s, unsigned *ctr, bool ctr_zeroed, bool after_layout,
                        const ScheduleTask *sched) {
    const int32_t row_bytes = c.H * 2;
    const int32_t row_pad = (row_bytes + 127) & ~127;
    const int32_t stage_bytes = row_pad + 128;
    const int NS = bulk_stages(row_bytes);
    const size_t smem = (size_t)NS * stage_bytes + kBulkMaxStages * (sizeof(uint64_t) + sizeof(int64_t));
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> attr_set[kMaxDevices_];  // zero-initialised: false
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(dispatch_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int32_t *err = nullptr;
    e = dispatch_error_word(&err);
    if (e != cudaSuccess) return e;
    const int occ = max_blocks_per_sm(reinterpret_cast<const void *>(dispatch_bulk_kernel), 32, smem);
    int64_t grid = (int64_t)sm_count(dev) * occ;
    if (grid > c.T) grid = c.T;
    // the schedule CTA (index 0) needs (2 R + 4) ints of the stage memory
    const int32_t sched_on = sched && (size_t)(2 * sched->R + 4) * sizeof(int32_t) <= smem ? 1 : 0;
    if (sched && !sched_on) return cudaErrorNotSupported;
    ScheduleTask st = sched ? *sched : ScheduleTask{};
    grid += sched_on;
    if (ctr && !ctr_zeroed) {
        e = cudaMemsetAsync(ctr, 0, sizeof(unsigned), s);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_layout ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, dispatch_bulk_kernel, reinterpret_cast<const char *>(x), slot,
                              reinterpret_cast<char *>(send), meta, c.T, c.k, row_bytes, row_pad, stage_bytes, NS,
                              (int64_t)c.T * c.k, err, ctr, st, sched_on);
}

}  // namespace

cudaError_t dispatch_error_word(int32_t **addr) {
    static std::atomic<int32_t *> cached[kMaxDevices_];  // zero-initialised: null
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices_) return cudaErrorInvalidDevice;
    if (!cached[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dispatch_error);
        if (e != cudaSuccess) return e;
        cached[dev] = static_cast<int32_t *>(p);
    }
    *addr = cached[dev];
    return cudaSuccess;
}

// Bulk path when k % 4 == 0 (the k slots of a token are one 16-byte multiple),
// the slot array is 16-byte aligned and rows are at least 1 KiB.
static bool use_bulk(const ep_config &c, const int32_t *slot) {
    const int32_t row_bytes = c.H * 2;
    return c.k % 4 == 0 && (reinterpret_cast<uintptr_t>(slot) & 15u) == 0 && row_bytes >= 1024 &&
           row_bytes <= 48 * 1024;
}

bool dispatch_uses_bulk(const ep_config &c, const int32_t *slot) { return c.T > 0 && use_bulk(c, slot); }

cudaError_t launch_dispatch(const ep_config &c, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send,
                            int32_t *meta, cudaStream_t s, unsigned *ctr, bool ctr_zeroed, bool after_layout,
                            const ScheduleTask *sched) {
    if (c.T == 0) return cudaSuccess;
    if (use_bulk(c, slot)) return launch_bulk(c, x, slot, send, meta, s, ctr, ctr_zeroed, after_layout, sched);
    if (sched) return cudaErrorNotSupported;  // only the bulk kernel builds a schedule
    switch (c.k) {
        case 1: return launch_k<1>(c, x, slot, send, meta, s);
        case 2: return launch_k<2>(c, x, slot, send, meta, s);
        case 4: return launch_k<4>(c, x, slot, send, meta, s);
        case 6: return launch_k<6>(c, x, slot, send, meta, s);
        case 8: return launch_k<8>(c, x, slot, send, meta, s);
        default: return launch_k<0>(c, x, slot, send, meta, s);
    }
}

}  // namespace ep

// layout.cu -- dispatch layout (ep_layout): counts, offsets, stable slots and
// the latency-homogenized chunk schedule.
//
// The UBEP article's BSP pipeline counts tokens, computes offsets by prefix
// sums and reorders tokens ("Three Bottlenecks" / BSP Serialization); its
// "Kernel Decomposition" replaces the global barriers between those phases by
// cores that poll global memory for the metadata they need. Here:
//
//  * rank phase (every CTA, on its own tokens): a warp walks its tpw tokens
//    (4 to 32, see fused_tiling) in order with one shared-memory counter per
//    expert (lanes j < k take the k
//    distinct experts of a token at once), giving each pair its rank among
//    the warp's earlier pairs of the same expert; the per-warp histograms are
//    scanned per expert. No atomic decides an order, so slots are
//    deterministic.
//
//  * fused path (one cooperative launch, all CTAs co-resident): each CTA
//    publishes its per-expert counts as one row of a [CTA][expert] table,
//    every entry marked valid, and reads the whole table by polling each
//    entry until it is marked (bounded; no grid barrier, no SyncAll-style
//    second kernel: see block_common.cuh). Every CTA computes, redundantly and
//    in parallel, the expert offsets and its own prefix inside each expert's
//    segment, and writes its final slots.
//    CTA 0 writes the counts/offsets and the last CTA the chunk schedule,
//    unless the caller defers the schedule to the dispatch kernel that
//    follows (its extra CTA builds it while the other CTAs copy rows).
//
//  * fallback (T beyond what one co-resident grid holds): three kernels --
//    rank, a one-CTA scan (+ schedule), finalize.
//
// Schedule ("Hierarchical Token-Level Scheduling" / Latency Homogenization):
// every worker gets an equal share of each hop class. One thread per worker
// finds where its share starts with a 4-ary search over the class prefix
// sums (the article's quaternary search: three independent pivot compares
// per step, ~log4(n) steps), then cuts its share at rank boundaries.
#include <climits>

#include "block_common.cuh"
#include "flag_ops.cuh"

namespace ep {

namespace {

constexpr int kScanThreads = 1024;
constexpr int kFusedMaxWarps = 32;
constexpr size_t kFusedSmemBudget = 160 * 1024;

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Shared memory of the fused kernel for nw warps of tpw tokens each.
size_t fused_smem_bytes(int nw, int tpw, int32_t E, int32_t R, int32_t k) {
    return sizeof(int32_t) * ((size_t)nw * E + 2 * (size_t)nw * tpw * k + 3 * (size_t)E + 2 + 2 * (size_t)R + 4);
}

// The single-kernel layout's tiling: nw warps (16, 8 or 32) of tpw tokens (4
// to 32) per CTA, nb CTAs. The rank phase was the kernel's longest (a warp
// ranks its pairs 32 at a time) and the count-table read comes next (a thread
// sums nb / tpe rows of its expert's column), so the CTAs are many and small
// and, where shared memory allows, wide: for each warp count the fewest tokens
// per warp (at least 4) that keep the grid at <= kLayoutTargetCTAs CTAs,
// preferring 16 warps, then 8, then 32; above the target the smallest grid.
// nw = 0 if nothing fits the shared-memory budget.
struct LayoutTiling {
    int nw = 0, tpw = 32;
    int64_t nb = 0;
};
constexpr int64_t kLayoutTargetCTAs = 64;

LayoutTiling fused_tiling(int64_t T, int32_t E, int32_t R, int32_t k) {
    LayoutTiling best;
    const int order[3] = {16, 8, 32};
    for (int i = 0; i < 3; ++i) {
        const int nw = order[i];
        int tpw = 4;
        while (tpw < 32 && (T + (int64_t)nw * tpw - 1) / ((int64_t)nw * tpw) > kLayoutTargetCTAs) tpw <<= 1;
        if (fused_smem_bytes(nw, tpw, E, R, k) > kFusedSmemBudget) continue;
        const int64_t nb = (T + (int64_t)nw * tpw - 1) / ((int64_t)nw * tpw);
        if (best.nw == 0 || nb < best.nb) {
            best.nw = nw;
            best.tpw = tpw;
            best.nb = nb;
        }
        if (nb <= kLayoutTargetCTAs) break;
    }
    return best;
}

}  // namespace

LayoutWorkspace layout_workspace(const ep_config &c) {
    LayoutWorkspace w;
    const int64_t nb = layout_blocks(c.T);
    w.block_counts_off = 0;
    const LayoutTiling t = fused_tiling(c.T, c.E, c.R, c.k);
    const int64_t nbf = t.nw > 0 ? t.nb : nb;
    w.table_words = (size_t)nbf * (size_t)c.E;
    const size_t fallback = align256(sizeof(int32_t) * (size_t)nb * (size_t)c.E);
    const size_t fused = align256(sizeof(int32_t) * w.table_words);
    w.bytes = c.T == 0 ? 0 : (fallback > fused ? fallback : fused);
    return w;
}

namespace {

// kMaxThreads: the CTA size the instance is compiled for (512, or 1024 for
// 32 warps, which leaves 64 registers a thread: there the table is read 16
// entries at a time instead of 32).
template <int kMaxThreads>
__global__ void __launch_bounds__(kMaxThreads)
layout_fused_kernel(const int32_t *__restrict__ idx, int32_t T, int32_t E, int32_t R, int32_t k, int32_t nb,
                    int32_t *__restrict__ counts, int32_t *__restrict__ expert_count,
                    int32_t *__restrict__ expert_offset, int32_t *__restrict__ rank_count,
                    int32_t *__restrict__ rank_offset, int32_t *__restrict__ slot, ep_chunk *__restrict__ chunks,
                    int32_t *__restrict__ n_chunks, int32_t *__restrict__ worker_begin, int32_t W,
                    HopTiers tiers, int32_t defer_schedule, int32_t tpw, unsigned *__restrict__ zero_ctr) {
    extern __shared__ int32_t sm[];
    // A dispatch launched after this kernel may start now and fetch x rows
    // (it waits for this grid before it reads a slot). Its token counter, if
    // any, is zeroed first: the dispatch grid can start only once every CTA
    // of this one has passed this point.
    if (zero_ctr != nullptr && blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            *zero_ctr = 0u;
            __threadfence();
        }
        __syncthreads();
    }
    grid_launch_dependents();
    // Launched right after the route kernel, this grid may start before that
    // one has finished: nothing it writes is read before this wait.
    grid_dependency_wait();
    const int nw = blockDim.x >> 5;
    int32_t *cnt = sm;                         // [nw][E]
    int32_t *tile_e = cnt + nw * E;            // [nw][tpw k]
    int32_t *tile_r = tile_e + nw * tpw * k;   // [nw][tpw k]
    int32_t *s_tot = tile_r + nw * tpw * k;    // [E]   pairs of expert e, all CTAs
    int32_t *s_pre = s_tot + E;                // [E]   pairs of expert e in CTAs before this one
    int32_t *s_eoff = s_pre + E;               // [E+2] expert offsets (+ total)
    int32_t *s_roff = s_eoff + E + 2;          // [R+1] rank offsets
    int32_t *s_P = s_roff + R + 1;             // [R+3] class prefix sums (schedule)
    __shared__ int s_warp32[32];

    __shared__ int s_fail;
    if (threadIdx.x == 0) s_fail = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        s_tot[e] = 0;
        s_pre[e] = 0;
    }

    const int b = blockIdx.x;
    const int64_t t_cta = (int64_t)b * tpw * nw;
    // s_eoff holds this CTA's per-expert counts until the table has been read.
    cta_rank_tokens(idx, T, E, k, t_cta, cnt, tile_e, tile_r, s_eoff, 1, tpw);

    // Publish them as row b of the count table and read every CTA's row
    // (block_common.cuh: entries marked valid, polled, no grid barrier).
    unsigned *tab = reinterpret_cast<unsigned *>(counts);
    const TablePublish pub = nb > 1 ? table_publish(tab + (int64_t)b * E, s_eoff, E) : TablePublish{};

    // Expert totals over all CTAs and this CTA's prefix inside each expert.
    // tpe warps share 32 consecutive columns of the table (a lane per column,
    // so each load of a warp is one 128-byte line), each summing every tpe-th
    // row of the other CTAs (this CTA's own counts come from shared memory);
    // integer adds into shared memory make the order irrelevant. (s_tot and
    // s_pre were zeroed before the rank phase, whose CTA barriers order that.)
    if (nb == 1) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) s_tot[e] = s_eoff[e];
    } else {
        const int tpe = threads_per_expert(E, nw);
        const int warp = (int)threadIdx.x >> 5;
        const int sub = warp % tpe;
        for (int e = (warp / tpe) * 32 + ((int)threadIdx.x & 31); e < E; e += (nw / tpe) * 32) {
            int tot, pre;
            if (!table_column_sums<kMaxThreads <= 512 ? 32 : 16>(tab, E, e, sub, tpe, nb, b, b, kBarrierSpinLimit,
                                                                 tot, pre)) {
                s_fail = 1;
                break;
            }
            if (sub == 0) tot += s_eoff[e];
            if (tpe == 1) {
                s_tot[e] = tot;
                s_pre[e] = pre;
            } else {
                atomicAdd(&s_tot[e], tot);
                atomicAdd(&s_pre[e], pre);
            }
        }
    }
    if (pub.late()) s_fail = 1;
    __syncthreads();
    if (s_fail) {
        if (threadIdx.x == 0) atomicExch(n_chunks, -1);
        return;
    }

    // Exclusive scan of the totals: each thread scans a contiguous run.
    {
        const int per = (E + blockDim.x - 1) / blockDim.x;
        const int e0 = threadIdx.x * per;
        const int e1 = e0 + per < E ? e0 + per : E;
        int local = 0;
        for (int e = e0; e < e1; ++e) local += s_tot[e];
        int total;
        int run = cta_exclusive_scan32(local, s_warp32, &total);
        for (int e = e0; e < e1; ++e) {
            s_eoff[e] = run;
            run += s_tot[e];
        }
        if (threadIdx.x == 0) s_eoff[E] = total;
    }
    __syncthreads();

    // Final slots of this CTA's pairs.
    {
        const int64_t left = (int64_t)T - t_cta;
        const int np = (left <= 0 ? 0 : (left >= tpw * nw ? tpw * nw : (int)left)) * k;
        for (int p = threadIdx.x; p < np; p += blockDim.x) {
            const int e = tile_e[p];
            const int r = tile_r[p];
            slot[t_cta * k + p] = r < 0 ? -1 : s_eoff[e] + s_pre[e] + cnt[(p / (tpw * k)) * E + e] + r;
        }
    }

    const int32_t epr = E / R;
    if (b == 0) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            expert_offset[e] = s_eoff[e];
            if (e < E) expert_count[e] = s_tot[e];
        }
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            rank_offset[r] = s_eoff[r * epr];
            rank_count[r] = s_eoff[(r + 1) * epr] - s_eoff[r * epr];
        }
        if (threadIdx.x == 0) rank_offset[R] = s_eoff[E];
    }
    if (b == nb - 1 && !defer_schedule) {
        for (int r = threadIdx.x; r <= R; r += blockDim.x) s_roff[r] = s_eoff[r * epr];
        __syncthreads();
        cta_build_schedule(s_roff, R, W, tiers, chunks, n_chunks, worker_begin, s_warp32, s_P, whole_cta());
    }
}

// ---------------------------------------------------------------------------
// fallback path: rank / scan (+ schedule) / finalize
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kLayoutWarps * 32)
layout_rank_kernel(const int32_t *__restrict__ idx, int32_t T, int32_t E, int32_t k, int32_t nb,
                   int32_t *__restrict__ block_counts, int32_t *__restrict__ slot) {
    extern __shared__ int32_t sm[];
    int32_t *cnt = sm;                                  // [warps][E]
    int32_t *tile_e = cnt + kLayoutWarps * E;           // [warps][32 k]
    int32_t *tile_r = tile_e + kLayoutWarps * 32 * k;   // [warps][32 k]
    const int64_t t_cta = (int64_t)blockIdx.x * kLayoutTokens;
    cta_rank_tokens(idx, T, E, k, t_cta, cnt, tile_e, tile_r, block_counts + blockIdx.x, nb);

    const int64_t left = (int64_t)T - t_cta;
    const int np = (left <= 0 ? 0 : (left >= kLayoutTokens ? kLayoutTokens : (int)left)) * k;
    for (int p = threadIdx.x; p < np; p += blockDim.x) {
        const int e = tile_e[p];
        const int r = tile_r[p];
        slot[t_cta * k + p] = r < 0 ? -1 : cnt[(p / (32 * k)) * E + e] + r;
    }
}

__global__ void __launch_bounds__(kScanThreads)
layout_scan_kernel(int32_t *__restrict__ block_counts, int32_t nb, int32_t E, int32_t R,
                   int32_t *__restrict__ expert_count, int32_t *__restrict__ expert_offset,
                   int32_t *__restrict__ rank_count, int32_t *__restrict__ rank_offset,
                   ep_chunk *__restrict__ chunks, int32_t *__restrict__ n_chunks,
                   int32_t *__restrict__ worker_begin, int32_t W, HopTiers tiers) {
    __shared__ int64_t s_warp[32];
    __shared__ int32_t s_eoff[kMaxE + 1];
    __shared__ int32_t s_roff[kMaxE + 1];
    __shared__ int32_t s_total;

    // (a) exclusive scan of the expert-major [E][nb] counts, in place.
    const int64_t n = (int64_t)E * nb;
    const int64_t per = (n + blockDim.x - 1) / blockDim.x;
    const int64_t b0 = per * threadIdx.x;
    const int64_t b1 = b0 + per < n ? b0 + per : n;
    int64_t local = 0;
    for (int64_t i = b0; i < b1; ++i) local += block_counts[i];
    int64_t total;
    int64_t run = cta_exclusive_scan(local, s_warp, &total);
    for (int64_t i = b0; i < b1; ++i) {
        const int32_t c = block_counts[i];
        block_counts[i] = (int32_t)run;
        run += c;
    }
    if (threadIdx.x == 0) s_total = (int32_t)total;
    __syncthreads();

    // (b) expert and rank offsets / counts. Row e of the scanned table starts
    // with the number of pairs of all experts below e.
    for (int e = threadIdx.x; e <= E; e += blockDim.x)
        s_eoff[e] = (e == E || nb == 0) ? (e == E ? s_total : 0) : block_counts[(int64_t)e * nb];
    __syncthreads();
    const int32_t epr = E / R;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        expert_offset[e] = s_eoff[e];
        if (e < E) expert_count[e] = s_eoff[e + 1] - s_eoff[e];
    }
    for (int r = threadIdx.x; r <= R; r += blockDim.x) {
        const int32_t v = s_eoff[r * epr];
        s_roff[r] = v;
        rank_offset[r] = v;
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) rank_count[r] = s_roff[r + 1] - s_roff[r];

    // (c) chunk schedule.
    __shared__ int s_warp32[32];
    __shared__ int32_t s_P[kMaxE + 3];
    cta_build_schedule(s_roff, R, W, tiers, chunks, n_chunks, worker_begin, s_warp32, s_P, whole_cta());
}

__global__ void __launch_bounds__(256)
layout_finalize_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ block_base,
                       int32_t *__restrict__ slot, int64_t npairs, int32_t k, int32_t E, int32_t nb) {
    grid_launch_dependents();  // as in layout_fused_kernel
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npairs; i += stride) {
        const int e = __ldg(idx + i);
        const int s = slot[i];
        if (s >= 0 && (unsigned)e < (unsigned)E) {
            const int64_t b = (i / k) / kLayoutTokens;
            slot[i] = s + __ldg(block_base + (int64_t)e * nb + b);
        }
    }
}

size_t rank_smem_bytes(int32_t E, int32_t k) {
    return sizeof(int32_t) * ((size_t)kLayoutWarps * E + 2 * (size_t)kLayoutWarps * 32 * k);
}

cudaError_t launch_fallback(const ep_config &c, int32_t W, const int32_t *idx, int32_t *expert_count,
                            int32_t *expert_offset, int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                            ep_chunk *chunks, int32_t *n_chunks, int32_t *worker_begin, void *workspace,
                            cudaStream_t s) {
    const int64_t nb = layout_blocks(c.T);
    int32_t *block_counts = static_cast<int32_t *>(workspace);
    if (nb > 0) {
        const size_t smem = rank_smem_bytes(c.E, c.k);
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(layout_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
        }
        layout_rank_kernel<<<(unsigned)nb, kLayoutWarps * 32, smem, s>>>(idx, c.T, c.E, c.k, (int32_t)nb,
                                                                          block_counts, slot);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    layout_scan_kernel<<<1, kScanThreads, 0, s>>>(block_counts, (int32_t)nb, c.E, c.R, expert_count, expert_offset,
                                                  rank_count, rank_offset, chunks, n_chunks, worker_begin, W,
                                                  hop_tiers(c));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (nb > 0) {
        const int64_t npairs = (int64_t)c.T * c.k;
        int64_t grid = (npairs + 255) / 256;
        const int64_t cap = (int64_t)current_device_sm_count() * 8;
        if (grid > cap) grid = cap;
        layout_finalize_kernel<<<(unsigned)grid, 256, 0, s>>>(idx, block_counts, slot, npairs, c.k, c.E,
                                                              (int32_t)nb);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

// The layout_fused_kernel instance for CTAs of nw warps.
static const void *layout_fused_fn(int nw) {
    return nw * 32 <= 512 ? reinterpret_cast<const void *>(layout_fused_kernel<512>)
                          : reinterpret_cast<const void *>(layout_fused_kernel<1024>);
}

static bool layout_fused_fits(const ep_config &c, int *nw_out, int64_t *nb_out, int *tpw_out = nullptr) {
    if (c.T == 0) return false;
    const LayoutTiling t = fused_tiling(c.T, c.E, c.R, c.k);
    const int nw = t.nw;
    if (nw == 0) return false;
    const int64_t nb = t.nb;
    const size_t smem = fused_smem_bytes(nw, t.tpw, c.E, c.R, c.k);
    static std::atomic<bool> attr_set[kMaxDevices_];  // zero-initialised: false
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices_) return false;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(layout_fused_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kFusedSmemBudget) != cudaSuccess ||
            cudaFuncSetAttribute(layout_fused_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kFusedSmemBudget) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        attr_set[dev] = true;
    }
    const int per_sm = max_blocks_per_sm(layout_fused_fn(nw), nw * 32, smem);
    if (nb > (int64_t)sm_count(dev) * per_sm) return false;
    *nw_out = nw;
    *nb_out = nb;
    if (tpw_out) *tpw_out = t.tpw;
    return true;
}

int layout_kernel_count(const ep_config &c) {
    int nw = 0;
    int64_t nb = 0;
    if (layout_fused_fits(c, &nw, &nb)) return 1;
    return layout_blocks(c.T) > 0 ? 3 : 1;
}

cudaError_t launch_layout(const ep_config &c, int32_t W, const int32_t *idx, int32_t *expert_count,
                          int32_t *expert_offset, int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                          ep_chunk *chunks, int32_t *n_chunks, int32_t *worker_begin, void *workspace,
                          cudaStream_t s, bool table_zeroed, bool defer_schedule, bool *deferred, bool after_route,
                          unsigned *zero_ctr) {
    if (deferred) *deferred = false;
    int nw = 0, tpw = 32;
    int64_t nb = 0;
    if (!layout_fused_fits(c, &nw, &nb, &tpw))
        return launch_fallback(c, W, idx, expert_count, expert_offset, rank_count, rank_offset, slot, chunks,
                               n_chunks, worker_begin, workspace, s);

    int32_t *counts = static_cast<int32_t *>(workspace);
    if (nb > 1 && !table_zeroed) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)nb * (size_t)c.E, s);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = fused_smem_bytes(nw, tpw, c.E, c.R, c.k);
    int32_t T = c.T, E = c.E, R = c.R, k = c.k, nbi = (int32_t)nb;
    HopTiers tiers = hop_tiers(c);
    int32_t defer = defer_schedule ? 1 : 0;
    if (deferred) *deferred = defer_schedule;
    // Set when a device refused the launch below; the plain cooperative launch
    // is then used (the same results, the route -> layout gap not hidden).
    static std::atomic<bool> no_dependent_coop[kMaxDevices_];  // zero-initialised: false
    int dev = 0;
    if (after_route && (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices_)) after_route = false;
    if (after_route && !no_dependent_coop[dev]) {
        // A cooperative launch that may also start before the route kernel in
        // front of it has finished (programmatic dependent launch).
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)nb);
        cfg.blockDim = dim3((unsigned)(nw * 32));
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        const cudaError_t e =
            nw * 32 <= 512
                ? cudaLaunchKernelEx(&cfg, layout_fused_kernel<512>, idx, T, E, R, k, nbi, counts, expert_count,
                                     expert_offset, rank_count, rank_offset, slot, chunks, n_chunks, worker_begin, W,
                                     tiers, defer, tpw, zero_ctr)
                : cudaLaunchKernelEx(&cfg, layout_fused_kernel<1024>, idx, T, E, R, k, nbi, counts, expert_count,
                                     expert_offset, rank_count, rank_offset, slot, chunks, n_chunks, worker_begin, W,
                                     tiers, defer, tpw, zero_ctr);
        if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return e;
        cudaGetLastError();  // the launch was refused before anything was enqueued
        no_dependent_coop[dev] = true;
    }
    void *args[] = {(void *)&idx, &T, &E, &R, &k, &nbi, (void *)&counts, (void *)&expert_count,
                    (void *)&expert_offset, (void *)&rank_count, (void *)&rank_offset, (void *)&slot,
                    (void *)&chunks, (void *)&n_chunks, (void *)&worker_begin, &W, &tiers, &defer, &tpw,
                    (void *)&zero_ctr};
    return cudaLaunchCooperativeKernel(layout_fused_fn(nw), dim3((unsigned)nb),
                                       dim3((unsigned)(nw * 32)), args, smem, s);
}

}  // namespace ep

// ---------------------------------------------------------------------------
// Self-check of the bounded grid barrier: CTAs 0 and 1 wait at a grid barrier
// that expects three arrivals; CTA 2 arrives only after one of them has given
// up (it waits, bounded, for the counter's top bit), the order in which the
// last arrival would let a CTA go on with a result missing. CTAs 0 and 1 must
// give up after max_polls polls and count themselves in *gave_up, and CTA 2
// must see the failure too; a second kernel sets *gave_up = -1 if it did not.
// CTA 3 runs the split dispatch's warp-wide wait on a ready flag that nothing
// sets and must give up after max_polls polls as well. CTAs 4 and 5 exchange
// a two-row count table the way the single-kernel layout does: CTA 4 publishes
// row 0 and reads both rows, but row 1 is published by CTA 5 only after CTA 4
// has given up and poisoned it; both must fail (a successful late publish also
// makes the second kernel set -1).
// ---------------------------------------------------------------------------
namespace ep {
namespace {

static __device__ unsigned g_check_arrivals[2];  // barrier arrivals, a flag nothing sets
static __device__ unsigned g_check_table[2];     // a count table of two rows and one expert
static __device__ int32_t g_check_late_passed;  // 1: a late CTA went on

__global__ void bounded_wait_check_kernel(unsigned *arrivals, unsigned *table, int32_t *late_passed,
                                          unsigned max_polls, int32_t *gave_up) {
    if (blockIdx.x >= 4) {
        if (threadIdx.x != 0) return;
        const int32_t own = 1;
        if (blockIdx.x == 4) {
            table_publish(table, &own, 1);
            int tot, pre;
            if (!table_column_sums(table, 1, 0, 0, 1, 2, 0, -1, max_polls, tot, pre)) atomicAdd(gave_up, 1);
            return;
        }
        const uint64_t limit = 4ull * max_polls + 1024ull;
        for (uint64_t i = 0; i < limit && ld_relaxed_gpu(table + 1) != kCountPoison; ++i) __nanosleep(64);
        if (table_publish(table + 1, &own, 1).late())
            atomicAdd(gave_up, 1);
        else
            *late_passed = 1;
        return;
    }
    if (blockIdx.x == 3) {
        // the split dispatch's wait on a tile's ready flag, on a flag nothing sets
        if (threadIdx.x < 32 && !warp_wait_flag(arrivals + 1, max_polls) && threadIdx.x == 0) atomicAdd(gave_up, 1);
        return;
    }
    if (blockIdx.x < 2) {
        if (!grid_barrier(arrivals, 3u, max_polls) && threadIdx.x == 0) atomicAdd(gave_up, 1);
        return;
    }
    if (threadIdx.x == 0) {
        const uint64_t limit = 4ull * max_polls + 1024ull;
        for (uint64_t i = 0; i < limit && (atomicOr(arrivals, 0u) & kBarrierPoison) == 0u; ++i) __nanosleep(64);
    }
    if (grid_barrier(arrivals, 3u, max_polls) && threadIdx.x == 0) *late_passed = 1;
}

__global__ void bounded_wait_verdict_kernel(const int32_t *late_passed, int32_t *gave_up) {
    if (*late_passed != 0) *gave_up = -1;
}

}  // namespace

cudaError_t launch_bounded_wait_check(uint32_t max_polls, int32_t *gave_up, cudaStream_t s) {
    void *arrivals = nullptr, *table = nullptr, *late = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&arrivals, g_check_arrivals);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetSymbolAddress(&table, g_check_table)) != cudaSuccess) return e;
    if ((e = cudaGetSymbolAddress(&late, g_check_late_passed)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(arrivals, 0, 2 * sizeof(unsigned), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(table, 0, 2 * sizeof(unsigned), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(late, 0, sizeof(int32_t), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(gave_up, 0, sizeof(int32_t), s)) != cudaSuccess) return e;
    bounded_wait_check_kernel<<<6, 32, 0, s>>>(static_cast<unsigned *>(arrivals), static_cast<unsigned *>(table),
                                               static_cast<int32_t *>(late), max_polls, gave_up);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bounded_wait_verdict_kernel<<<1, 1, 0, s>>>(static_cast<const int32_t *>(late), gave_up);
    return cudaGetLastError();
}

}  // namespace ep

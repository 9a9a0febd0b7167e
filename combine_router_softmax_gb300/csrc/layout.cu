// layout.cu -- dispatch layout (ep_layout): counts, offsets, stable slots and
// the latency-homogenized chunk schedule.
//
// The UBEP article's BSP pipeline counts tokens, computes offsets by prefix
// sums and reorders tokens ("Three Bottlenecks" / BSP Serialization); its
// "Kernel Decomposition" gives those metadata steps to a few cores and the
// row movement to the rest. Here the metadata is three short kernels:
//
//  1. rank   : each CTA takes 256 consecutive tokens (32 per warp). A warp
//              walks its 32 tokens in order with one shared-memory counter per
//              expert (lanes j < k handle the k distinct experts of a token at
//              once), which yields each pair's rank among the warp's earlier
//              pairs of the same expert. The 8 warp histograms are then
//              scanned per expert, giving each pair its rank inside the CTA
//              and the CTA's per-expert count (written expert-major to the
//              workspace). No atomics decide an order, so slots are
//              deterministic.
//  2. scan   : one CTA scans the expert-major [E][nb] counts (exclusive),
//              which turns every CTA's count into the base of its run inside
//              the expert's segment; it then writes the expert and rank
//              counts/offsets and builds the chunk schedule.
//  3. final  : slot = CTA base of (expert, CTA) + rank inside the CTA.
//
// Schedule ("Hierarchical Token-Level Scheduling" / Latency Homogenization):
// every worker gets an equal share of each hop class. One thread per worker
// finds where its share starts with a 4-ary search over the class prefix
// sums (the article's quaternary search: three independent pivot compares
// per step, ~log4(n) steps), then cuts its share at rank boundaries.
#include <climits>

#include "ep_internal.cuh"

namespace ep {

LayoutWorkspace layout_workspace(int64_t T, int32_t E) {
    LayoutWorkspace w;
    const int64_t nb = layout_blocks(T);
    w.block_counts_off = 0;
    size_t bytes = sizeof(int32_t) * (size_t)nb * (size_t)E;
    w.bytes = (bytes + 255) & ~(size_t)255;
    return w;
}

namespace {

constexpr int kScanThreads = 1024;

// ---------------------------------------------------------------------------
// 1. per-CTA ranks and histograms
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLayoutWarps * 32)
layout_rank_kernel(const int32_t *__restrict__ idx, int32_t T, int32_t E, int32_t k, int32_t nb,
                   int32_t *__restrict__ block_counts, int32_t *__restrict__ slot) {
    extern __shared__ int32_t sm[];
    int32_t *cnt = sm;                                  // [warps][E]
    int32_t *tile_e = cnt + kLayoutWarps * E;           // [warps][32 k] expert ids
    int32_t *tile_r = tile_e + kLayoutWarps * 32 * k;   // [warps][32 k] rank within the warp

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) cnt[i] = 0;

    const int64_t t0 = (int64_t)blockIdx.x * kLayoutTokens + (int64_t)warp * 32;
    const int64_t left = (int64_t)T - t0;
    const int ntok = left <= 0 ? 0 : (left >= 32 ? 32 : (int)left);
    const int npair = ntok * k;
    int32_t *te = tile_e + warp * 32 * k;
    int32_t *tr = tile_r + warp * 32 * k;
    int32_t *wc = cnt + warp * E;
    for (int i = lane; i < npair; i += 32) te[i] = __ldg(idx + t0 * k + i);
    __syncthreads();

    for (int tt = 0; tt < ntok; ++tt) {
        if (lane < k) {
            const int e = te[tt * k + lane];
            int r = -1;
            if ((unsigned)e < (unsigned)E) {
                r = wc[e];
                wc[e] = r + 1;
            }
            tr[tt * k + lane] = r;
        }
        __syncwarp();
    }
    __syncthreads();

    // Exclusive scan over the warps, per expert; the CTA total goes out.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int c = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += c;
        }
        block_counts[(int64_t)e * nb + blockIdx.x] = run;
    }
    __syncthreads();

    for (int i = lane; i < npair; i += 32) {
        const int e = te[i];
        const int r = tr[i];
        slot[t0 * k + i] = r < 0 ? -1 : wc[e] + r;
    }
}

// ---------------------------------------------------------------------------
// 2. scan, counts/offsets, chunk schedule (one CTA)
// ---------------------------------------------------------------------------

// Exclusive scan of one value per thread over the CTA; returns the prefix and
// stores the CTA total in *total. Uses s_warp[32].
__device__ __forceinline__ int64_t cta_exclusive_scan(int64_t x, int64_t *s_warp, int64_t *total) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int64_t inc = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int64_t wv = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t o = __shfl_up_sync(0xffffffffu, wv, d);
            if (lane >= d) wv += o;
        }
        if (lane < nwarps) s_warp[lane] = wv;  // inclusive warp prefix
    }
    __syncthreads();
    const int64_t base = warp > 0 ? s_warp[warp - 1] : 0;
    *total = s_warp[nwarps - 1];
    __syncthreads();  // s_warp may be reused by the caller
    return base + inc - x;
}

// Class prefix sums in closed form. Class 0 (near) is ranks [n_lo, n_hi);
// class 1 (far) is [0, n_lo) followed by [n_hi, R). P_c(i) is the number of
// rows in the first i ranks of class c; rank_of(c, i) is that i-th rank.
struct ClassView {
    const int32_t *ro;  // rank_offset, R + 1 entries
    int32_t n_lo, n_hi, R;
    __device__ int32_t size(int c) const { return c == 0 ? n_hi - n_lo : R - (n_hi - n_lo); }
    __device__ int32_t rank_of(int c, int32_t i) const {
        return c == 0 ? n_lo + i : (i < n_lo ? i : i + (n_hi - n_lo));
    }
    __device__ int64_t prefix(int c, int32_t i) const {
        if (c == 0) return (int64_t)ro[n_lo + i] - ro[n_lo];
        if (i <= n_lo) return ro[i];
        return (int64_t)ro[n_lo] + ((int64_t)ro[i + (n_hi - n_lo)] - ro[n_hi]);
    }
};

// Largest i in [0, n) with P(i) <= x, for P non-decreasing and P(0) <= x.
// 4-ary search: three independent pivot compares narrow the range 4x per step.
__device__ __forceinline__ int32_t quaternary_search(const ClassView &cv, int c, int32_t n, int64_t x) {
    int32_t lo = 0, hi = n;  // answer in [lo, hi), P(lo) <= x
    while (hi - lo > 1) {
        const int32_t len = hi - lo;
        const int32_t q1 = lo + len / 4, q2 = lo + len / 2, q3 = lo + (3 * len) / 4;
        const bool c1 = cv.prefix(c, q1) <= x;
        const bool c2 = cv.prefix(c, q2) <= x;
        const bool c3 = cv.prefix(c, q3) <= x;
        if (c3) {
            lo = q3;
        } else if (c2) {
            lo = q2;
            hi = q3;
        } else if (c1) {
            lo = q1;
            hi = q2;
        } else {
            hi = q1;
        }
    }
    return lo;
}

// Walk worker w's share of class c; count chunks, or write them from `pos`.
__device__ int32_t worker_class_chunks(const ClassView &cv, int c, int64_t N, int32_t w, int32_t W,
                                       ep_chunk *chunks, int32_t pos, bool write) {
    const int64_t lo = N * w / W;
    const int64_t hi = N * (w + 1) / W;
    if (hi <= lo) return 0;
    const int32_t n = cv.size(c);
    int32_t i = quaternary_search(cv, c, n, lo);
    int32_t cnt = 0;
    for (; i < n; ++i) {
        const int64_t seg_lo = cv.prefix(c, i);
        if (seg_lo >= hi) break;
        const int64_t seg_hi = cv.prefix(c, i + 1);
        const int64_t a = lo > seg_lo ? lo : seg_lo;
        const int64_t b = hi < seg_hi ? hi : seg_hi;
        if (b <= a) continue;
        if (write) {
            const int32_t r = cv.rank_of(c, i);
            ep_chunk ch;
            ch.worker = w;
            ch.hop_class = c;
            ch.dst_rank = r;
            ch.row_begin = (int32_t)(cv.ro[r] + (a - seg_lo));
            ch.row_count = (int32_t)(b - a);
            chunks[pos + cnt] = ch;
        }
        ++cnt;
    }
    return cnt;
}

__global__ void __launch_bounds__(kScanThreads)
layout_scan_kernel(int32_t *__restrict__ block_counts, int32_t nb, int32_t E, int32_t R,
                   int32_t *__restrict__ expert_count, int32_t *__restrict__ expert_offset,
                   int32_t *__restrict__ rank_count, int32_t *__restrict__ rank_offset,
                   ep_chunk *__restrict__ chunks, int32_t *__restrict__ n_chunks,
                   int32_t *__restrict__ worker_begin, int32_t W, int32_t ranks_per_node, int32_t self_rank) {
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
    ClassView cv;
    cv.ro = s_roff;
    cv.R = R;
    const int32_t node = self_rank / ranks_per_node;
    cv.n_lo = node * ranks_per_node;
    cv.n_hi = cv.n_lo + ranks_per_node < R ? cv.n_lo + ranks_per_node : R;
    const int64_t N0 = (int64_t)s_roff[cv.n_hi] - s_roff[cv.n_lo];
    const int64_t N1 = (int64_t)s_total - N0;

    int64_t carry = 0;
    for (int32_t wb = 0; wb < W; wb += blockDim.x) {
        const int32_t w = wb + (int32_t)threadIdx.x;
        int32_t c1 = 0, c0 = 0;
        if (w < W) {
            c1 = worker_class_chunks(cv, 1, N1, w, W, chunks, 0, false);
            c0 = worker_class_chunks(cv, 0, N0, w, W, chunks, 0, false);
        }
        int64_t tile_total;
        const int64_t first = carry + cta_exclusive_scan(c1 + c0, s_warp, &tile_total);
        if (w < W) {
            worker_begin[w] = (int32_t)first;
            worker_class_chunks(cv, 1, N1, w, W, chunks, (int32_t)first, true);
            worker_class_chunks(cv, 0, N0, w, W, chunks, (int32_t)(first + c1), true);
        }
        carry += tile_total;
    }
    if (threadIdx.x == 0) {
        worker_begin[W] = (int32_t)carry;
        *n_chunks = (int32_t)carry;
    }
}

// ---------------------------------------------------------------------------
// 3. slot = CTA base + rank inside the CTA
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
layout_finalize_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ block_base,
                       int32_t *__restrict__ slot, int64_t npairs, int32_t k, int32_t E, int32_t nb) {
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

}  // namespace

cudaError_t launch_layout(const ep_config &c, int32_t W, const int32_t *idx, int32_t *expert_count,
                          int32_t *expert_offset, int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                          ep_chunk *chunks, int32_t *n_chunks, int32_t *worker_begin, void *workspace,
                          cudaStream_t s) {
    const int64_t nb = layout_blocks(c.T);
    const LayoutWorkspace ws = layout_workspace(c.T, c.E);
    int32_t *block_counts = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + ws.block_counts_off);

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
                                                  c.ranks_per_node, c.self_rank);
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

}  // namespace ep

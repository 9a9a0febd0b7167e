// block_common.cuh -- CTA-wide building blocks shared by the layout kernels
// and the fused dispatch: CTA scans, the per-warp ranking of (token, expert)
// pairs, the chunk schedule, a bounded grid barrier and a count table that
// CTAs exchange without one.
#pragma once

#include <climits>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr unsigned kBarrierSpinLimit = 1u << 22;  // polls of ~64 ns before giving up

// Top bit of a grid barrier's arrival counter: set by a CTA that gave up
// waiting while the barrier was still incomplete (see grid_barrier).
constexpr unsigned kBarrierPoison = 0x80000000u;

// ---------------------------------------------------------------------------
// shared device pieces
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

// 32-bit exclusive scan of one value per thread over the CTA (s_warp: 32 ints).
__device__ __forceinline__ int cta_exclusive_scan32(int x, int *s_warp, int *total) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int inc = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int wv = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wv, d);
            if (lane >= d) wv += o;
        }
        if (lane < nwarps) s_warp[lane] = wv;
    }
    __syncthreads();
    const int base = warp > 0 ? s_warp[warp - 1] : 0;
    *total = s_warp[nwarps - 1];
    __syncthreads();
    return base + inc - x;
}

// A set of whole warps of one CTA that works as a unit: thread tid of nthr
// (warp-aligned, tid = threadIdx.x - first thread), synchronised by named
// barrier BAR (0: the whole CTA with __syncthreads). The barrier id is a
// compile-time constant so that a kernel reserves only the barriers it uses.
template <int BAR>
struct ThreadGroup {
    int tid, nthr;
    __device__ __forceinline__ void sync() const {
        if (BAR == 0)
            __syncthreads();
        else
            asm volatile("bar.sync %0, %1;" ::"n"(BAR), "r"(nthr) : "memory");
    }
};

__device__ __forceinline__ ThreadGroup<0> whole_cta() { return ThreadGroup<0>{(int)threadIdx.x, (int)blockDim.x}; }

// cta_exclusive_scan32 over a ThreadGroup.
template <int BAR>
__device__ __forceinline__ int group_exclusive_scan32(int x, int *s_warp, int *total, const ThreadGroup<BAR> &g) {
    const int lane = g.tid & 31;
    const int warp = g.tid >> 5;
    const int nwarps = g.nthr >> 5;
    int inc = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) s_warp[warp] = inc;
    g.sync();
    if (warp == 0) {
        int wv = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wv, d);
            if (lane >= d) wv += o;
        }
        if (lane < nwarps) s_warp[lane] = wv;
    }
    g.sync();
    const int base = warp > 0 ? s_warp[warp - 1] : 0;
    *total = s_warp[nwarps - 1];
    g.sync();
    return base + inc - x;
}

// Threads that share one expert's work in a CTA of nw warps: the largest power
// of two <= min(32 nw / E, nw, 32), at least 1.
__device__ __forceinline__ int threads_per_expert(int32_t E, int nw) {
    int cap = (32 * nw) / E;
    if (cap > nw) cap = nw;
    if (cap > 32) cap = 32;
    int t = 1;
    while (2 * t <= cap) t <<= 1;
    return t;
}

// Ranks the CTA's np pairs held in tile_e in token order; warp w takes the
// contiguous pairs [w ppw, min(np, (w + 1) ppw)). On return (after a CTA
// barrier): tile_r[p] is p's rank among the same warp's earlier pairs of its
// expert (-1 for an id outside [0, E)); cnt[w][e] holds the number of pairs
// of expert e in warps < w; and cta_count[e * stride] the CTA's total.
//
// A warp ranks 32 consecutive pairs per step: __match_any_sync groups the
// lanes holding the same expert, a lane's rank inside the step is the number
// of lower lanes in its group, and the group's highest lane advances the
// warp's shared counter for that expert. The k experts of one token are
// distinct, so lanes of one token never match each other.
__device__ void cta_rank_pairs(const int32_t *tile_e, int np, int ppw, int32_t E, int32_t *cnt, int32_t *tile_r,
                               int32_t *cta_count, int64_t stride) {
    const int nw = blockDim.x >> 5;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();

    int32_t *wc = cnt + warp * E;
    const int p_begin = warp * ppw;
    const int p_end = p_begin + ppw < np ? p_begin + ppw : np;
    const unsigned below = (1u << lane) - 1u;
    const unsigned above = ~((2u << lane) - 1u);
    for (int p0 = p_begin; p0 < p_end; p0 += 32) {
        const int p = p0 + lane;
        const int e = p < p_end ? tile_e[p] : -1;
        const bool valid = (unsigned)e < (unsigned)E;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : E + lane);
        const int basec = valid ? wc[e] : 0;
        __syncwarp();
        if (valid && (peers & above) == 0) wc[e] = basec + __popc(peers);
        if (p < p_end) tile_r[p] = valid ? basec + __popc(peers & below) : -1;
        __syncwarp();
    }
    __syncthreads();

    // Exclusive scan over the warps, per expert. tpe consecutive threads share
    // an expert, each scanning a contiguous run of nw / tpe warps; a shuffle
    // scan joins the runs. Rounds are uniform across the CTA (shuffles need
    // every lane).
    const int tpe = threads_per_expert(E, nw);
    const int sub = (int)threadIdx.x % tpe;
    const int runlen = nw / tpe;
    const int per_round = blockDim.x / tpe;
    for (int base = 0; base < E; base += per_round) {
        const int e0 = base + (int)threadIdx.x / tpe;
        const bool act = e0 < E;
        int local = 0;
        if (act)
            for (int w = sub * runlen; w < (sub + 1) * runlen; ++w) local += cnt[w * E + e0];
        int incl = local;
        for (int d = 1; d < tpe; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, d, tpe);
            if (sub >= d) incl += o;
        }
        if (act) {
            int run = incl - local;
            for (int w = sub * runlen; w < (sub + 1) * runlen; ++w) {
                const int c = cnt[w * E + e0];
                cnt[w * E + e0] = run;
                run += c;
            }
            if (sub == tpe - 1) cta_count[(int64_t)e0 * stride] = incl;
        }
    }
    __syncthreads();
}

// Rank phase for the CTA's tokens [t_cta, t_cta + tpw nw): loads their pairs
// into tile_e (tpw tokens per warp) and ranks them with cta_rank_pairs.
__device__ void cta_rank_tokens(const int32_t *__restrict__ idx, int32_t T, int32_t E, int32_t k, int64_t t_cta,
                                int32_t *cnt, int32_t *tile_e, int32_t *tile_r, int32_t *cta_count,
                                int64_t stride, int tpw = 32) {
    const int nw = blockDim.x >> 5;
    const int64_t left = (int64_t)T - t_cta;
    const int ntok = left <= 0 ? 0 : (left >= tpw * nw ? tpw * nw : (int)left);
    const int np = ntok * k;
    for (int i = threadIdx.x; i < np; i += blockDim.x) tile_e[i] = __ldcg(idx + t_cta * k + i);
    cta_rank_pairs(tile_e, np, tpw * k, E, cnt, tile_r, cta_count, stride);
}

// Largest i in [0, n) with P[i] <= x, for P non-decreasing with P[0] <= x.
// 4-ary search: three independent pivot compares narrow the range 4x per step.
__device__ __noinline__ int32_t quaternary_search(const int32_t *P, int32_t n, int32_t x) {
    int32_t lo = 0, hi = n;  // answer in [lo, hi), P[lo] <= x
    while (hi - lo > 1) {
        const int32_t len = hi - lo;
        const int32_t q1 = lo + len / 4, q2 = lo + len / 2, q3 = lo + (3 * len) / 4;
        const bool c1 = P[q1] <= x;
        const bool c2 = P[q2] <= x;
        const bool c3 = P[q3] <= x;
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

// floor(N w / W) for the share boundaries (32-bit whenever it cannot overflow).
__device__ __forceinline__ int32_t share_bound(int32_t N, int32_t w, int32_t W) {
    if ((uint64_t)(uint32_t)N * (uint32_t)W <= 0xffffffffull) return (int32_t)((uint32_t)N * (uint32_t)w / (uint32_t)W);
    return (int32_t)((int64_t)N * w / W);
}

// The two-class chunk schedule (no pod tier), built by one whole CTA from rank
// offsets in shared memory. Class 0 (near) is ranks [n_lo, n_hi) of
// self_rank's node; class 1 (far) is [0, n_lo) followed by [n_hi, R). s_P (R + 2 ints of shared memory)
// receives each class's prefix sums P_c[i] = rows in its first i ranks. A
// worker finds the first and last rank its share touches by two quaternary
// searches per class, counts the non-empty ranks in between, and after a CTA
// scan over the counts writes its chunks.
__device__ void build_schedule_two_tiers(const int32_t *s_roff, int32_t R, int32_t W, int32_t ranks_per_node,
                                         int32_t self_rank, ep_chunk *chunks, int32_t *n_chunks,
                                         int32_t *worker_begin, int *s_warp, int32_t *s_P) {
    const int32_t node = self_rank / ranks_per_node;
    const int32_t n_lo = node * ranks_per_node;
    const int32_t n_hi = n_lo + ranks_per_node < R ? n_lo + ranks_per_node : R;
    const int32_t n0 = n_hi - n_lo, n1 = R - n0;
    int32_t *P1 = s_P;           // far class: n1 + 1 entries
    int32_t *P0 = s_P + n1 + 1;  // near class: n0 + 1 entries
    for (int32_t i = threadIdx.x; i <= n1; i += blockDim.x)
        P1[i] = i <= n_lo ? s_roff[i] : s_roff[n_lo] + (s_roff[i + n0] - s_roff[n_hi]);
    for (int32_t i = threadIdx.x; i <= n0; i += blockDim.x) P0[i] = s_roff[n_lo + i] - s_roff[n_lo];
    __syncthreads();
    const int32_t N[2] = {P0[n0], P1[n1]};

    int carry = 0;
    for (int32_t wb = 0; wb < W; wb += blockDim.x) {
        const int32_t w = wb + (int32_t)threadIdx.x;
        int32_t first[2] = {0, 0}, last[2] = {-1, -1}, lo[2] = {0, 0}, hi[2] = {0, 0};
        int cnt = 0;
        if (w < W) {
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const int32_t *P = c ? P1 : P0;
                const int32_t n = c ? n1 : n0;
                lo[c] = share_bound(N[c], w, W);
                hi[c] = share_bound(N[c], w + 1, W);
                if (hi[c] > lo[c]) {
                    first[c] = quaternary_search(P, n, lo[c]);
                    last[c] = quaternary_search(P, n, hi[c] - 1);
                    for (int32_t i = first[c]; i <= last[c]; ++i) cnt += P[i + 1] > P[i] ? 1 : 0;
                }
            }
        }
        int tile_total;
        const int pos0 = carry + cta_exclusive_scan32(cnt, s_warp, &tile_total);
        if (w < W) {
            worker_begin[w] = pos0;
            int pos = pos0;
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 1 - cc;  // other-node traffic first
                const int32_t *P = c ? P1 : P0;
                for (int32_t i = first[c]; i <= last[c]; ++i) {
                    if (P[i + 1] == P[i]) continue;
                    const int32_t r = c ? (i < n_lo ? i : i + n0) : n_lo + i;
                    const int32_t a = lo[c] > P[i] ? lo[c] : P[i];
                    const int32_t bnd = hi[c] < P[i + 1] ? hi[c] : P[i + 1];
                    ep_chunk ch;
                    ch.worker = w;
                    ch.hop_class = c;
                    ch.dst_rank = r;
                    ch.row_begin = s_roff[r] + (a - P[i]);
                    ch.row_count = bnd - a;
                    chunks[pos++] = ch;
                }
            }
        }
        carry += tile_total;
    }
    if (threadIdx.x == 0) {
        worker_begin[W] = carry;
        *n_chunks = carry;
    }
}

// The ranks of one hop class: at most two runs of consecutive ranks,
// [a0, a0 + n0) then [a1, a1 + n - n0), in ascending order.
struct ClassRuns {
    int32_t a0, n0, a1, n;
    __device__ __forceinline__ int32_t rank(int32_t i) const { return i < n0 ? a0 + i : a1 + (i - n0); }
};

// Class c's runs for the sending rank's node [nl, nh) inside its pod [pl, ph)
// (the pod is [0, R) when there is no pod tier): class 0 = the node, class 1
// = the pod around it, class 2 = everything outside the pod.
__device__ __forceinline__ ClassRuns class_runs(int c, int32_t R, int32_t nl, int32_t nh, int32_t pl, int32_t ph) {
    ClassRuns q;
    if (c == 0) {
        q.a0 = nl; q.n0 = nh - nl; q.a1 = nh; q.n = nh - nl;
    } else if (c == 1) {
        q.a0 = pl; q.n0 = nl - pl; q.a1 = nh; q.n = (nl - pl) + (ph - nh);
    } else {
        q.a0 = 0; q.n0 = pl; q.a1 = ph; q.n = pl + (R - ph);
    }
    return q;
}

// The chunk schedule, built by a group of threads from rank offsets in shared
// memory (NC = 2 or 3 hop classes). s_P (R + 3 ints of shared memory)
// receives each class's prefix sums P_c[i] = rows in the class's first i
// ranks. A worker finds the first and last rank its share of each class
// touches by two quaternary searches, counts the non-empty ranks in between,
// and after a group scan over the counts writes its chunks, farthest class
// first. Used for three classes; the two-class table has its own builder
// above, which measured faster inside the layout and fused kernels (this one,
// inlined there or called, cost them 2-4 us more).
template <int NC, int BAR>
__device__ __noinline__ void build_schedule_nc(const int32_t *s_roff, int32_t R, int32_t W, HopTiers h,
                                               ep_chunk *chunks, int32_t *n_chunks, int32_t *worker_begin,
                                               int *s_warp, int32_t *s_P, ThreadGroup<BAR> g) {
    const int32_t nl = h.self_rank / h.ranks_per_node * h.ranks_per_node;
    const int32_t nh = nl + h.ranks_per_node < R ? nl + h.ranks_per_node : R;
    const int32_t pl = NC == 3 ? h.self_rank / h.ranks_per_pod * h.ranks_per_pod : 0;
    const int32_t ph = NC == 3 ? (pl + h.ranks_per_pod < R ? pl + h.ranks_per_pod : R) : R;
    ClassRuns q[NC];
    int32_t *P[NC];
    int32_t base = 0;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        q[c] = class_runs(c, R, nl, nh, pl, ph);
        P[c] = s_P + base;
        base += q[c].n + 1;
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const ClassRuns qc = q[c];
        for (int32_t i = g.tid; i <= qc.n; i += g.nthr)
            P[c][i] = i <= qc.n0 ? s_roff[qc.a0 + i] - s_roff[qc.a0]
                                 : (s_roff[qc.a0 + qc.n0] - s_roff[qc.a0]) + (s_roff[qc.a1 + (i - qc.n0)] - s_roff[qc.a1]);
    }
    g.sync();
    int32_t N[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) N[c] = P[c][q[c].n];

    int carry = 0;
    for (int32_t wb = 0; wb < W; wb += g.nthr) {
        const int32_t w = wb + (int32_t)g.tid;
        int32_t first[NC], last[NC], lo[NC], hi[NC];
        int cnt = 0;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            first[c] = 0;
            last[c] = -1;
            lo[c] = 0;
            hi[c] = 0;
        }
        if (w < W) {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                lo[c] = share_bound(N[c], w, W);
                hi[c] = share_bound(N[c], w + 1, W);
                if (hi[c] > lo[c]) {
                    first[c] = quaternary_search(P[c], q[c].n, lo[c]);
                    last[c] = quaternary_search(P[c], q[c].n, hi[c] - 1);
                    for (int32_t i = first[c]; i <= last[c]; ++i) cnt += P[c][i + 1] > P[c][i] ? 1 : 0;
                }
            }
        }
        int tile_total;
        const int pos0 = carry + group_exclusive_scan32(cnt, s_warp, &tile_total, g);
        if (w < W) {
            worker_begin[w] = pos0;
            int pos = pos0;
#pragma unroll
            for (int c = NC - 1; c >= 0; --c) {
                const int32_t *Pc = P[c];
                for (int32_t i = first[c]; i <= last[c]; ++i) {
                    if (Pc[i + 1] == Pc[i]) continue;
                    const int32_t r = q[c].rank(i);
                    const int32_t a = lo[c] > Pc[i] ? lo[c] : Pc[i];
                    const int32_t bnd = hi[c] < Pc[i + 1] ? hi[c] : Pc[i + 1];
                    ep_chunk ch;
                    ch.worker = w;
                    ch.hop_class = c;
                    ch.dst_rank = r;
                    ch.row_begin = s_roff[r] + (a - Pc[i]);
                    ch.row_count = bnd - a;
                    chunks[pos++] = ch;
                }
            }
        }
        carry += tile_total;
    }
    if (g.tid == 0) {
        worker_begin[W] = carry;
        *n_chunks = carry;
    }
}

template <int BAR>
__device__ __forceinline__ void cta_build_schedule(const int32_t *s_roff, int32_t R, int32_t W, HopTiers h,
                                                   ep_chunk *chunks, int32_t *n_chunks, int32_t *worker_begin,
                                                   int *s_warp, int32_t *s_P, ThreadGroup<BAR> g) {
    if (h.ranks_per_pod > 0)
        build_schedule_nc<3, BAR>(s_roff, R, W, h, chunks, n_chunks, worker_begin, s_warp, s_P, g);
    else if (BAR == 0)
        build_schedule_two_tiers(s_roff, R, W, h.ranks_per_node, h.self_rank, chunks, n_chunks, worker_begin, s_warp,
                                 s_P);
    else
        build_schedule_nc<2, BAR>(s_roff, R, W, h, chunks, n_chunks, worker_begin, s_warp, s_P, g);
}

// ---------------------------------------------------------------------------
// fused path
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier for co-resident CTAs: after a CTA barrier, thread 0 arrives
// with a release add and polls with acquire loads, then a CTA barrier releases
// the other threads. Bounded: a CTA that has polled max_polls times gives up
// by setting the counter's top bit (kBarrierPoison) with a compare-and-swap
// that only succeeds on a count below `expected`. So the top bit is set only
// while the barrier is incomplete, and once set it is seen by every CTA that
// reads the counter later: they all return false, and no CTA of the launch
// goes on with another's results missing (in particular none writes a chunk
// count over the -1 a failing CTA leaves in *n_chunks). If the swap finds that
// the last arrival came in meanwhile, the CTA goes on as if it had seen it.
// The success path costs nothing extra: the check reads the value the poll
// already loaded. The counter must be zero before the launch.
//
// grid_arrive and grid_wait are its two halves, for a CTA with work of its own
// (touching nothing the other CTAs wait for) between its arrival and its wait.
__device__ __forceinline__ void grid_arrive(unsigned *arrivals) {
    __syncthreads();
    // The CTA barrier above orders every thread's writes before this release
    // add (release is cumulative); the acquire loads in grid_wait and its CTA
    // barrier order every thread's later reads after the wait. No separate
    // fence is needed on either side.
    if (threadIdx.x == 0) red_release_gpu_add(arrivals, 1u);
}
__device__ __forceinline__ bool grid_wait(unsigned *arrivals, unsigned expected, unsigned max_polls = kBarrierSpinLimit) {
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        unsigned spins = 0, v;
        while ((v = ld_acquire_gpu(arrivals)) < expected) {
            if (++spins > max_polls) {
                // Each failed swap means the counter moved (an arrival, or another
                // CTA's poison): at most expected + 1 rounds.
                for (;;) {
                    const unsigned prev = atomicCAS(arrivals, v, v | kBarrierPoison);
                    if (prev == v) {
                        v |= kBarrierPoison;
                        break;
                    }
                    v = prev;
                    if ((v & kBarrierPoison) != 0u || v >= expected) break;
                }
                __threadfence();  // acquire side for the case that the last arrival did come in
                break;
            }
            if (spins > 64) __nanosleep(32);
        }
        s_ok = (v & kBarrierPoison) == 0u && v >= expected;
    }
    __syncthreads();
    return s_ok != 0;
}
__device__ bool grid_barrier(unsigned *arrivals, unsigned expected, unsigned max_polls = kBarrierSpinLimit) {
    grid_arrive(arrivals);
    return grid_wait(arrivals, expected, max_polls);
}

// ---------------------------------------------------------------------------
// Count table exchanged without a grid barrier
// ---------------------------------------------------------------------------
// CTA b of a cooperative launch publishes its per-expert counts as row b of a
// [CTA][E] table of 32-bit words in global memory, each entry marked by its top
// bit (kCountValid), and every CTA reads the whole table by polling each entry
// until it carries the mark. A reader thus starts on the rows already there
// while later CTAs still rank, and needs no arrival counter: one round of
// polls replaces the barrier's arrive-and-poll plus the table read after it.
// The table must be zero before the launch. Entries are self-contained (one
// 32-bit word each), so relaxed loads suffice; nothing else crosses CTAs.
//
// Bounded: a reader that has polled max_polls times swaps kCountPoison into
// every entry it still misses (compare-and-swap from zero). The owner publishes
// with a compare-and-swap from zero too, so a poisoned entry never becomes
// valid; every CTA needs every entry, so all of them fail and none goes on
// with a count missing (a CTA that fails writes *n_chunks = -1 and no chunk
// count can overwrite it). The owner learns from its own swaps that it was
// late and fails as well.
constexpr unsigned kCountValid = 0x80000000u;
constexpr unsigned kCountPoison = 0x40000000u;

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Publishes row `row` from own[0, E) (own[e] < 2^30). Each thread swaps at
// most four entries (E <= 4 blockDim.x); it returns the OR of the values its
// swaps found, non-zero when an entry was not zero any more (poisoned by a
// reader that gave up). Read the result late: the swaps complete meanwhile.
struct TablePublish {
    unsigned old[4];
    __device__ __forceinline__ bool late() const { return (old[0] | old[1] | old[2] | old[3]) != 0u; }
};
__device__ __forceinline__ TablePublish table_publish(unsigned *row, const int32_t *own, int32_t E) {
    TablePublish r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = (int)threadIdx.x + i * (int)blockDim.x;
        r.old[i] = e < E ? atomicCAS(row + e, 0u, kCountValid | (unsigned)own[e]) : 0u;
    }
    return r;
}

// Sums column e of the table over rows q = sub, sub + step, ... < nb (tot)
// and over those rows below b (pre), polling every entry until it is valid,
// with up to NB loads in flight; row `skip` is left out (the caller's own,
// which it holds already: -1 for none). False if it gave up after max_polls
// rounds of polls (poisoning what it still missed) or met a poisoned entry.
template <int NB = 32>
__device__ __forceinline__ bool table_column_sums(unsigned *tab, int32_t E, int e, int sub, int step, int nb,
                                                  int b, int skip, uint32_t max_polls, int &tot, int &pre) {
    tot = 0;
    pre = 0;
    for (int q0 = sub; q0 < nb; q0 += NB * step) {
        unsigned cv[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int q = q0 + u * step;
            cv[u] = q < nb && q != skip ? ld_relaxed_gpu(tab + (int64_t)q * E + e) : kCountValid;
        }
        for (uint32_t polls = 0;; ++polls) {
            bool all = true, poisoned = false;
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                all = all && (cv[u] & kCountValid) != 0u;
                poisoned = poisoned || cv[u] == kCountPoison;
            }
            if (all) break;
            if (poisoned) return false;
            if (polls >= max_polls) {
#pragma unroll
                for (int u = 0; u < NB; ++u) {
                    const int q = q0 + u * step;
                    if ((cv[u] & kCountValid) == 0u) {
                        const unsigned prev = atomicCAS(tab + (int64_t)q * E + e, 0u, kCountPoison);
                        cv[u] = prev == 0u ? kCountPoison : prev;
                    }
                }
                bool now = true;
#pragma unroll
                for (int u = 0; u < NB; ++u) now = now && (cv[u] & kCountValid) != 0u;
                if (!now) return false;
                break;  // the missing entries arrived just in time
            }
            if (polls > 64) __nanosleep(32);
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int q = q0 + u * step;
                if ((cv[u] & kCountValid) == 0u) cv[u] = ld_relaxed_gpu(tab + (int64_t)q * E + e);
            }
        }
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int c = (int)(cv[u] & ~kCountValid);  // 0 for the padding past nb and row skip
            tot += c;
            pre += q0 + u * step < b ? c : 0;
        }
    }
    return true;
}

}  // namespace
}  // namespace ep

// fused_kernel.cuh -- the small-batch dispatch kernel of ep_dispatch_fused
// (fused.cu has its description and the host code).
#pragma once

#include "block_common.cuh"
#include "flag_ops.cuh"
#include "route_token.cuh"

namespace ep {
namespace {

constexpr int kFusedWarps = 8;
constexpr int kFusedThreads = 32 * kFusedWarps;
constexpr int kMaxTilePairs = 2048;   // tokens per tile * k
constexpr int kMaxFusedStages = 8;
constexpr int kMaxFusedCTAs = 1024;
constexpr uint32_t kFusedMaxPolls = 1u << 22;
constexpr size_t kFusedSmemLimit = 200 * 1024;
constexpr int kSplitMaxT = 160;  // split form up to this many tokens
// Above this many tokens the route, layout and dispatch kernels beat the fused
// kernel (measured per layer, E = 256, k = 8, H = 7168: T = 1536 78.4 against
// 81.1 us, T = 2000 98.0 against 94.9, T = 2400 113.7 against 110.2; the lines
// cross near 1760).
constexpr int kFusedMaxT = 1760;
constexpr int64_t kHistMaxPairs = 16384;
constexpr int kFusedTileCap = 128;  // single-role form up to 1024 tokens: at most this many tiles

size_t align128(size_t b) { return (b + 127) & ~(size_t)127; }

// Shared-memory carve-up, in this order (each piece 128-byte aligned):
// stages, mbarriers, tile_e, tile_r, tile_s, cnt [8][E], group logits [8][E],
// cand [8][32] int2, pick [8][32] int2, s_tot [E], s_eoff [E+2], s_base [E],
// s_roff [R+1], s_P [R+3], s_col [E + 1024] (the column scan's counts).
struct SmemLayout {
    size_t stages, bars, tile_e, tile_r, tile_s, cnt, glog, cand, pick, tot, eoff, base, roff, P, col, bytes;
};

__host__ __device__ inline SmemLayout smem_layout(int ns, int row_pad, int tb, int32_t k, int32_t E, int32_t R,
                                                  bool groups) {
    SmemLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += (bytes + 127) & ~(size_t)127;
        return at;
    };
    L.stages = take((size_t)ns * row_pad);
    L.bars = take(sizeof(uint64_t) * kMaxFusedStages);
    L.tile_e = take(sizeof(int32_t) * (size_t)tb * k);
    L.tile_r = take(sizeof(int32_t) * (size_t)tb * k);
    L.tile_s = take(sizeof(int32_t) * (size_t)tb * k);
    L.cnt = take(sizeof(int32_t) * kFusedWarps * (size_t)E);
    L.glog = take(groups ? sizeof(float) * kFusedWarps * (size_t)E : 0);
    L.cand = take(sizeof(int2) * kFusedWarps * 32);
    L.pick = take(sizeof(int2) * kFusedWarps * 32);
    L.tot = take(sizeof(int32_t) * (size_t)E);
    L.eoff = take(sizeof(int32_t) * ((size_t)E + 2));
    L.base = take(sizeof(int32_t) * (size_t)E);
    L.roff = take(sizeof(int32_t) * ((size_t)R + 1));
    L.P = take(sizeof(int32_t) * ((size_t)R + 3));
    L.col = take(sizeof(int32_t) * ((size_t)E + kMaxFusedCTAs));  // my experts x tiles <= E + nb
    L.bytes = o;
    return L;
}

struct FusedArgs {
    const float *logits;
    const char *x;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *expert_count, *expert_offset, *rank_count, *rank_offset, *slot;
    ep_chunk *chunks;
    int32_t *n_chunks, *worker_begin;
    char *send;
    int32_t *meta;
    int32_t *counts;  // [nb][E] per-tile counts
    int32_t *bases;   // [nb][E] per-tile base inside each expert
    int32_t *totals;  // [E]
    unsigned *sync;   // [2] arrivals of the two grid barriers
    int32_t *err;
    int32_t T, H, E, R, k, n_groups, topk_groups, renormalize, W;
    HopTiers tiers;
    int32_t nb, tb, ns, row_pad;
    int32_t early_dependents;  // signal dependents at the dispatch phase (small sends only)
    int32_t sched_cta;         // 1: CTA nb holds no tile and builds the chunk schedule
    // Split form only: n_data data CTAs after the tile (and schedule) CTAs move
    // the rows in units of unit_rows rows of one token (1, 2, 4, ... or k = the
    // whole token; the last unit of a token may hold fewer); ready[q] is set
    // (release) once tile q's slots are written.
    int32_t n_data, unit_rows;
    unsigned *ready;
    // 1: after barrier C every CTA reads all of topk_idx and counts, in shared
    // memory, every expert's pairs (the totals) and those of the tokens before
    // its tile (its bases); steps D and E are skipped.
    int32_t hist;
};

// The rows of one token (up to unit_rows of them from top-k position jj0), moved by
// a data CTA of the split form: wait until the tile that owns the token has
// published its slots, then bulk-store the staged x row to each slot.
__device__ __forceinline__ bool split_data_unit(const FusedArgs &a, int64_t t, int jj0, unsigned char *stage,
                                                uint64_t *bar, uint32_t parity, int lane) {
    const int32_t row_bytes = a.H * 2;
    const int64_t rows = (int64_t)a.T * a.k;
    // tile q holds tokens [floor(q T / nb), floor((q + 1) T / nb)): the owner of t
    const int q = (int)(((t + 1) * a.nb + a.T - 1) / a.T) - 1;
    if (!warp_wait_flag(a.ready + q, kFusedMaxPolls)) return false;  // each lane's slot load is ordered after it
    if (!mbar_wait_bounded(bar, parity, kFusedMaxPolls)) return false;
    if (a.early_dependents) grid_launch_dependents();
    if (lane < a.unit_rows) {
        const int j = jj0 + lane;
        const int sv = j < a.k ? a.slot[t * a.k + j] : -1;
        if (sv >= 0 && (int64_t)sv < rows) {
            bulk_s2g(a.send + (int64_t)sv * row_bytes, stage, (uint32_t)row_bytes);
            a.meta[sv] = (int32_t)(t * a.k + j);
        }
        bulk_commit();
    }
    return true;
}

// kSplit: the split form (tile CTAs, the schedule CTA, data CTAs).
template <int VPL, bool kSplit>
__global__ void __launch_bounds__(kFusedThreads, 2) dispatch_fused_kernel(FusedArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_warp32[32];
    const SmemLayout L = smem_layout(a.ns, a.row_pad, a.tb, a.k, a.E, a.R, a.n_groups > 1);
    unsigned char *stages = smem + L.stages;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bars);
    int32_t *tile_e = reinterpret_cast<int32_t *>(smem + L.tile_e);
    int32_t *tile_r = reinterpret_cast<int32_t *>(smem + L.tile_r);
    int32_t *tile_s = reinterpret_cast<int32_t *>(smem + L.tile_s);
    int32_t *cnt = reinterpret_cast<int32_t *>(smem + L.cnt);
    float *glog = reinterpret_cast<float *>(smem + L.glog);
    int2 *cand = reinterpret_cast<int2 *>(smem + L.cand);
    int2 *pick = reinterpret_cast<int2 *>(smem + L.pick);
    int32_t *s_tot = reinterpret_cast<int32_t *>(smem + L.tot);
    int32_t *s_eoff = reinterpret_cast<int32_t *>(smem + L.eoff);
    int32_t *s_base = reinterpret_cast<int32_t *>(smem + L.base);
    int32_t *s_roff = reinterpret_cast<int32_t *>(smem + L.roff);
    int32_t *s_P = reinterpret_cast<int32_t *>(smem + L.P);
    int32_t *s_col = reinterpret_cast<int32_t *>(smem + L.col);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int b = blockIdx.x;
    const int E = a.E, k = a.k;
    // The schedule CTA (index nb, when present) holds no tile: it only joins the
    // two grid barriers, then builds the chunk schedule while the tile CTAs
    // write their slots and rows.
    const bool sched_only = a.sched_cta && b == a.nb;
    const unsigned arrivals = (unsigned)(a.nb + a.sched_cta);
    // (the split form moves at most 160 tokens' pairs: always the count of all
    // picks, and its instances carry no column scan)
    const bool hist = kSplit || a.hist;
    // tile b = tokens [floor(b T / nb), floor((b + 1) T / nb)): every CTA within one token of the others
    const int64_t t0 = sched_only ? a.T : (int64_t)b * a.T / a.nb;
    const int ntok = sched_only ? 0 : (int)((int64_t)(b + 1) * a.T / a.nb - t0);  // may be 0 when T < nb
    const int np = ntok * k;
    const int32_t row_bytes = a.H * 2;

    if (kSplit && b >= a.nb + a.sched_cta) {
        // Data CTA (split form): its first x row is fetched at once, while
        // the tile CTAs compute the metadata; then, unit by unit, it waits for
        // the owning tile's flag and stores the rows. Warp 0 does it all.
        if (warp != 0) return;
        const int upt = (k + a.unit_rows - 1) / a.unit_rows;  // units per token
        const int64_t n_units = (int64_t)a.T * upt;
        const int64_t j = b - a.nb - a.sched_cta;
        if (lane == 0) {
            mbar_init(&bar[0], 1);
            fence_mbar_init();
        }
        __syncwarp();
        int64_t cur = -1;  // token in the stage
        uint32_t loads = 0;
        bool good = true;
        for (int64_t u = j; good && u < n_units; u += a.n_data) {
            const int64_t t = upt == 1 ? u : u / upt;
            const int jj0 = upt == 1 ? 0 : (int)(u - t * upt) * a.unit_rows;
            if (t != cur) {
                if (cur >= 0) {
                    if (lane < a.unit_rows) bulk_wait_read<0>();  // the stage's previous row is read out
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar[0], (uint32_t)row_bytes);
                    bulk_g2s(stages, a.x + t * row_bytes, (uint32_t)row_bytes, &bar[0]);
                }
                if (cur < 0) grid_dependency_wait();  // the ready flags are zeroed by the grid before this one
                ++loads;
                cur = t;
            }
            good = split_data_unit(a, t, jj0, stages, &bar[0], (loads - 1) & 1u, lane);
        }
        if (!good) {
            if (lane == 0) atomicOr(a.err, kErrFusedWait);
            mbar_wait_bounded(&bar[0], (loads - 1) & 1u, kFusedMaxPolls);  // the last load lands before exit
        }
        if (lane < a.unit_rows) bulk_wait<0>();
        return;
    }

    // 0. start the tile's first x rows into shared memory
    if (!kSplit && a.ns > 0 && threadIdx.x == 0) {
        for (int s = 0; s < a.ns; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        for (int s = 0; s < a.ns && s < ntok; ++s) {
            mbar_arrive_expect_tx(&bar[s], (uint32_t)row_bytes);
            bulk_g2s(stages + (size_t)s * a.row_pad, a.x + (t0 + s) * row_bytes, (uint32_t)row_bytes, &bar[s]);
        }
    }

    if (hist)
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            s_tot[e] = 0;
            s_base[e] = 0;
        }
    // A. route the tile, one warp per token
    for (int i = warp; i < ntok; i += kFusedWarps) {
        const int64_t t = t0 + i;
        int e;
        float w;
        route_token<VPL, true>(a.logits + t * E, E, k, a.n_groups, a.topk_groups, a.renormalize, lane,
                               glog + warp * E, cand + warp * 32, pick + warp * 32, e, w);
        if (lane < k) {
            tile_e[i * k + lane] = e;
            a.topk_idx[t * k + lane] = e;
            a.topk_w[t * k + lane] = w;
        }
        __syncwarp();
    }
    __syncthreads();

    // B. rank the tile's pairs; publish the tile's counts
    // C. (a single CTA needs no grid barrier: after a CTA barrier its own
    // global writes are visible to all its threads). The barrier words and
    // ready flags are zeroed by the grid launched before this one.
    // With hist the others need only this tile's picks (in topk_idx since A):
    // arrive first and rank while they arrive (the counts stay in shared
    // memory, as a single CTA's do: they are its totals). One call site each,
    // to keep the kernel's code short.
    const int ppw = np > 0 ? (np + kFusedWarps - 1) / kFusedWarps : 1;
    if (hist) {
        grid_dependency_wait();
        grid_arrive(&a.sync[0]);
    }
    if (!sched_only)
        cta_rank_pairs(tile_e, np, ppw, E, cnt, tile_r,
                       arrivals == 1 ? s_tot : (hist ? s_col : a.counts + (int64_t)b * E), 1);
    if (!hist) {
        grid_dependency_wait();
        if (arrivals > 1) grid_arrive(&a.sync[0]);
    }
    bool ok = arrivals > 1 ? grid_wait(&a.sync[0], arrivals) : (__syncthreads(), true);
    // The schedule CTA's last step (the schedule) need not hold back a
    // dependent's launch, which waits for this whole grid before it touches
    // memory anyway (measured per layer: T = 4 -1.1 us, T = 8 -0.5 to -1.5,
    // T = 1 Zipf -1.3, uniform +0.2, T = 32 -0.25, T = 64 and 128 even).
    if (sched_only && a.early_dependents) grid_launch_dependents();
    // C'. (hist) every tile's picks are in topk_idx now: the expert totals and
    // this tile's bases counted from them directly, 8 loads in flight a thread.
    if (ok && hist) {
        const int64_t n = (int64_t)a.T * k, before = t0 * k;
        for (int64_t i0 = threadIdx.x; i0 < n; i0 += 8 * (int64_t)blockDim.x) {
            int ev[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t i = i0 + (int64_t)u * blockDim.x;
                ev[u] = i < n ? __ldcg(a.topk_idx + i) : -1;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t i = i0 + (int64_t)u * blockDim.x;
                const int e = ev[u];
                if ((unsigned)e < (unsigned)E) {
                    atomicAdd(&s_tot[e], 1);
                    if (i < before) atomicAdd(&s_base[e], 1);
                }
            }
        }
    }

    // D. column scan: CTA b owns experts b, b + nb, ...; all their counts over
    // every tile are read in one batch, then scanned over the tiles. (A single
    // CTA skips it and the global reads of step F: its counts, kept in shared
    // memory, are the totals and its bases are zero: T = 1 and 8 -1.4 to -2.3
    // us per layer.)
    if (ok && !sched_only && arrivals > 1 && !hist) {
        const int nb = a.nb;
        const int my_n = b < E ? (E - b + nb - 1) / nb : 0;
        const int nv = my_n * nb;
        for (int v = threadIdx.x; v < nv; v += blockDim.x) {
            const int q = v % nb;
            const int e = b + (v / nb) * nb;
            s_col[v] = __ldcg(a.counts + (int64_t)q * E + e);
        }
        __syncthreads();
        if (nb <= 64) {
            // many experts, few tiles: one thread walks each expert's tiles
            for (int j = threadIdx.x; j < my_n; j += blockDim.x) {
                const int e = b + j * nb;
                int run = 0;
                for (int q = 0; q < nb; ++q) {
                    a.bases[(int64_t)q * E + e] = run;
                    run += s_col[j * nb + q];
                }
                a.totals[e] = run;
            }
        } else {
            // few experts, many tiles: the CTA scans one expert's tiles at a time
            for (int j = 0; j < my_n; ++j) {
                const int e = b + j * nb;
                const int per = (nb + blockDim.x - 1) / blockDim.x;
                const int q0 = threadIdx.x * per;
                int local = 0;
                for (int q = q0; q < q0 + per && q < nb; ++q) local += s_col[j * nb + q];
                int total;
                int run = cta_exclusive_scan32(local, s_warp32, &total);
                for (int q = q0; q < q0 + per && q < nb; ++q) {
                    a.bases[(int64_t)q * E + e] = run;
                    run += s_col[j * nb + q];
                }
                if (threadIdx.x == 0) a.totals[e] = total;
            }
        }
    }
    // E.
    if (ok) ok = arrivals > 1 && !hist ? grid_barrier(&a.sync[1], arrivals) : (__syncthreads(), true);

    if (ok) {
        // F. expert offsets and this tile's slots
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            if (arrivals == 1) {
                s_base[e] = 0;
            } else if (!hist) {
                s_tot[e] = __ldcg(a.totals + e);
                if (!sched_only) s_base[e] = __ldcg(a.bases + (int64_t)b * E + e);
            }
        }
        __syncthreads();
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
        for (int p = threadIdx.x; p < np; p += blockDim.x) {
            const int e = tile_e[p];
            const int r = tile_r[p];
            const int sv = r < 0 ? -1 : s_eoff[e] + s_base[e] + cnt[(p / ppw) * E + e] + r;
            tile_s[p] = sv;
            a.slot[t0 * k + p] = sv;
        }
        if (kSplit && !sched_only) {
            // The CTA barrier orders every thread's slot stores before the
            // release store (release is cumulative): a data CTA that acquires
            // the flag sees the slots.
            __syncthreads();
            if (threadIdx.x == 0) st_release_u32(a.ready + b, 1u);
        }
        const int32_t epr = E / a.R;
        if (b == 0) {
            for (int e = threadIdx.x; e <= E; e += blockDim.x) {
                a.expert_offset[e] = s_eoff[e];
                if (e < E) a.expert_count[e] = s_tot[e];
            }
            for (int r = threadIdx.x; r < a.R; r += blockDim.x) {
                a.rank_offset[r] = s_eoff[r * epr];
                a.rank_count[r] = s_eoff[(r + 1) * epr] - s_eoff[r * epr];
            }
            if (threadIdx.x == 0) a.rank_offset[a.R] = s_eoff[E];
        }
        if (a.sched_cta ? sched_only : b == a.nb - 1) {
            for (int r = threadIdx.x; r <= a.R; r += blockDim.x) s_roff[r] = s_eoff[r * epr];
            __syncthreads();
            cta_build_schedule(s_roff, a.R, a.W, a.tiers, a.chunks, a.n_chunks, a.worker_begin, s_warp32, s_P,
                               whole_cta());
        }
        __syncthreads();
    } else if (threadIdx.x == 0) {
        atomicOr(a.err, kErrFusedWait);
        atomicExch(a.n_chunks, -1);
    }

    // G. dispatch the tile. When the rows to move are few, a combine launched
    // after this kernel may get ready now (it waits for this grid before it
    // touches memory); with more rows its waiting CTAs slowed this phase down.
    if (a.early_dependents) grid_launch_dependents();
    if (kSplit) return;  // the data CTAs move the rows
    const int64_t rows = (int64_t)a.T * k;
    if (a.ns > 0) {
        if (warp != 0) return;
        int i = 0;
        bool good = ok;
        for (; good && i < ntok; ++i) {
            const int s = i % a.ns;
            if (!mbar_wait_bounded(&bar[s], (uint32_t)((i / a.ns) & 1), kFusedMaxPolls)) {
                good = false;
                break;
            }
            const unsigned char *st = stages + (size_t)s * a.row_pad;
            if (lane < k) {
                const int sv = tile_s[i * k + lane];
                if (sv >= 0 && (int64_t)sv < rows) {
                    bulk_s2g(a.send + (int64_t)sv * row_bytes, st, (uint32_t)row_bytes);
                    a.meta[sv] = (int32_t)((t0 + i) * k + lane);
                }
                bulk_commit();
            }
            // refill the stage of row i - 1 once its stores have read it
            if (i >= 1 && i - 1 + a.ns < ntok) {
                if (lane < k) bulk_wait_read<1>();
                __syncwarp();
                if (lane == 0) {
                    const int sp = (i - 1) % a.ns;
                    mbar_arrive_expect_tx(&bar[sp], (uint32_t)row_bytes);
                    bulk_g2s(stages + (size_t)sp * a.row_pad, a.x + (t0 + i - 1 + a.ns) * row_bytes,
                             (uint32_t)row_bytes, &bar[sp]);
                }
            }
        }
        if (!good) {
            // Let every load already issued land before the CTA goes away.
            if (lane == 0) atomicOr(a.err, kErrFusedWait);
            const int issued = (i >= 1 ? i - 1 + a.ns : a.ns) < ntok ? (i >= 1 ? i - 1 + a.ns : a.ns) : ntok;
            for (int j = i; j < issued; ++j)
                mbar_wait_bounded(&bar[j % a.ns], (uint32_t)((j / a.ns) & 1), kFusedMaxPolls);
        }
        if (lane < k) bulk_wait<0>();
    } else if (ok) {
        // rows not suited to bulk copies: 16-byte vector copy by every warp
        const int hv = a.H / 8;
        const uint4 *x4 = reinterpret_cast<const uint4 *>(a.x);
        uint4 *s4 = reinterpret_cast<uint4 *>(a.send);
        for (int i = warp; i < ntok; i += kFusedWarps) {
            const int64_t t = t0 + i;
            for (int v = lane; v < hv; v += 32) {
                const uint4 val = ld_stream_v4(x4 + t * hv + v);
                for (int j = 0; j < k; ++j) {
                    const int sv = tile_s[i * k + j];
                    if (sv >= 0 && (int64_t)sv < rows) st_v4(s4 + (int64_t)sv * hv + v, val);
                }
            }
            if (lane < k) {
                const int sv = tile_s[i * k + lane];
                if (sv >= 0 && (int64_t)sv < rows) a.meta[sv] = (int32_t)(t * k + lane);
            }
        }
    }
}

}  // namespace

}  // namespace ep

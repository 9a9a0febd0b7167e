// fused.cu -- ep_dispatch_fused: route, layout and dispatch in one cooperative
// launch (the UBEP article's "Kernel Decomposition": metadata work and token
// movement in one kernel, with the SyncAll barriers between separate phases
// replaced by cores that poll global memory for the metadata they need).
//
// Each CTA owns a contiguous tile of tokens (tiles differ by at most one
// token, two CTAs per SM) and takes it through every step:
//   0. one thread starts TMA bulk loads of the tile's first x rows into
//      shared-memory stages (they land while the metadata is computed);
//   A. route: one warp per token (route_token.cuh), picks kept in shared memory;
//   B. rank: the tile's (token, expert) pairs are ranked per expert
//      (cta_rank_pairs) and the tile's per-expert counts published;
//   C. bounded grid barrier;
//   D. column scan: CTA q reads the counts of experts q, q + nb, ... over all
//      tiles in one batch and publishes each tile's base inside each of those
//      experts and their totals;
//   E. bounded grid barrier;
//      (up to 16384 pairs, D and E give way to C': every CTA reads all of
//      topk_idx, written in A, and counts the totals and its bases itself);
//   F. each CTA reads its tile's bases and the totals, scans the totals into
//      expert offsets and writes its slots; CTA 0 writes counts and offsets.
//      The chunk schedule is built by one extra CTA that holds no tile (it
//      joins both barriers, skips steps 0, A, B, D and G, and so overlaps the
//      schedule with the other CTAs' row copies); with a single tile CTA there
//      is no extra CTA, that CTA builds it, and the barriers reduce to
//      __syncthreads;
//   G. dispatch of the CTA's own tile from the prefetched stages: lanes j < k
//      bulk-store each row to its k send rows. When the send buffer is small
//      (<= 16 MB) every CTA signals programmatic dependents here, so that a
//      combine launched after it can start its prologue early.
// Up to 160 tokens the split form of the same kernel is used instead (the
// article's metadata/data decomposition): the tile CTAs (up to 8 tokens each,
// one per routing warp) stop after F, releasing a per-tile ready flag once
// their slots are written, and separate data CTAs -- as many as still fit on
// the GPU, one per send row when there are enough, else one per token --
// fetch their x row at once, acquire-poll the owning tile's flag (bounded)
// and bulk-store the rows. Up to 8 tokens the metadata is then one CTA with no
// grid barrier, and the rows leave from many SMs instead of one (measured per
// layer: T = 8 21.6 -> 19.5 us, T = 16 22.7 -> 21.0, T = 96 25.1 -> 23.0, T = 160
// 28.6 -> 27.3, T = 1 -0.5, T = 64 -0.3; at T = 192 and 256 within +-0.2 us, at
// T = 512 +4 us, so the split form stops at T = 160).
// The barrier words and ready flags are zeroed by a one-CTA kernel launched
// just before, of which the fused kernel is a programmatic dependent.
// Every result equals what ep_route, ep_layout and ep_dispatch write.
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

static __device__ int32_t g_fused_error;

struct FusedPlan {
    int nb = 0;       // CTAs (tiles)
    int n_data = 0;   // split form: data CTAs (0: the tile CTAs move their own rows)
    int unit_rows = 0;  // split form: rows per data unit (1 or k)
    int tb = 0;       // tokens in the largest tile
    int ns = 0;       // x-row stages per CTA (bulk path), 0 = vector copy
    int row_pad = 0;  // bytes per stage
    size_t smem = 0;
    int sched_cta = 0;  // 1: one more CTA, without a tile, builds the chunk schedule
};

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
    // the rows in units of unit_rows rows of one token (1, or k = the whole
    // token); ready[q] is set (release) once tile q's slots are written.
    int32_t n_data, unit_rows;
    unsigned *ready;
    // 1: after barrier C every CTA reads all of topk_idx and counts, in shared
    // memory, every expert's pairs (the totals) and those of the tokens before
    // its tile (its bases); steps D and E are skipped.
    int32_t hist;
};

// The rows of one token (unit_rows of them from top-k position jj0), moved by
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
        const int sv = a.slot[t * a.k + j];
        if (sv >= 0 && (int64_t)sv < rows) {
            bulk_s2g(a.send + (int64_t)sv * row_bytes, stage, (uint32_t)row_bytes);
            a.meta[sv] = (int32_t)(t * a.k + j);
        }
        bulk_commit();
    }
    return true;
}

// Zeroes the fused kernel's barrier words and ready flags. The fused kernel,
// launched right after it as its programmatic dependent, loads x rows, routes
// and ranks meanwhile, and waits for this grid only before it touches them
// (a memset node in its place cost 1.5-2 us per call at small T).
__global__ void __launch_bounds__(256) fused_zero_kernel(unsigned *p, int n) {
    grid_launch_dependents();
    for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0u;
}

// kSolo: the split form with a single tile CTA (up to 8 tokens), compiled
// without the grid barriers and the multi-CTA count steps it never runs (at
// these sizes the kernel's time follows its code size: it is fetched from HBM
// after the cache flush).
template <int VPL, bool kSplit, bool kSolo>
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
    const bool sched_only = !kSolo && a.sched_cta && b == a.nb;
    const unsigned arrivals = kSolo ? 1u : (unsigned)(a.nb + a.sched_cta);
    const bool hist = !kSolo && a.hist;
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
        const int64_t n_units = a.unit_rows == k ? (int64_t)a.T : (int64_t)a.T * k;
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
            const int64_t t = a.unit_rows == k ? u : u / k;
            const int jj0 = a.unit_rows == k ? 0 : (int)(u % k);
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
    const int ppw = np > 0 ? (np + kFusedWarps - 1) / kFusedWarps : 1;
    bool ok;
    if (hist) {
        // The others need only this tile's picks (in topk_idx since A): arrive
        // first, rank while they arrive (the counts stay in shared memory).
        grid_dependency_wait();
        grid_arrive(&a.sync[0]);
        if (!sched_only) cta_rank_pairs(tile_e, np, ppw, E, cnt, tile_r, s_col, 1);
        ok = grid_wait(&a.sync[0], arrivals);
    } else {
        // (a single CTA keeps its counts in shared memory: they are the totals)
        if (!sched_only)
            cta_rank_pairs(tile_e, np, ppw, E, cnt, tile_r, arrivals == 1 ? s_tot : a.counts + (int64_t)b * E, 1);
        grid_dependency_wait();
        ok = arrivals > 1 ? grid_barrier(&a.sync[0], arrivals) : (__syncthreads(), true);
    }
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
        if (!kSolo && a.sched_cta ? sched_only : b == a.nb - 1) {
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

using FusedKernel = void (*)(FusedArgs);

template <bool kSplit, bool kSolo>
FusedKernel pick_kernel_t(int32_t E) {
    const int vpl = (E + 31) / 32;
    if (vpl <= 1) return dispatch_fused_kernel<1, kSplit, kSolo>;
    if (vpl <= 2) return dispatch_fused_kernel<2, kSplit, kSolo>;
    if (vpl <= 4) return dispatch_fused_kernel<4, kSplit, kSolo>;
    if (vpl <= 8) return dispatch_fused_kernel<8, kSplit, kSolo>;
    if (vpl <= 16) return dispatch_fused_kernel<16, kSplit, kSolo>;
    return dispatch_fused_kernel<32, kSplit, kSolo>;
}

// form 0: single-role, 1: split, 2: split with a single tile CTA
FusedKernel pick_kernel(int32_t E, int form) {
    return form == 2 ? pick_kernel_t<true, true>(E) : form == 1 ? pick_kernel_t<true, false>(E)
                                                                : pick_kernel_t<false, false>(E);
}

// Lets a kernel use up to kFusedSmemLimit of dynamic shared memory (once per
// device and kernel); false if the device refuses.
bool allow_fused_smem(FusedKernel kern, int dev, int32_t E, int form) {
    static std::atomic<bool> attr_set[kMaxDevices_][3][6];  // zero-initialised: false
    const int vpl = (E + 31) / 32;
    const int vi = vpl <= 1 ? 0 : vpl <= 2 ? 1 : vpl <= 4 ? 2 : vpl <= 8 ? 3 : vpl <= 16 ? 4 : 5;
    if (attr_set[dev][form][vi]) return true;
    if (cudaFuncSetAttribute(reinterpret_cast<const void *>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFusedSmemLimit) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    attr_set[dev][form][vi] = true;
    return true;
}

// The split form (kernel decomposition with separate data CTAs): tiles of up
// to 8 tokens (one per routing warp), the schedule CTA when there are several
// tiles, and as many data CTAs as still fit on the GPU, each moving units of
// one row (when every row can have its own CTA) or of a whole token. false if
// the shape does not suit it (then the caller uses the other forms).
bool plan_split(const ep_config &c, FusedPlan *p) {
    if (c.T <= 0 || c.T > kSplitMaxT) return false;
    const int32_t row_bytes = c.H * 2;
    if (row_bytes < 1024 || row_bytes > 48 * 1024) return false;  // rows move as bulk copies
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices_) return false;
    const int nb = (int)((c.T + kFusedWarps - 1) / kFusedWarps);
    const int form = nb == 1 ? 2 : 1;
    const FusedKernel kern = pick_kernel(c.E, form);
    if (!allow_fused_smem(kern, dev, c.E, form)) return false;
    if (nb > kMaxFusedCTAs) return false;
    const int tb = (int)((c.T + nb - 1) / nb);
    const int sched = nb > 1 ? 1 : 0;
    const int row_pad = (int)align128((size_t)row_bytes);
    const SmemLayout L = smem_layout(1, row_pad, tb, c.k, c.E, c.R, c.n_groups > 1);
    if (L.bytes > kFusedSmemLimit) return false;
    const int64_t cap = (int64_t)sm_count(dev) * max_blocks_per_sm(reinterpret_cast<const void *>(kern),
                                                                     kFusedThreads, L.bytes);
    const int64_t room = cap - nb - sched;
    if (room < 1) return false;
    const int64_t pairs = (int64_t)c.T * c.k;
    const int unit_rows = pairs <= room ? 1 : c.k;
    const int64_t n_units = unit_rows == 1 ? pairs : c.T;
    p->nb = nb;
    p->sched_cta = sched;
    p->tb = tb;
    p->ns = 1;
    p->row_pad = row_pad;
    p->smem = L.bytes;
    p->n_data = (int)(n_units < room ? n_units : room);
    p->unit_rows = unit_rows;
    return true;
}

// Choose the tiling: as many CTAs as fit on the GPU at once (two per SM when
// shared memory allows, at most 1024 and at most T), tiles within one token
// of each other in size. false if the fused kernel
// cannot run this shape (then the caller runs the three separate steps).
bool plan_fused(const ep_config &c, FusedPlan *p) {
    if (c.T <= 0 || c.T > kFusedMaxT) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices_) return false;
    const FusedKernel kern = pick_kernel(c.E, 0);
    if (!allow_fused_smem(kern, dev, c.E, 0)) return false;
    const int32_t row_bytes = c.H * 2;
    const bool bulk = c.k % 4 == 0 && row_bytes >= 1024 && row_bytes <= 48 * 1024;
    const int sms = sm_count(dev);
    // Try 2, then 1 CTA per SM (more CTAs = smaller tiles = shorter metadata phases).
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        int nb = sms * per_sm - 1;  // one resident slot kept for the schedule CTA
        if (nb > kMaxFusedCTAs) nb = kMaxFusedCTAs;
        if (nb > c.T) nb = c.T;
        if (nb < 1) nb = 1;
        const int tb = (int)((c.T + nb - 1) / nb);  // largest tile
        // Routing needs a warp per token to keep its latency hidden; when a
        // warp would route more than one token the separate route kernel
        // (64 warps per SM) is faster, so the fused kernel is not used. (A
        // variant that stopped after the slots, with up to 1024 small CTAs
        // and the dispatch kernel after it, measured 6 us slower than the
        // separate kernels at T = 4096 and equal at T = 16384.)
        if (tb > kFusedWarps || (int64_t)tb * c.k > kMaxTilePairs) return false;
        const int row_pad = (int)align128((size_t)row_bytes);
        const SmemLayout base = smem_layout(0, row_pad, tb, c.k, c.E, c.R, c.n_groups > 1);
        int ns = 0;
        if (bulk) {
            const size_t budget = kFusedSmemLimit / per_sm - base.bytes - 2048;
            ns = (int)(budget / row_pad);
            if (ns > kMaxFusedStages) ns = kMaxFusedStages;
            if (ns > tb) ns = tb;
            if (ns < 1) continue;
        }
        const SmemLayout L = smem_layout(ns, row_pad, tb, c.k, c.E, c.R, c.n_groups > 1);
        if (L.bytes > kFusedSmemLimit) continue;
        const int occ = max_blocks_per_sm(reinterpret_cast<const void *>(kern), kFusedThreads, L.bytes);
        const int sched = nb > 1 ? 1 : 0;
        if (nb + sched > sms * occ) continue;
        p->nb = nb;
        p->sched_cta = sched;
        p->tb = tb;
        p->ns = ns;
        p->row_pad = row_pad;
        p->smem = L.bytes;
        return true;
    }
    return false;
}

}  // namespace

cudaError_t fused_error_word(int32_t **addr) {
    static std::atomic<int32_t *> cached[kMaxDevices_];  // zero-initialised: null
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices_) return cudaErrorInvalidDevice;
    if (!cached[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fused_error);
        if (e != cudaSuccess) return e;
        cached[dev] = static_cast<int32_t *>(p);
    }
    *addr = cached[dev];
    return cudaSuccess;
}

size_t fused_tables_bytes(const ep_config &c);

// The dispatch counter sits after both the layout's workspace and the fused tables.
size_t fused_counter_offset(const ep_config &c) {
    const size_t lw = layout_workspace(c).bytes, ft = fused_tables_bytes(c);
    return ((lw > ft ? lw : ft) + 255) & ~(size_t)255;
}

// Fused tables (counts, bases, totals, barrier words), then the dispatch counter.
size_t fused_tables_bytes(const ep_config &c) {
    const int64_t nb = c.T < kMaxFusedCTAs ? c.T : kMaxFusedCTAs;
    const size_t tables = 2 * sizeof(int32_t) * (size_t)nb * (size_t)c.E;
    // then the two barrier words and one ready flag per tile (split form)
    return ((tables + sizeof(int32_t) * (size_t)c.E + 255) & ~(size_t)255) +
           ((sizeof(unsigned) * (2 + (size_t)kMaxFusedCTAs) + 255) & ~(size_t)255);
}

size_t fused_workspace_bytes(const ep_config &c) {
    return c.T == 0 ? 0 : fused_counter_offset(c) + 256;
}

int fused_call_kernels(const ep_config &c) {
    FusedPlan p;
    const bool split = plan_split(c, &p);
    if (!split && !plan_fused(c, &p)) return 2 + layout_kernel_count(c);  // route, layout, dispatch
    return split || p.nb + p.sched_cta > 1 ? 2 : 1;  // (the zeroing kernel,) the fused kernel
}

cudaError_t launch_dispatch_fused(const ep_config &c, int32_t W, const float *logits, const ep_bf16 *x,
                                  int32_t *topk_idx, float *topk_w, int32_t *expert_count, int32_t *expert_offset,
                                  int32_t *rank_count, int32_t *rank_offset, int32_t *slot, ep_chunk *chunks,
                                  int32_t *n_chunks, int32_t *worker_begin, ep_bf16 *send, int32_t *meta,
                                  void *workspace, cudaStream_t s) {
    FusedPlan p;
    const bool split = plan_split(c, &p);
    if (!split && !plan_fused(c, &p)) {
        // Three kernels; the route kernel zeroes the single-kernel layout's
        // count table (and the dispatch counter unless the layout does, below),
        // so no memset sits between the kernels.
        char *ws = static_cast<char *>(workspace);
        unsigned *table = reinterpret_cast<unsigned *>(ws + layout_workspace(c).block_counts_off);
        unsigned *ctr = reinterpret_cast<unsigned *>(ws + fused_counter_offset(c));
        // When the bulk dispatch follows the single-kernel layout, an extra CTA of
        // the dispatch builds the chunk schedule, so the layout does not hold the
        // dispatch back for it; the route kernel zeroes n_chunks, which the
        // layout sets to -1 if it fails.
        const bool defer = dispatch_uses_bulk(c, slot);
        // The single-kernel layout zeroes the dispatch counter itself. While
        // the route kernel runs in one wave the layout is its programmatic
        // dependent (the dispatch, the layout's dependent, may then start
        // while the route kernel still runs). Measured: prefill -1.4 us;
        // with several waves of route CTAs the early grids took resources from
        // the later ones (T = 32768: +4.6 us), so there the layout waits.
        const bool single = layout_kernel_count(c) == 1;
        const bool after_route = single && route_one_wave(c);
        const int table_words = single ? (int)layout_workspace(c).table_words : 0;
        cudaError_t e = launch_route(c, logits, topk_idx, topk_w, s, table, table_words, single ? nullptr : ctr,
                                     single ? 0 : 1, defer ? n_chunks : nullptr);
        if (e != cudaSuccess) return e;
        bool deferred = false;
        e = launch_layout(c, W, topk_idx, expert_count, expert_offset, rank_count, rank_offset, slot, chunks,
                          n_chunks, worker_begin, workspace, s, true, defer, &deferred, after_route,
                          single ? ctr : nullptr);
        if (e != cudaSuccess) return e;
        const ScheduleTask st{rank_offset, chunks, n_chunks, worker_begin, c.R, W, hop_tiers(c)};
        return launch_dispatch(c, x, slot, send, meta, s, ctr, true, true, deferred ? &st : nullptr);
    }
    FusedArgs a;
    a.logits = logits;
    a.x = reinterpret_cast<const char *>(x);
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.expert_count = expert_count;
    a.expert_offset = expert_offset;
    a.rank_count = rank_count;
    a.rank_offset = rank_offset;
    a.slot = slot;
    a.chunks = chunks;
    a.n_chunks = n_chunks;
    a.worker_begin = worker_begin;
    a.send = reinterpret_cast<char *>(send);
    a.meta = meta;
    char *ws = static_cast<char *>(workspace);
    const size_t table = sizeof(int32_t) * (size_t)p.nb * (size_t)c.E;
    a.counts = reinterpret_cast<int32_t *>(ws);
    a.bases = reinterpret_cast<int32_t *>(ws + table);
    a.totals = reinterpret_cast<int32_t *>(ws + 2 * table);
    const size_t sync_off = (2 * table + sizeof(int32_t) * (size_t)c.E + 255) & ~(size_t)255;
    a.sync = reinterpret_cast<unsigned *>(ws + sync_off);
    cudaError_t e = fused_error_word(&a.err);
    if (e != cudaSuccess) return e;
    a.T = c.T;
    a.H = c.H;
    a.E = c.E;
    a.R = c.R;
    a.k = c.k;
    a.n_groups = c.n_groups;
    a.topk_groups = c.topk_groups;
    a.renormalize = c.renormalize;
    a.W = W;
    a.tiers = hop_tiers(c);
    a.nb = p.nb;
    a.sched_cta = p.sched_cta;
    a.tb = p.tb;
    a.ns = p.ns;
    a.row_pad = p.row_pad;
    a.n_data = p.n_data;
    a.unit_rows = p.unit_rows;
    a.ready = a.sync + 2;
    // Up to kHistMaxPairs pairs every CTA reads all of topk_idx after the first
    // barrier instead of the column scan and the second barrier (measured per
    // layer: T = 64 -1.6 us, T = 160 -2.1, decode -2.3, T = 512 -2.1, T = 1024
    // -1.6, T = 1760 +-0.3).
    a.hist = p.nb + p.sched_cta > 1 && (int64_t)c.T * c.k <= kHistMaxPairs ? 1 : 0;
    // measured: T = 1..64 (<= 7.3 MB of send rows) gain 1-2 us, T = 256 even, T = 512 (59 MB) loses 1.8 us
    a.early_dependents = (int64_t)c.T * c.k * c.H * 2 <= (int64_t)16 << 20 ? 1 : 0;
    // The barrier words and (split form) the tiles' ready flags are zeroed by a
    // one-CTA kernel in front of the fused one; a single CTA of the single-role
    // form uses neither.
    const int n_zero = split ? 2 + p.nb : (p.nb + p.sched_cta > 1 ? 2 : 0);
    if (n_zero > 0) {
        fused_zero_kernel<<<1, 256, 0, s>>>(a.sync, n_zero);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const FusedKernel kern = pick_kernel(c.E, split ? (p.nb == 1 && p.sched_cta == 0 ? 2 : 1) : 0);
    const dim3 grid((unsigned)(p.nb + p.sched_cta + p.n_data));
    // Set when a device refused the cooperative launch with the dependent-launch
    // attribute; the plain cooperative launch is then used (the same results).
    static std::atomic<bool> no_dependent_coop[kMaxDevices_];  // zero-initialised: false
    int dev = 0;
    if (n_zero > 0 && current_device(&dev) == cudaSuccess && !no_dependent_coop[dev]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kFusedThreads);
        cfg.dynamicSmemBytes = p.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kern, a);
        if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return e;
        cudaGetLastError();  // the launch was refused before anything was enqueued
        no_dependent_coop[dev] = true;
    }
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), grid, dim3(kFusedThreads), args, p.smem,
                                       s);
}

}  // namespace ep

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
//      Up to 16384 pairs (every split-form launch, and the single-role form
//      at small k) D and E give way to C': the CTAs arrive at barrier C as
//      soon as A has stored their picks in topk_idx, rank while the others
//      arrive, and then every CTA reads all of topk_idx and counts the totals
//      and its bases itself, in shared memory;
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
// article's metadata/data decomposition): the tile CTAs (up to 4 tokens each
// up to T = 64, else up to 8, one per routing warp) stop after F, releasing
// a per-tile ready flag once their slots are written, and separate data CTAs
// -- as many as still fit on the GPU, one per send row when there are enough,
// else one per 2, 4, ... rows of a token -- fetch their x row at once, acquire-poll the owning
// tile's flag (bounded) and bulk-store the rows; the schedule CTA is there
// even for a single tile. The rows leave from many SMs instead of a few
// (measured per layer against the single-role form: T = 8 21.6 -> 19.5 us,
// T = 16 22.7 -> 21.0, T = 96 25.1 -> 23.0, T = 160 28.6 -> 27.3, T = 1 -0.5,
// T = 64 -0.3; at T = 192 and 256 within +-0.2 us, at T = 512 +4 us, so the
// split form stops at T = 160).
// The barrier words and ready flags are zeroed by a one-CTA kernel launched
// just before, of which the fused kernel is a programmatic dependent.
// Every result equals what ep_route, ep_layout and ep_dispatch write.
#include "fused_kernel.cuh"

namespace ep {
namespace {

static __device__ int32_t g_fused_error;

struct FusedPlan {
    int nb = 0;       // CTAs (tiles)
    int n_data = 0;   // split form: data CTAs (0: the tile CTAs move their own rows)
    int unit_rows = 0;  // split form: rows per data unit (1, 2, 4, ... or k)
    int tb = 0;       // tokens in the largest tile
    int ns = 0;       // x-row stages per CTA (bulk path), 0 = vector copy
    int row_pad = 0;  // bytes per stage
    size_t smem = 0;
    int sched_cta = 0;  // 1: one more CTA, without a tile, builds the chunk schedule
};

// Zeroes the fused kernel's barrier words and ready flags. The fused kernel,
// launched right after it as its programmatic dependent, loads x rows, routes
// and ranks meanwhile, and waits for this grid only before it touches them
// (a memset node in its place cost 1.5-2 us per call at small T).
__global__ void __launch_bounds__(256) fused_zero_kernel(unsigned *p, int n) {
    grid_launch_dependents();
    for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0u;
}

using FusedKernel = void (*)(FusedArgs);

template <bool kSplit>
FusedKernel pick_kernel_t(int32_t E) {
    const int vpl = (E + 31) / 32;
    if (vpl <= 1) return dispatch_fused_kernel<1, kSplit>;
    if (vpl <= 2) return dispatch_fused_kernel<2, kSplit>;
    if (vpl <= 4) return dispatch_fused_kernel<4, kSplit>;
    if (vpl <= 8) return dispatch_fused_kernel<8, kSplit>;
    if (vpl <= 16) return dispatch_fused_kernel<16, kSplit>;
    return dispatch_fused_kernel<32, kSplit>;
}

// form 0: single-role, 1: split
FusedKernel pick_kernel(int32_t E, int form) {
    return form == 1 ? pick_kernel_t<true>(E) : pick_kernel_t<false>(E);
}

// Lets a kernel use up to kFusedSmemLimit of dynamic shared memory (once per
// device and kernel); false if the device refuses.
bool allow_fused_smem(FusedKernel kern, int dev, int32_t E, int form) {
    static std::atomic<bool> attr_set[kMaxDevices_][2][6];  // zero-initialised: false
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
// to 4 or 8 tokens, the schedule CTA, and as many data CTAs as still fit on
// the GPU, each moving units of a few of a token's rows. false if the shape
// does not suit it (then the caller uses the other forms).
bool plan_split(const ep_config &c, FusedPlan *p) {
    if (c.T <= 0 || c.T > kSplitMaxT) return false;
    const int32_t row_bytes = c.H * 2;
    if (row_bytes < 1024 || row_bytes > 48 * 1024) return false;  // rows move as bulk copies
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices_) return false;
    // Tiles of 4 tokens up to T = 64, else 8 (one per routing warp). Measured
    // per layer against 8 everywhere, on two boxes: T = 8 (two tiles and the
    // schedule CTA instead of one tile CTA that also built the schedule) -0.5
    // and -1.5 us, T = 64 -1.5 and +-0.1, T = 16 +-0.1; at T = 96 and 160
    // tiles of 4 were even or +0.3.
    const int tile = c.T <= 64 ? 4 : kFusedWarps;
    const int nb = (int)((c.T + tile - 1) / tile);
    const FusedKernel kern = pick_kernel(c.E, 1);
    if (!allow_fused_smem(kern, dev, c.E, 1)) return false;
    if (nb > kMaxFusedCTAs) return false;
    const int tb = (int)((c.T + nb - 1) / nb);
    // The schedule CTA even for a single tile: it builds the chunk schedule
    // while the tile CTA writes its slots, at the price of a grid barrier
    // (measured against one tile CTA doing both, compiled as an instance of its
    // own without the barrier: T = 1 +-0.05 and -0.25 us, T = 2 -0.1, T = 4 -0.8).
    const int sched = 1;
    const int row_pad = (int)align128((size_t)row_bytes);
    const SmemLayout L = smem_layout(1, row_pad, tb, c.k, c.E, c.R, c.n_groups > 1);
    if (L.bytes > kFusedSmemLimit) return false;
    const int64_t cap = (int64_t)sm_count(dev) * max_blocks_per_sm(reinterpret_cast<const void *>(kern),
                                                                     kFusedThreads, L.bytes);
    const int64_t room = cap - nb - sched;
    if (room < 1) return false;
    // A data CTA per unit of unit_rows of a token's k send rows: the fewest
    // rows (1, 2, 4, ... or all k) that give every unit a CTA of its own
    // (measured against whole tokens once rows outnumber the CTAs: T = 40 -0.9
    // and -1.4 us per layer, T = 64, 96 and 128 within +-0.1).
    int unit_rows = 1;
    while (unit_rows < c.k && (int64_t)c.T * ((c.k + unit_rows - 1) / unit_rows) > room) unit_rows *= 2;
    if (unit_rows > c.k) unit_rows = c.k;
    const int64_t n_units = (int64_t)c.T * ((c.k + unit_rows - 1) / unit_rows);
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
        // Up to 1024 tokens, at most 128 tiles (two to eight tokens each in
        // place of one or two: decode -0.8 us per layer, T = 192 -0.5, T = 512
        // -0.9, T = 1024 -1.9; above 1024 the 8-token tiles that the same count
        // would need measured 5-9 us slower than the smaller ones).
        if (c.T <= 1024 && nb > kFusedTileCap) nb = kFusedTileCap;
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
    a.hist = p.nb + p.sched_cta > 1 && (split || (int64_t)c.T * c.k <= kHistMaxPairs) ? 1 : 0;
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
    const FusedKernel kern = pick_kernel(c.E, split ? 1 : 0);
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

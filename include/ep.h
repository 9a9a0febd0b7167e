/*
 * ep.h -- C ABI of the GB300 (sm_103a) MoE expert-parallel hot path:
 * router softmax + top-k, dispatch layout, dispatch scatter, combine.
 *
 * The operations are the ones the UBEP article ("NJU x Huawei UBEP:
 * Reengineering MoE Expert Parallelism", kad8.com) names for an expert-parallel
 * communication library: a token goes to the device of each expert chosen for
 * it, and the experts' outputs return to it in the Combine step (opening
 * section); the dispatch needs token counts, offsets from prefix sums and a
 * reordering of tokens ("Three Bottlenecks" / BSP Serialization, "Kernel
 * Decomposition"); and per-worker traffic is balanced across hop-latency
 * classes ("Hierarchical Token-Level Scheduling" / Latency Homogenization).
 * Here the R expert-parallel ranks are R contiguous partitions of one send
 * buffer on one GPU: there is no peer traffic and no collective.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA memory)
 *    on the current device, row-major and densely packed. The caller allocates
 *    and owns every buffer; the library allocates nothing and keeps no state
 *    between calls besides cached device attributes (and the fixed scratch
 *    array of ep_layout_static, below).
 *  - Work is enqueued on `stream` (0 = legacy default stream) and is
 *    asynchronous: results are ready when the stream reaches that point.
 *    ep_combine, and the dispatch kernel inside ep_dispatch_fused, are
 *    launched as programmatic dependents of the kernel before them on the
 *    stream: their CTAs may become resident early, but each waits for that
 *    kernel to complete (griddepcontrol.wait) before it touches memory. Stream
 *    order is therefore kept whenever that kernel itself ends after the work
 *    queued before it -- any kernel launched without programmatic stream
 *    serialization, or one launched with it that waits on its own
 *    predecessor before it ends.
 *  - bf16 tensors are passed as `ep_bf16` (the 16-bit pattern of a bfloat16).
 *    x, send, y and out must be 16-byte aligned; H must be a multiple of 8 so
 *    that every row is a whole number of 16-byte vectors.
 *  - Arguments are checked on the host before anything is launched: a bad
 *    argument returns EP_ERR_INVALID_ARG / EP_ERR_UNSUPPORTED /
 *    EP_ERR_CAPACITY with nothing enqueued. EP_ERR_CUDA reports a launch error
 *    (cudaGetLastError after the launch). No C++ exception crosses the ABI.
 *  - T = 0 is valid: route, dispatch and combine enqueue nothing; layout still
 *    writes its (all-zero) counts, offsets and schedule.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ep_status {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1, /* null pointer, inconsistent sizes, misaligned buffer      */
    EP_ERR_UNSUPPORTED = 2, /* outside the built kernels: H % 8 != 0, k > 32, E > 1024,
                               n_groups > 32                                            */
    EP_ERR_CUDA = 3,        /* a CUDA launch or attribute query failed                  */
    EP_ERR_CAPACITY = 4     /* chunk table or workspace smaller than required           */
} ep_status;

/* One layer's shape. */
typedef struct ep_config {
    int32_t T;              /* tokens on this GPU (>= 0); T * k <= INT32_MAX              */
    int32_t H;              /* hidden size: bf16 elements per token row (> 0)             */
    int32_t E;              /* experts (1 .. 1024)                                        */
    int32_t R;              /* virtual expert-parallel ranks; E % R == 0; rank r owns
                               experts [r E/R, (r+1) E/R)                                 */
    int32_t k;              /* experts per token (1 .. min(E, 32))                        */
    int32_t n_groups;       /* expert groups for group-limited routing; 1 = no limit;
                               E % n_groups == 0, n_groups <= 32                          */
    int32_t topk_groups;    /* groups kept per token (1 .. n_groups);
                               topk_groups * (E / n_groups) >= k                           */
    int32_t renormalize;    /* 1: top-k weights renormalised to sum to 1; 0: raw softmax  */
    int32_t ranks_per_node; /* ranks sharing one node: defines the hop classes (>= 1)     */
    int32_t self_rank;      /* the sending rank whose view the schedule models [0, R)     */
    int32_t num_workers;    /* W, workers of the chunk schedule; 0 = the device SM count  */
    int32_t ranks_per_pod;  /* ranks sharing one pod (a second switch tier): 0 = no pod
                               tier (hop classes 0 and 1); else a multiple of
                               ranks_per_node, and ranks in another pod form class 2   */
} ep_config;

/* One record of the chunk schedule: rows [row_begin, row_begin + row_count)
 * of the send buffer, all bound for dst_rank, handled by `worker`.
 * hop_class 0 = a rank on the sender's node, 1 = a rank on another node (of
 * the same pod, when pods are given), 2 = a rank in another pod. */
typedef struct ep_chunk {
    int32_t worker;
    int32_t hop_class;
    int32_t dst_rank;
    int32_t row_begin;
    int32_t row_count;
} ep_chunk;

typedef uint16_t ep_bf16;

/* Human-readable name of a status code (static string, never NULL). */
const char *ep_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int ep_version(void);

/* Device-side error flags of the current device, read and cleared
 * (synchronous: waits for work already enqueued on the device). Kernels never
 * trap; a wait that runs out sets a flag here instead and the kernel returns.
 *   bit 0 (1): an ep_dispatch CTA gave up waiting for a bulk copy to land; its
 *              remaining rows were not written.
 *   bit 1 (2): an ep_dispatch_fused CTA gave up waiting (grid barrier or bulk
 *              copy); its slots or rows were not written.
 *   bit 2 (4): an ep_dispatch_expert_sp CTA gave up waiting (a row that never
 *              arrived, or a bulk copy); its rows were not all written.
 *   bit 3 (8): an ep_dispatch_scheduled CTA gave up waiting on a bulk copy,
 *              or its chunk table named rows outside the send buffer.
 * (ep_layout reports its own bounded wait through *n_chunks = -1.) */
ep_status ep_device_error(int32_t *flags);

/* Diagnostics: checks that the library's device-side waits are bounded and
 * that a failure cannot be hidden. Launches two CTAs into a grid barrier (the
 * kind ep_dispatch_fused uses) that expects three arrivals, so the wait cannot
 * complete in time; each CTA must give up after max_polls polls (> 0) and
 * count itself in *gave_up (device int32, zeroed first). A third CTA makes the
 * last arrival only after one of them has given up; it must see the failure
 * as well, else *gave_up is set to -1. A fourth CTA waits, as
 * ep_dispatch_fused's data CTAs do, on a ready flag that nothing sets, and
 * must give up after max_polls polls and count itself. A fifth and a sixth CTA
 * exchange a two-row count table the way ep_layout's CTAs do: the fifth
 * publishes its row and polls for the other, which the sixth publishes only
 * after the fifth has given up; both must count themselves (the sixth learns
 * from its publish that it came too late; in ep_layout that keeps a late CTA
 * from going on and a chunk count from overwriting *n_chunks = -1), else
 * *gave_up is set to -1. Expected result: 5. The kernels return normally;
 * nothing faults or hangs. */
ep_status ep_check_bounded_wait(int32_t max_polls, int32_t *gave_up, cudaStream_t stream);

/* Bytes of device scratch that ep_layout needs for `cfg` (it depends on T and
 * E only). The workspace needs no initialisation and may be reused across
 * calls on the same stream. */
ep_status ep_layout_workspace_size(const ep_config *cfg, size_t *bytes);

/* Number of ep_chunk records ep_layout may write for `cfg`: C W + R, with C
 * the number of hop classes (2, or 3 when ranks_per_pod > 0) and W =
 * num_workers, or the current device's SM count when num_workers = 0. */
ep_status ep_schedule_capacity(const ep_config *cfg, int32_t *capacity);

/* Number of kernels one ep_route + ep_layout + ep_dispatch + ep_combine pass
 * enqueues for `cfg` on the current device (the layout is one cooperative
 * kernel when all its CTAs fit on the GPU at once, else three), for callers
 * that size CUDA graphs or count launches. */
ep_status ep_step_kernel_count(const ep_config *cfg, int32_t *kernels);

/* The same for one ep_dispatch_fused + ep_combine pass (2 when the fused
 * kernel runs, else 4 or 6). */
ep_status ep_fused_step_kernel_count(const ep_config *cfg, int32_t *kernels);

/*
 * ep_route -- router softmax and top-k for every token.
 *
 * Defines (the pages give no router, only that a token travels to the device
 * of the expert chosen for it, UBEP article, opening section; this is the
 * plainest gate that chooses experts per token):
 *   p[t, e]       = softmax over all E experts of logits[t, :]
 *   topk_idx[t,:] = the k experts with the largest logits, in descending order;
 *                   equal logits go to the lower expert index. With
 *                   n_groups > 1 only experts of the topk_groups groups with
 *                   the largest per-group maximum logit are eligible (ties to
 *                   the lower group index).
 *   topk_w[t, j]  = p[t, idx_j] / sum_i p[t, idx_i] if renormalize, else p[t, idx_j]
 *
 * logits   : const float [T, E]  gate logits; must be finite
 * topk_idx : int32 [T, k]        output
 * topk_w   : float [T, k]        output (fp32; within a few ulp of exact)
 */
ep_status ep_route(const ep_config *cfg, const float *logits, int32_t *topk_idx, float *topk_w,
                   cudaStream_t stream);

/*
 * ep_layout -- counts, offsets, the stable slot of every (token, expert)
 * pair and the per-destination chunk schedule.
 *
 * Defines (token counting, prefix sums, offsets and reordering of the BSP
 * pipeline, done here as one metadata pass):
 *   expert_count[e]  = #{(t, j) : topk_idx[t, j] = e}
 *   expert_offset[e] = sum_{e' < e} expert_count[e'];     expert_offset[E] = T k
 *   rank_offset[r]   = expert_offset[r E / R];            rank_offset[R] = T k
 *   rank_count[r]    = rank_offset[r + 1] - rank_offset[r]
 *   slot[t, j]       = expert_offset[e] + #{t' < t : e in topk_idx[t', :]}, e = topk_idx[t, j]
 * i.e. send rows are ordered by (destination rank, expert, source token).
 *
 * Chunk schedule (Latency Homogenization; the same section extends it to
 * more switch tiers): hop_class(r) = 0 if rank r is on the node of self_rank
 * (r / ranks_per_node == self_rank / ranks_per_node); else 2 if
 * ranks_per_pod > 0 and r / ranks_per_pod != self_rank / ranks_per_pod;
 * else 1. For each class c, the class's rank segments concatenated in
 * ascending rank hold N_c rows; worker w takes positions
 * [floor(N_c w / W), floor(N_c (w + 1) / W)) of each class, cut at rank
 * boundaries into non-empty chunks. The table is ordered by worker, then
 * class descending (the farthest traffic first), then rank; worker_begin[w]
 * is the index of worker w's first chunk and worker_begin[W] = *n_chunks.
 *
 * topk_idx      : const int32 [T, k]; each row holds k distinct experts in
 *                 [0, E) (as ep_route writes). An id outside [0, E) gets
 *                 slot -1 and is not counted; a repeated id within one row
 *                 gives unspecified (but in-range) slots.
 * expert_count  : int32 [E]      output
 * expert_offset : int32 [E + 1]  output
 * rank_count    : int32 [R]      output
 * rank_offset   : int32 [R + 1]  output
 * slot          : int32 [T, k]   output
 * chunks        : ep_chunk [chunk_capacity] output; chunk_capacity >= C W + R
 *                 (ep_schedule_capacity), else EP_ERR_CAPACITY
 * n_chunks      : int32 [1]      output (device memory)
 * worker_begin  : int32 [W + 1]  output
 * workspace     : device scratch of >= ep_layout_workspace_size bytes,
 *                 256-byte aligned; else EP_ERR_CAPACITY / EP_ERR_INVALID_ARG
 *
 * When every layout CTA fits on the GPU at once, the layout is one
 * cooperative launch whose CTAs exchange their per-expert counts through a
 * [CTA][E] table in the workspace (zeroed by an enqueued memset when there is
 * more than one CTA): each CTA publishes its row with every entry marked
 * valid and polls the others' entries until they are, with no grid barrier.
 * That wait is bounded: a CTA that gives up marks the entries it still misses
 * as failed, sets *n_chunks = -1 and leaves its slots unwritten; every other
 * CTA, including the late owner of those entries, then fails too, so no chunk
 * count overwrites the -1 (this cannot happen under a cooperative launch,
 * which only starts when all CTAs are resident).
 * Larger T uses three ordinary kernels.
 */
ep_status ep_layout(const ep_config *cfg, const int32_t *topk_idx,
                    int32_t *expert_count, int32_t *expert_offset,
                    int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                    ep_chunk *chunks, int32_t chunk_capacity, int32_t *n_chunks,
                    int32_t *worker_begin, void *workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/*
 * ep_dispatch -- scatter each token row to the send-buffer rows of its k
 * slots (UBEP article, opening section: a token has to reach the device that
 * holds each expert chosen for it; here the send buffer is partitioned by
 * destination rank):
 *   send[slot[t, j], :] = x[t, :]        (bit copy)
 *   slot_meta[slot[t, j]] = t k + j      (source token and top-k position)
 *
 * x         : const bf16 [T, H]
 * slot      : const int32 [T, k]  as written by ep_layout; entries outside
 *             [0, T k) are skipped
 * send      : bf16 [T k, H]       output
 * slot_meta : int32 [T k]         output
 */
ep_status ep_dispatch(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send,
                      int32_t *slot_meta, cudaStream_t stream);

/*
 * ep_dispatch_fused -- ep_route, ep_layout and ep_dispatch in one call, with
 * identical outputs (every argument means what it means there).
 *
 * Follows the UBEP article's "Kernel Decomposition": instead of separate
 * phases joined by global barriers, one cooperative kernel gives every CTA a
 * tile of tokens to route, rank and dispatch; the CTAs exchange the per-expert
 * counts through global memory at bounded grid barriers (in the workspace; up
 * to 16384 (token, expert) pairs one barrier, after which every CTA counts
 * the totals and its bases from all of topk_idx)
 * and each CTA's x rows are fetched with bulk copies while that metadata is
 * being computed. Up to 160 tokens the rows are moved by separate data CTAs
 * instead, each waiting (bounded) on a ready flag that the tile holding its
 * token releases once its slots are written. The barrier words and flags are
 * zeroed by a one-CTA kernel launched just before the fused kernel, which is
 * its programmatic dependent. It pays off at small T (decode batches), where
 * the phases are latency-bound; above 1760 tokens (measured: there the
 * separate kernels are faster) the call runs the three separate steps instead (the route kernel zeroing the
 * layout's count table, the single-kernel layout -- launched as a
 * programmatic dependent of the route kernel when that one runs in a single
 * wave -- zeroing the dispatch's token counter, the dispatch taking tokens
 * dynamically and building the chunk schedule in one extra CTA while the
 * others copy rows), with the same results.
 *
 * workspace : >= ep_dispatch_fused_workspace_size bytes, 256-byte aligned.
 * A CTA that gives up a bounded wait sets ep_device_error bit 1 (2) and
 * *n_chunks = -1 (it cannot happen under the cooperative launch used).
 */
ep_status ep_dispatch_fused_workspace_size(const ep_config *cfg, size_t *bytes);

ep_status ep_dispatch_fused(const ep_config *cfg, const float *logits, const ep_bf16 *x,
                            int32_t *topk_idx, float *topk_w,
                            int32_t *expert_count, int32_t *expert_offset,
                            int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                            ep_chunk *chunks, int32_t chunk_capacity, int32_t *n_chunks,
                            int32_t *worker_begin, ep_bf16 *send, int32_t *slot_meta,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * ep_dispatch_scheduled -- the dispatch driven by the chunk schedule
 * (the UBEP article, "Hierarchical Token-Level Scheduling": each worker moves
 * the rows of its own chunk list).
 *
 * Writes the same send and slot_meta as ep_dispatch, by pulling rows: first
 * slot_meta[slot[t, j]] = t k + j for every valid slot, then CTA c serves
 * worker w = c mod W and copies send[s, :] = x[slot_meta[s] / k, :] for the
 * rows s of worker w's chunks (CTA c takes the part c / W of each chunk, in
 * ep_dispatch_scheduled_ctas / W parts). chunks / n_chunks / worker_begin are
 * device pointers from ep_layout on the same cfg (or any table of the same
 * form whose chunks tile the rows once); rows outside every chunk are not
 * written. Each x row is read k times (from L2 when x fits there).
 *
 * x          : const bf16 [T, H], 16-byte aligned; rows of at most 48 KiB
 *              (EP_ERR_UNSUPPORTED otherwise)
 * slot       : const int32 [T, k] (ep_layout)
 * send       : bf16 [T k, H] output, 16-byte aligned
 * slot_meta  : int32 [T k] output
 * cta_ns     : optional int64 [ep_dispatch_scheduled_ctas][2] output (or
 *              NULL): %globaltimer (ns) when CTA c started and when its last
 *              store had landed, for per-worker timing.
 * A CTA that gives up a bounded wait, or meets a chunk outside [0, T k),
 * sets ep_device_error bit 3 (8).
 */
ep_status ep_dispatch_scheduled_ctas(const ep_config *cfg, int32_t *ctas);

ep_status ep_dispatch_scheduled(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot,
                                const ep_chunk *chunks, const int32_t *n_chunks, const int32_t *worker_begin,
                                ep_bf16 *send, int32_t *slot_meta, int64_t *cta_ns, cudaStream_t stream);

/*
 * Data-as-Flag by Token-Flag Fusion (the UBEP article, "Data-as-Flag", TFF):
 * the 512-byte block codec.
 *
 * Each send row (T k rows of H bf16) travels as ceil(2 H / 480) blocks of 512
 * bytes: 32 bytes of metadata, then 480 bytes of payload (zero after the
 * row's last byte). Metadata: uint32 little-endian {epoch, row, block,
 * nbytes, 0, 0, 0, 0}, where epoch is the flag the receiver waits for, row
 * the send row, block the index inside the row and nbytes the payload bytes
 * the block carries. Row r's blocks are consecutive; rows follow each other.
 *
 * ep_tff_framed_bytes : bytes of the framed buffer, T k ceil(2H/480) 512.
 * ep_tff_encode       : rows [T k, H] -> framed. Every block's payload and
 *                       metadata are stored before its epoch word, which is a
 *                       release store (the GPU has no 512-byte atomic store).
 * ep_tff_decode       : framed -> rows [T k, H]. A block is accepted when its
 *                       metadata reads exactly {epoch, row, block, nbytes}
 *                       (epoch acquire-loaded first); its payload is copied to
 *                       the row. Rejected blocks leave their row bytes as
 *                       they were and are added to *bad_blocks (uint32 in
 *                       device memory, accumulated, not cleared).
 * framed and rows 16-byte aligned; T k ceil(2H/480) <= INT32_MAX.
 */
#define EP_TFF_BLOCK_BYTES 512
#define EP_TFF_META_BYTES 32
#define EP_TFF_PAYLOAD_BYTES 480

ep_status ep_tff_framed_bytes(const ep_config *cfg, size_t *bytes);

ep_status ep_tff_encode(const ep_config *cfg, const ep_bf16 *rows, void *framed, uint32_t epoch,
                        cudaStream_t stream);

ep_status ep_tff_decode(const ep_config *cfg, const void *framed, uint32_t epoch, ep_bf16 *rows,
                        uint32_t *bad_blocks, cudaStream_t stream);

/*
 * Data-as-Flag by Sentinel Polling (the UBEP article, "Data-as-Flag" / SP).
 *
 * The receiver fills its buffer with a sentinel no payload can take, the
 * sender writes raw payload only, and the receiver polls until the sentinel
 * is gone: no flag and no control message. Sentinel: the bf16 bit pattern
 * 0xFFFF (a NaN); finite activations never take it, so x must hold no such
 * value (a row that kept it would be waited on until the bound runs out).
 *
 * ep_sentinel_arm  : fills send [T k, H] with the sentinel (done once; every
 *                    ep_dispatch_expert_sp call leaves it armed again).
 * ep_expert_scale  : the bulk-synchronous counterpart of the consumer below:
 *                    y[s, :] = bf16_rne(float(send[s, :]) * expert_scale[e]),
 *                    e the expert that owns row s (expert_offset, E + 1).
 * ep_dispatch_expert_sp : one cooperative kernel. Producer CTAs dispatch x as
 *                    ep_dispatch does (send, slot_meta); one consumer CTA per
 *                    chunk-schedule worker (chunks / n_chunks / worker_begin,
 *                    all device pointers, from ep_layout on the same cfg)
 *                    polls the rows of its chunks,
 *                    writes y as ep_expert_scale would and writes the
 *                    sentinel back into send. On return y equals
 *                    ep_dispatch + ep_expert_scale, slot_meta equals
 *                    ep_dispatch's, and send is armed again (its payload is
 *                    consumed). Needs k % 4 == 0 and rows of 1..48 KiB
 *                    (EP_ERR_UNSUPPORTED otherwise); slot 16-byte aligned. A
 *                    CTA that gives up a bounded wait sets ep_device_error
 *                    bit 2 (4).
 */
#define EP_SENTINEL_BF16 0xFFFFu

/*
 * ep_dispatch_expert_sw -- the stop-and-wait baseline the same section
 * measures Data-as-Flag against (write data, then a completion flag; the
 * receiver polls the flag, then consumes the data), in the same
 * producer/consumer kernel as ep_dispatch_expert_sp: a producer lane waits
 * until its row has landed, then release-stores `epoch` into row_flag[s]; a
 * consumer acquire-polls row_flag[s] == epoch and then reads the row. send is
 * left holding the payload (nothing to re-arm). Outputs and requirements are
 * those of ep_dispatch_expert_sp; additionally
 *   row_flag : uint32 [T k] device, 4-byte aligned, holding no `epoch` on
 *              entry (e.g. zero-filled once, epoch = 1, 2, ... per call);
 *              holds `epoch` for every row on return.
 * A CTA that gives up a bounded wait sets ep_device_error bit 2 (4).
 */
ep_status ep_dispatch_expert_sw(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot,
                                const int32_t *expert_offset, const float *expert_scale,
                                const ep_chunk *chunks, const int32_t *n_chunks, const int32_t *worker_begin,
                                ep_bf16 *send, int32_t *slot_meta, ep_bf16 *y, uint32_t *row_flag,
                                uint32_t epoch, cudaStream_t stream);

ep_status ep_sentinel_arm(const ep_config *cfg, ep_bf16 *send, cudaStream_t stream);

ep_status ep_expert_scale(const ep_config *cfg, const ep_bf16 *send, const int32_t *expert_offset,
                          const float *expert_scale, ep_bf16 *y, cudaStream_t stream);

ep_status ep_dispatch_expert_sp(const ep_config *cfg, const ep_bf16 *x, const int32_t *slot,
                                const int32_t *expert_offset, const float *expert_scale,
                                const ep_chunk *chunks, const int32_t *n_chunks, const int32_t *worker_begin,
                                ep_bf16 *send, int32_t *slot_meta, ep_bf16 *y, cudaStream_t stream);

/*
 * ep_combine -- gather the k expert-output rows of every token back to token
 * order and sum them with the top-k weights (UBEP article, opening section:
 * the expert outputs come back to their token in the Combine step):
 *   acc = 0; for j = 0 .. k-1: acc = fmaf(topk_w[t, j], y[slot[t, j], h], acc)
 *   out[t, h] = bf16 round-to-nearest-even(acc)
 * in fp32 with one fused multiply-add per term, in fixed j order.
 *
 * y      : const bf16 [T k, H]  expert outputs, in send-buffer (slot) order
 * slot   : const int32 [T, k]   entries outside [0, T k) contribute nothing
 * topk_w : const float [T, k]
 * out    : bf16 [T, H]          output
 */
ep_status ep_combine(const ep_config *cfg, const ep_bf16 *y, const int32_t *slot, const float *topk_w,
                     ep_bf16 *out, cudaStream_t stream);

/*
 * ep_layout_static -- ep_layout for callers that cannot allocate device memory.
 *
 * The paper has no counterpart: this is a property of this library, not of the
 * method. Some callers cannot call cudaMalloc (or any allocator) when they run
 * the layout -- for example an engine that hands a library only the input and
 * output buffers it owns, with all of its device memory carved up once at
 * start-up and no allocator to lend, or code running where a device
 * allocation is not allowed. They cannot pass ep_layout's workspace.
 *
 * This entry point computes exactly what ep_layout computes (same arguments
 * and outputs, same errors) but takes its scratch from a fixed device array
 * inside the library of EP_LAYOUT_STATIC_SCRATCH_BYTES (1 MiB), which every
 * GPU that loads the library holds until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *  - Limit: shapes whose ep_layout_workspace_size exceeds
 *    EP_LAYOUT_STATIC_SCRATCH_BYTES return EP_ERR_CAPACITY with nothing
 *    enqueued. That size is max(a(4 E ceil(T / 256)), a(4 E n)) bytes,
 *    a() rounding up to a multiple of 256 and n <= max(ceil(T / 256), 64)
 *    the single-kernel layout's CTA count: E = 256 allows T <= 262144 tokens
 *    (exactly 1 MiB at T = 262144).
 *  - Set-up: the first call on a device (made with that device current) looks
 *    up the array's device address; make that first call before any stream
 *    capture. Later calls on the device reuse the address, so a
 *    cudaDeviceReset (or anything else that destroys the device's primary
 *    context) leaves it stale: after one, do not call ep_layout_static on that
 *    device again in the same process.
 *  - Sharing: every call on a device shares the one array, which keeps the
 *    last call's contents (the kernels overwrite all of it they read). Calls
 *    whose work overlaps on the GPU -- on different streams, or from
 *    different threads -- race on it: order them on one stream.
 */
#define EP_LAYOUT_STATIC_SCRATCH_BYTES (1u << 20)

ep_status ep_layout_static(const ep_config *cfg, const int32_t *topk_idx,
                           int32_t *expert_count, int32_t *expert_offset,
                           int32_t *rank_count, int32_t *rank_offset, int32_t *slot,
                           ep_chunk *chunks, int32_t chunk_capacity, int32_t *n_chunks,
                           int32_t *worker_begin, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */

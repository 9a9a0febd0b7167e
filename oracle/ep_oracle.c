/*
 * ep_oracle.c -- the CPU oracle for the MoE expert-parallel route -> layout ->
 * dispatch -> combine path.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline / reference arm may load this library. The product path (the CUDA
 * library in combine_router_softmax_gb300/) never calls it, shares no code,
 * header, table or helper with it, and fails if its own extension is missing.
 *
 * Plain, slow, single-threaded C99: every result is written out from its
 * definition with no blocking, fusion or reordering. Floating point is fp64
 * except where the path fixes it: the combine accumulates in fp32 with one
 * fused multiply-add per top-k term in fixed order, then rounds to bf16.
 *
 * Source: "NJU x Huawei UBEP: Reengineering MoE Expert Parallelism" (kad8.com)
 * and the UBEP abstract (arXiv 2607.06202). The pages state the problem
 * (tokens are sent to the device of each selected expert and gathered back
 * in the Combine phase; counts, offsets and reordering are the metadata
 * phases) but define no router, layout or schedule formula. Where they are
 * silent the plainest reading is taken; each such reading is named at the
 * function that makes it.
 *
 * All functions return 0 on success and a negative code on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)
#define ORC_ECAP (-3)

/* ------------------------------------------------------------------------- */
/* bf16 <-> binary32. bf16 is the upper half of an IEEE binary32 word.        */
/* ------------------------------------------------------------------------- */

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest bf16, ties to even (IEEE 754
 * roundTiesToEven applied at bit 16). Overflow rounds to infinity; NaN keeps
 * its sign and becomes a quiet NaN. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t low = u & 0xffffu;          /* the 16 bits that are dropped   */
    uint32_t keep = u >> 16;             /* truncated result               */
    if (low > 0x8000u || (low == 0x8000u && (keep & 1u)))
        keep += 1u;                      /* carries into the exponent: ok  */
    return (uint16_t)keep;
}

/* ------------------------------------------------------------------------- */
/* Route: softmax over the E gate logits, top-k selection, renormalisation.   */
/* ------------------------------------------------------------------------- */

/*
 * The pages say only that MoE models activate a sparse set of experts per
 * token and that each token goes to the device of its selected expert
 * (UBEP article, opening section). They define no router. The plainest
 * reading, used here:
 *
 *   p[t, e]  = exp(l[t, e] - m) / sum_e' exp(l[t, e'] - m),  m = max_e l[t, e]
 *              (softmax over all E experts, fp64)
 *   idx[t, :] = the k experts with the largest logits, in descending order of
 *              logit; equal logits go to the lower expert index. Softmax is
 *              monotone, so this is also descending probability.
 *   w[t, j]  = p[t, idx[t, j]] / sum_i p[t, idx[t, i]]  when renormalize,
 *              else p[t, idx[t, j]].
 *
 * Group-limited routing (n_groups > 1): experts split into n_groups
 * contiguous groups of E / n_groups; a group's score is its largest logit;
 * the topk_groups best groups are kept (ties to the lower group index) and
 * the top-k is taken among the kept experts only. The softmax denominator
 * still runs over all E experts.
 *
 * Output w is fp64 (the pages fix no precision).
 */
int orc_route(int64_t T, int32_t E, int32_t k, int32_t n_groups, int32_t topk_groups,
              int32_t renormalize, const float *logits, int32_t *idx, double *w)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E || n_groups <= 0 || E % n_groups != 0 ||
        topk_groups <= 0 || topk_groups > n_groups || (int64_t)topk_groups * (E / n_groups) < k)
        return ORC_EINVAL;
    if (T > 0 && (!logits || !idx || !w))
        return ORC_EINVAL;

    const int32_t gsize = E / n_groups;
    char *eligible = (char *)malloc((size_t)E);
    char *taken = (char *)malloc((size_t)E);
    char *gkept = (char *)malloc((size_t)n_groups);
    float *gscore = (float *)malloc(sizeof(float) * (size_t)n_groups);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    if (!eligible || !taken || !gkept || !gscore || !p) {
        free(eligible); free(taken); free(gkept); free(gscore); free(p);
        return ORC_ENOMEM;
    }

    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * (int64_t)E;

        /* Which experts may be chosen. */
        for (int32_t e = 0; e < E; ++e) eligible[e] = 1;
        if (n_groups > 1) {
            for (int32_t g = 0; g < n_groups; ++g) {
                float s = l[g * gsize];
                for (int32_t i = 1; i < gsize; ++i)
                    if (l[g * gsize + i] > s) s = l[g * gsize + i];
                gscore[g] = s;
                gkept[g] = 0;
            }
            for (int32_t r = 0; r < topk_groups; ++r) {
                int32_t best = -1;
                for (int32_t g = 0; g < n_groups; ++g)
                    if (!gkept[g] && (best < 0 || gscore[g] > gscore[best])) best = g;
                gkept[best] = 1;
            }
            for (int32_t e = 0; e < E; ++e) eligible[e] = gkept[e / gsize];
        }

        /* Top-k by raw logit: repeatedly take the largest remaining logit,
         * scanning experts upwards so that a tie keeps the lower index. */
        for (int32_t e = 0; e < E; ++e) taken[e] = 0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (eligible[e] && !taken[e] && (best < 0 || l[e] > l[best])) best = e;
            taken[best] = 1;
            idx[t * k + j] = best;
        }

        /* Softmax over all E experts, fp64. */
        double m = (double)l[0];
        for (int32_t e = 1; e < E; ++e)
            if ((double)l[e] > m) m = (double)l[e];
        double S = 0.0;
        for (int32_t e = 0; e < E; ++e) {
            p[e] = exp((double)l[e] - m);
            S += p[e];
        }
        for (int32_t e = 0; e < E; ++e) p[e] /= S;

        /* Top-k weights, renormalised over the chosen k when asked. */
        double s = 0.0;
        for (int32_t j = 0; j < k; ++j) s += p[idx[t * k + j]];
        for (int32_t j = 0; j < k; ++j)
            w[t * k + j] = renormalize ? p[idx[t * k + j]] / s : p[idx[t * k + j]];
    }

    free(eligible); free(taken); free(gkept); free(gscore); free(p);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Layout: counts, offsets and the stable slot of every (token, expert) pair. */
/* ------------------------------------------------------------------------- */

/*
 * The BSP pipeline the UBEP article describes ("Three Bottlenecks", BSP
 * Serialization; "Kernel Decomposition") counts tokens, computes offsets by
 * prefix sums and reorders tokens. Written out for one device holding R
 * virtual expert-parallel ranks:
 *
 *   rank(e)          = e / (E / R)            contiguous blocks of experts per
 *                                             rank (the pages say nothing;
 *                                             plainest reading)
 *   expert_count[e]  = #{(t, j) : idx[t, j] = e}
 *   expert_offset[e] = sum_{e' < e} expert_count[e'],  expert_offset[E] = T k
 *   rank_offset[r]   = expert_offset[r E / R],         rank_offset[R] = T k
 *   rank_count[r]    = rank_offset[r + 1] - rank_offset[r]
 *   slot[t, j]       = expert_offset[e] + #{t' < t : e in idx[t', :]},  e = idx[t, j]
 *
 * so the send buffer is ordered by (destination rank, expert, source token).
 * No capacity limit and no dropping: the send buffer has exactly T k rows.
 * The k experts of one token must be distinct and in [0, E); anything else
 * is rejected.
 */
int orc_layout(int64_t T, int32_t E, int32_t R, int32_t k, const int32_t *idx,
               int32_t *expert_count, int32_t *expert_offset,
               int32_t *rank_count, int32_t *rank_offset, int32_t *slot)
{
    if (T < 0 || E <= 0 || R <= 0 || E % R != 0 || k <= 0 || k > E)
        return ORC_EINVAL;
    if (T * k > INT32_MAX)
        return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = idx[t * k + j];
            if (e < 0 || e >= E) return ORC_EINVAL;
            for (int32_t i = 0; i < j; ++i)
                if (idx[t * k + i] == e) return ORC_EINVAL;
        }

    for (int32_t e = 0; e < E; ++e) expert_count[e] = 0;
    for (int64_t i = 0; i < T * k; ++i) expert_count[idx[i]] += 1;

    expert_offset[0] = 0;
    for (int32_t e = 0; e < E; ++e) expert_offset[e + 1] = expert_offset[e] + expert_count[e];

    const int32_t epr = E / R;
    for (int32_t r = 0; r <= R; ++r) rank_offset[r] = expert_offset[r * epr];
    for (int32_t r = 0; r < R; ++r) rank_count[r] = rank_offset[r + 1] - rank_offset[r];

    /* Tokens in ascending order, one cursor per expert: the cursor of e has
     * advanced once for every earlier token that chose e. */
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!cursor) return ORC_ENOMEM;
    for (int32_t e = 0; e < E; ++e) cursor[e] = expert_offset[e];
    for (int64_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = idx[t * k + j];
            slot[t * k + j] = cursor[e];
            cursor[e] += 1;
        }
    free(cursor);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Chunk schedule: latency homogenization over hop classes.                   */
/* ------------------------------------------------------------------------- */

/*
 * "Hierarchical Token-Level Scheduling" / "Latency Homogenization" (UBEP
 * article): tokens are classed by network hop count and every worker gets a
 * balanced mixture of the latency classes; the same section says the scheme
 * extends to fabrics with more switch tiers. The pages give the goal, not the
 * heuristic; the plainest closed form is used:
 *
 *   hop_class(r) = 0 if r / ranks_per_node == self_rank / ranks_per_node
 *                  (same node, self included);
 *                  2 if ranks_per_pod > 0 and
 *                  r / ranks_per_pod != self_rank / ranks_per_pod (another
 *                  pod: one more switch tier);
 *                  1 otherwise (another node: the two-hop access of
 *                  "Topology-Agnostic Scheduling").
 *                  ranks_per_pod = 0 means no pod tier (classes 0 and 1 only);
 *                  else it is a multiple of ranks_per_node.
 *   S_c          = the rank segments [rank_offset[r], rank_offset[r+1]) of
 *                  class c concatenated in ascending r; N_c rows in all.
 *   worker w     takes positions [floor(N_c w / W), floor(N_c (w+1) / W)) of
 *                  every S_c (64-bit products), so any two workers' shares
 *                  of a class differ by at most one row.
 *
 * A share cut at rank boundaries gives chunks {worker, hop_class, dst_rank,
 * row_begin, row_count}; empty chunks are omitted. Table order: worker
 * ascending, then class descending (the farthest traffic first), then rank
 * ascending. worker_begin[w] is the index of worker w's first chunk and
 * worker_begin[W] the number of chunks. chunks holds 5 int32 per record.
 */
static int orc_hop_class(int32_t r, int32_t ranks_per_node, int32_t ranks_per_pod, int32_t self_rank)
{
    if (r / ranks_per_node == self_rank / ranks_per_node) return 0;
    if (ranks_per_pod > 0 && r / ranks_per_pod != self_rank / ranks_per_pod) return 2;
    return 1;
}

int orc_schedule(int32_t R, int32_t ranks_per_node, int32_t ranks_per_pod, int32_t self_rank, int32_t W,
                 const int32_t *rank_offset, int32_t *chunks, int32_t capacity,
                 int32_t *n_chunks, int32_t *worker_begin)
{
    if (R <= 0 || ranks_per_node <= 0 || self_rank < 0 || self_rank >= R || W <= 0 || capacity < 0)
        return ORC_EINVAL;
    if (ranks_per_pod < 0 || (ranks_per_pod > 0 && ranks_per_pod % ranks_per_node != 0))
        return ORC_EINVAL;
    int64_t N[3] = {0, 0, 0};
    for (int32_t r = 0; r < R; ++r)
        N[orc_hop_class(r, ranks_per_node, ranks_per_pod, self_rank)] +=
            (int64_t)rank_offset[r + 1] - rank_offset[r];

    int32_t n = 0;
    for (int32_t w = 0; w < W; ++w) {
        worker_begin[w] = n;
        for (int c = 2; c >= 0; --c) {
            int64_t lo = N[c] * w / W;
            int64_t hi = N[c] * (w + 1) / W;
            int64_t pos = 0; /* start of the current rank's segment inside S_c */
            for (int32_t r = 0; r < R; ++r) {
                if (orc_hop_class(r, ranks_per_node, ranks_per_pod, self_rank) != c) continue;
                int64_t seg_lo = pos;
                int64_t seg_hi = pos + ((int64_t)rank_offset[r + 1] - rank_offset[r]);
                pos = seg_hi;
                int64_t a = lo > seg_lo ? lo : seg_lo;
                int64_t b = hi < seg_hi ? hi : seg_hi;
                if (b <= a) continue;
                if (n >= capacity) return ORC_ECAP;
                int32_t *rec = chunks + 5 * (int64_t)n;
                rec[0] = w;
                rec[1] = c;
                rec[2] = r;
                rec[3] = (int32_t)(rank_offset[r] + (a - seg_lo));
                rec[4] = (int32_t)(b - a);
                n += 1;
            }
        }
    }
    worker_begin[W] = n;
    *n_chunks = n;
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Dispatch and combine.                                                      */
/* ------------------------------------------------------------------------- */

/*
 * Dispatch (UBEP article, opening section: a token travels to the device that
 * holds each expert chosen for it): every token row is copied, bit for bit, to
 * the send-buffer row of each of its k slots, and that row records where it
 * came from:  send[slot[t, j], :] = x[t, :],  meta[slot[t, j]] = t k + j.
 */
int orc_dispatch(int64_t T, int32_t H, int32_t k, const uint16_t *x, const int32_t *slot,
                 uint16_t *send, int32_t *meta)
{
    if (T < 0 || H <= 0 || k <= 0) return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int64_t s = slot[t * k + j];
            if (s < 0 || s >= T * k) return ORC_EINVAL;
            for (int32_t h = 0; h < H; ++h)
                send[s * H + h] = x[t * H + h];
            meta[s] = (int32_t)(t * k + j);
        }
    return ORC_OK;
}

/*
 * Combine (the same section: tokens are gathered back in the Combine phase):
 * the k expert outputs of token t are summed with its top-k weights,
 *
 *   acc = 0;  for j = 0 .. k-1:  acc = fmaf(w[t, j], y[slot[t, j], h], acc)
 *   out[t, h] = bf16_rne(acc)
 *
 * in fp32 with one fused multiply-add per term, in fixed j order (the
 * accumulation order and precision are fixed for this path; the pages
 * are silent).
 */
int orc_combine(int64_t T, int32_t H, int32_t k, const uint16_t *y, const int32_t *slot,
                const float *w, uint16_t *out)
{
    if (T < 0 || H <= 0 || k <= 0) return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                int64_t s = slot[t * k + j];
                if (s < 0 || s >= T * k) return ORC_EINVAL;
                acc = fmaf(w[t * k + j], orc_bf16_to_f32(y[s * H + h]), acc);
            }
            out[t * H + h] = orc_f32_to_bf16(acc);
        }
    return ORC_OK;
}

/*
 * The synthetic expert of the test harness (not part of the path): the
 * output row of slot s is its input row scaled by (e + 1) / E, e the expert
 * that owns s, rounded to bf16:
 *   y[s, h] = bf16_rne(float(send[s, h]) * ((float)(e + 1) / (float)E)).
 * With identity != 0 the expert is the identity instead (y = send).
 */
int orc_expert_scale(int64_t rows, int32_t H, int32_t E, const int32_t *expert_offset,
                     int32_t identity, const uint16_t *send, uint16_t *y)
{
    if (rows < 0 || H <= 0 || E <= 0) return ORC_EINVAL;
    int32_t e = 0;
    for (int64_t s = 0; s < rows; ++s) {
        while (e < E - 1 && s >= expert_offset[e + 1]) ++e;
        float scale = (float)(e + 1) / (float)E;
        for (int32_t h = 0; h < H; ++h) {
            if (identity)
                y[s * H + h] = send[s * H + h];
            else
                y[s * H + h] = orc_f32_to_bf16(orc_bf16_to_f32(send[s * H + h]) * scale);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Data-as-Flag: the Token-Flag Fusion block codec.                           */
/* ------------------------------------------------------------------------- */

/*
 * "Data-as-Flag" / TFF (UBEP article): each 512-byte block carries 32 bytes
 * of synchronization metadata and 480 bytes of token payload, so the flag
 * travels with the data. The pages give the split, not the fields; the
 * plainest reading, in the order the pages list the two parts:
 *
 *   block = [ metadata 32 B | payload 480 B ]
 *   metadata = uint32 { epoch, row, block, nbytes, 0, 0, 0, 0 }
 *     epoch : the flag (the value the receiver waits for)
 *     row   : the send-buffer row the block belongs to
 *     block : its index inside the row
 *     nbytes: payload bytes it carries (480, or the row's remainder)
 *   payload = row bytes [480 block, 480 block + nbytes), zero after nbytes.
 *
 * A row of row_bytes bytes takes ceil(row_bytes / 480) blocks; row r's
 * blocks are consecutive and rows follow each other. Integers are stored
 * little-endian.
 */
#define ORC_TFF_BLOCK 512
#define ORC_TFF_META 32
#define ORC_TFF_PAYLOAD 480

int64_t orc_tff_blocks_per_row(int64_t row_bytes)
{
    return (row_bytes + ORC_TFF_PAYLOAD - 1) / ORC_TFF_PAYLOAD;
}

static void orc_put_u32(unsigned char *p, uint32_t v)
{
    p[0] = (unsigned char)(v & 0xFFu);
    p[1] = (unsigned char)((v >> 8) & 0xFFu);
    p[2] = (unsigned char)((v >> 16) & 0xFFu);
    p[3] = (unsigned char)((v >> 24) & 0xFFu);
}

static uint32_t orc_get_u32(const unsigned char *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

int orc_tff_encode(int64_t rows, int64_t row_bytes, const unsigned char *in, uint32_t epoch,
                   unsigned char *framed)
{
    if (rows < 0 || row_bytes <= 0) return ORC_EINVAL;
    const int64_t nblk = orc_tff_blocks_per_row(row_bytes);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nblk; ++b) {
            unsigned char *blk = framed + (r * nblk + b) * ORC_TFF_BLOCK;
            const int64_t off = b * ORC_TFF_PAYLOAD;
            const int64_t n = row_bytes - off < ORC_TFF_PAYLOAD ? row_bytes - off : ORC_TFF_PAYLOAD;
            memset(blk, 0, ORC_TFF_BLOCK);
            orc_put_u32(blk + 0, epoch);
            orc_put_u32(blk + 4, (uint32_t)r);
            orc_put_u32(blk + 8, (uint32_t)b);
            orc_put_u32(blk + 12, (uint32_t)n);
            memcpy(blk + ORC_TFF_META, in + r * row_bytes + off, (size_t)n);
        }
    return ORC_OK;
}

/*
 * The receiver's side: a block is accepted when its metadata reads
 * {epoch, row, block, nbytes} as the encoder wrote them; its payload is then
 * copied to the row. Blocks that do not match are counted in *bad and their
 * bytes are left as they were in `out`.
 */
int orc_tff_decode(int64_t rows, int64_t row_bytes, const unsigned char *framed, uint32_t epoch,
                   unsigned char *out, int64_t *bad)
{
    if (rows < 0 || row_bytes <= 0 || !bad) return ORC_EINVAL;
    const int64_t nblk = orc_tff_blocks_per_row(row_bytes);
    int64_t nbad = 0;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nblk; ++b) {
            const unsigned char *blk = framed + (r * nblk + b) * ORC_TFF_BLOCK;
            const int64_t off = b * ORC_TFF_PAYLOAD;
            const int64_t n = row_bytes - off < ORC_TFF_PAYLOAD ? row_bytes - off : ORC_TFF_PAYLOAD;
            if (orc_get_u32(blk + 0) != epoch || orc_get_u32(blk + 4) != (uint32_t)r ||
                orc_get_u32(blk + 8) != (uint32_t)b || orc_get_u32(blk + 12) != (uint32_t)n) {
                nbad += 1;
                continue;
            }
            memcpy(out + r * row_bytes + off, blk + ORC_TFF_META, (size_t)n);
        }
    *bad = nbad;
    return ORC_OK;
}

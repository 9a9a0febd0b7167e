// route_token.cuh -- one token's softmax + top-k on one warp (ep_route and the
// fused dispatch share it).
//
// Lane l holds logits e = l + 32 i (coalesced 128-byte loads). Selection
// compares raw fp32 logits under the total order (logit desc, index asc), so
// the chosen experts do not depend on the exp implementation:
//   1. tau = the k-th largest of the 32 lane maxima (a 15-step bitonic sort of
//      one float per lane). At least k logits are >= tau, so the top k all are.
//   2. The logits >= tau are the candidates; a warp prefix sum packs them into
//      shared memory (usually 8-12 of them for k = 8).
//   3. If there are at most 32, each candidate counts the candidates ordered
//      before it; that count is its rank, and the top k are written straight
//      to their places. Otherwise (massive ties) k rounds of a butterfly
//      arg-max pick them.
// Group-limited routing keeps the topk_groups groups with the largest
// per-group maximum logit (ties to the lower group) before step 1.
//
// Weights: with renormalisation the full softmax denominator cancels, so
// w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k picks only; pick 0
// is the global maximum (the group holding it always survives group
// limiting). Without it, w_j = exp(l_j - l_max) / sum over all E.
#pragma once

#include <climits>

#include "ep_internal.cuh"

namespace ep {
namespace {

// (va, ia) ranks before (vb, ib): larger logit, or equal logit and lower index.
// INT_MAX marks "no candidate" and never ranks before a real entry.
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
    if (ia == INT_MAX) return false;
    if (ib == INT_MAX) return true;
    return va > vb || (va == vb && ia < ib);
}

// Butterfly arg-max over the warp under `before`; every lane ends with the winner.
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, m);
        const int oi = __shfl_xor_sync(0xffffffffu, i, m);
        if (before(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// Bitonic sort of one float per lane, descending in lane order.
__device__ __forceinline__ float warp_sort_desc(float s, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, s, stride);
            const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
            s = keep_max ? fmaxf(s, o) : fminf(s, o);
        }
    }
    return s;
}

// Group limiting: clears the elig bits of experts outside the topk_groups
// groups with the largest per-group maximum logit (ties to the lower group).
//
// When a group is a power-of-two run of at most 32 experts (every group then
// lies in gsize consecutive lanes of one register), the group maxima come from
// shuffles inside each run and each group's rank is counted against all the
// others (lane g < n_groups holds group g); otherwise through shared memory
// with topk_groups rounds of arg-max. Both keep the same groups.
template <int VPL>
__device__ __forceinline__ uint32_t group_limit(const float (&v)[VPL], uint32_t elig, int32_t E, int32_t n_groups,
                                                int32_t topk_groups, int lane, float *s_glog) {
    const int gsize = E / n_groups;
    if (gsize <= 32 && (32 % gsize) == 0) {
        float gm[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            float m = lane + 32 * i < E ? v[i] : -INFINITY;
            for (int off = gsize >> 1; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            gm[i] = m;
        }
        // lane g < n_groups fetches group g's maximum: register g gsize / 32, lane g gsize % 32
        const int src = (lane * gsize) & 31, reg = (lane * gsize) >> 5;
        float gs = -INFINITY;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const float t = __shfl_sync(0xffffffffu, gm[i], src);
            if (i == reg) gs = t;
        }
        const bool mine = lane < n_groups;
        int rank = 0;  // groups ordered before mine: larger maximum, or equal and lower index
        for (int g = 0; g < n_groups; ++g) {
            const float o = __shfl_sync(0xffffffffu, gs, g);
            rank += (o > gs || (o == gs && g < lane)) ? 1 : 0;
        }
        const uint32_t kept = __ballot_sync(0xffffffffu, mine && rank < topk_groups);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((kept >> (e / gsize)) & 1u)) elig &= ~(1u << i);
        }
        return elig;
    }
    float *sl = s_glog;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) sl[e] = v[i];
    }
    __syncwarp();
    float gs = -INFINITY;
    bool avail = lane < n_groups;
    if (avail) {
        gs = sl[lane * gsize];
        for (int q = 1; q < gsize; ++q) {
            const float c = sl[lane * gsize + q];
            if (c > gs) gs = c;
        }
    }
    uint32_t kept = 0;
    for (int r = 0; r < topk_groups; ++r) {
        float bv = gs;
        int bi = avail ? lane : INT_MAX;
        warp_argmax(bv, bi);
        kept |= 1u << bi;
        if (lane == bi) avail = false;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((kept >> (e / gsize)) & 1u)) elig &= ~(1u << i);
    }
    return elig;
}

// Massive ties (more than 32 candidates): k rounds of arg-max; lane j ends
// with pick j.
template <int VPL>
__device__ __forceinline__ void topk_by_rounds(const float (&v)[VPL], uint32_t elig, int32_t k, int lane,
                                               float &my_v, int &my_e) {
    uint32_t avail = elig;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (((avail >> i) & 1u) && (bi == INT_MAX || v[i] > bv)) {  // ascending e: strict > keeps the lower index
                bv = v[i];
                bi = lane + 32 * i;
            }
        }
        warp_argmax(bv, bi);
        if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
        if (lane == j) {
            my_v = bv;
            my_e = bi;
        }
    }
}

// The same two, out of line: in the fused small-batch kernel, whose time at
// small T goes largely to fetching its own code after the caches were emptied,
// rarely taken paths are kept out of the instruction stream of the common one
// (measured: T = 1 -1.0 us, T = 8 -1.0 us, T = 64 -1.7 us, decode -0.6 us per
// layer; in the route kernel, with many tokens per launch, they stay inline:
// there the calls cost 0.6 us at prefill and 2 us at mid).
template <int VPL>
__device__ __noinline__ uint32_t group_limit_cold(const float (&v)[VPL], uint32_t elig, int32_t E, int32_t n_groups,
                                                  int32_t topk_groups, int lane, float *s_glog) {
    return group_limit<VPL>(v, elig, E, n_groups, topk_groups, lane, s_glog);
}
template <int VPL>
__device__ __noinline__ void topk_by_rounds_cold(const float (&v)[VPL], uint32_t elig, int32_t k, int lane,
                                                 float &my_v, int &my_e) {
    topk_by_rounds<VPL>(v, elig, k, lane, my_v, my_e);
}

// Routes the token whose logits start at `row`; on return lane j < k holds
// pick j (out_e, out_w). s_glog: E floats (group-limited routing only);
// s_cand, s_pick: 32 int2 each. The whole warp must call it. kColdOutOfLine:
// call the out-of-line group limiting and tie fallback.
template <int VPL, bool kColdOutOfLine = false>
__device__ __forceinline__ void route_token(const float *__restrict__ row, int32_t E, int32_t k, int32_t n_groups,
                                            int32_t topk_groups, int32_t renormalize, int lane, float *s_glog,
                                            int2 *s_cand, int2 *s_pick, int &out_e, float &out_w) {
    float v[VPL];
    uint32_t elig = 0;  // bit i: value i may be picked
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            v[i] = __ldg(row + e);
            elig |= 1u << i;
        } else {
            v[i] = -INFINITY;
        }
    }

    if (n_groups > 1) {
        // Group score = largest logit of the group; keep the topk_groups best.
        elig = kColdOutOfLine ? group_limit_cold<VPL>(v, elig, E, n_groups, topk_groups, lane, s_glog)
                              : group_limit<VPL>(v, elig, E, n_groups, topk_groups, lane, s_glog);
    }

    // 1. tau = k-th largest lane maximum.
    float lmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if ((elig >> i) & 1u) lmax = fmaxf(lmax, v[i]);
    const float tau = __shfl_sync(0xffffffffu, warp_sort_desc(lmax, lane), k - 1);

    // 2. candidates (eligible logits >= tau), packed by a warp prefix sum.
    int c = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) c += (((elig >> i) & 1u) && v[i] >= tau) ? 1 : 0;
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    const int C = __shfl_sync(0xffffffffu, incl, 31);

    float my_v = -INFINITY;
    int my_e = INT_MAX;  // lane j < k ends with pick j
    if (C <= 32) {
        int pos = incl - c;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (((elig >> i) & 1u) && v[i] >= tau) {
                s_cand[pos] = make_int2(__float_as_int(v[i]), lane + 32 * i);
                ++pos;
            }
        }
        __syncwarp();
        // 3. a candidate's rank is the number of candidates ordered before it
        //    (unique: indices differ); the top k go straight to their place.
        if (lane < C) {
            const int2 me = s_cand[lane];
            const float mv = __int_as_float(me.x);
            int rank = 0;
            for (int j = 0; j < C; ++j) {
                const int2 o = s_cand[j];
                const float ov = __int_as_float(o.x);
                rank += (ov > mv || (ov == mv && o.y < me.y)) ? 1 : 0;
            }
            if (rank < k) s_pick[rank] = me;
        }
        __syncwarp();
        if (lane < k) {
            const int2 pk = s_pick[lane];
            my_v = __int_as_float(pk.x);
            my_e = pk.y;
        }
    } else if (kColdOutOfLine) {
        topk_by_rounds_cold<VPL>(v, elig, k, lane, my_v, my_e);  // massive ties
    } else {
        topk_by_rounds<VPL>(v, elig, k, lane, my_v, my_e);  // massive ties
    }

    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    float w;
    if (renormalize) {
        const float ex = lane < k ? expf(my_v - m) : 0.f;
        w = ex / warp_sum(ex);
    } else {
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (lane + 32 * i < E) part += expf(v[i] - m);
        w = expf(my_v - m) / warp_sum(part);
    }
    out_e = my_e;
    out_w = w;
}

}  // namespace
}  // namespace ep

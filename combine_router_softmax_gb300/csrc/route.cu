// route.cu -- router softmax + top-k (ep_route).
//
// What it computes is fixed by ep.h: top-k experts by raw logit (ties to the
// lower index, optionally restricted to the best groups by per-group maximum),
// and their softmax weights, renormalised over the k chosen when asked. The
// UBEP article only says each token goes to the device of its selected expert
// (opening section); the router itself is the plainest reading.
//
// Design: one warp per token. Lane l holds logits e = l + 32 i (coalesced
// 128-byte loads), VPL values per lane. Each of the k picks is a lane-local
// scan followed by a 5-step butterfly arg-max over (logit desc, index asc),
// which every lane resolves identically. Selection compares raw fp32 logits,
// so the chosen experts do not depend on the exp implementation.
//
// Weights: with renormalisation the full softmax denominator cancels, so
// w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k picks only; pick 0
// is the global maximum (the group holding it always survives group
// limiting). Without it, w_j = exp(l_j - l_max) / sum over all E.
#include <cfloat>
#include <climits>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kRouteWarps = 8;  // tokens per CTA

// Butterfly arg-max step on (v, i): larger v wins, equal v -> smaller i wins;
// i == INT_MAX marks "no candidate" and never wins.
__device__ __forceinline__ void argmax_xor(float &v, int &i, int lane_mask) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, lane_mask);
    const int oi = __shfl_xor_sync(0xffffffffu, i, lane_mask);
    const bool take = (oi != INT_MAX) && (i == INT_MAX || ov > v || (ov == v && oi < i));
    if (take) {
        v = ov;
        i = oi;
    }
}

__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) argmax_xor(v, i, m);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

template <int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const float *__restrict__ logits, int32_t T, int32_t E, int32_t k, int32_t n_groups,
             int32_t topk_groups, int32_t renormalize, int32_t *__restrict__ topk_idx,
             float *__restrict__ topk_w) {
    extern __shared__ float s_logits[];  // [kRouteWarps][E], group-limited routing only
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * kRouteWarps + warp;
    if (t >= T) return;  // whole warp leaves together; no CTA-wide barrier follows

    const float *row = logits + t * E;
    float v[VPL];
    uint32_t out = 0;  // bit i set: value i cannot be picked (absent, masked or taken)
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            v[i] = __ldg(row + e);
        } else {
            v[i] = -FLT_MAX;
            out |= 1u << i;
        }
    }

    if (n_groups > 1) {
        // Group score = largest logit of the group; keep the topk_groups best.
        float *sl = s_logits + warp * E;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) sl[e] = v[i];
        }
        __syncwarp();
        const int gsize = E / n_groups;
        float gs = -FLT_MAX;
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
            if (e < E && !((kept >> (e / gsize)) & 1u)) out |= 1u << i;
        }
    }

    // k picks; lane j keeps pick j.
    float my_v = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -FLT_MAX;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (!((out >> i) & 1u) && (bi == INT_MAX || v[i] > bv)) {  // ascending e: strict > keeps the lower index
                bv = v[i];
                bi = lane + 32 * i;
            }
        }
        warp_argmax(bv, bi);
        if ((bi & 31) == lane) out |= 1u << (bi >> 5);
        if (lane == j) {
            my_v = bv;
            my_e = bi;
        }
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
    if (lane < k) {
        topk_idx[t * k + lane] = my_e;
        topk_w[t * k + lane] = w;
    }
}

template <int VPL>
cudaError_t launch_vpl(const ep_config &c, const float *logits, int32_t *idx, float *w, cudaStream_t s) {
    const size_t smem = c.n_groups > 1 ? sizeof(float) * kRouteWarps * (size_t)c.E : 0;
    const unsigned grid = (unsigned)((c.T + kRouteWarps - 1) / kRouteWarps);
    route_kernel<VPL><<<grid, kRouteWarps * 32, smem, s>>>(logits, c.T, c.E, c.k, c.n_groups, c.topk_groups,
                                                         c.renormalize, idx, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const ep_config &c, const float *logits, int32_t *idx, float *w, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    const int vpl = (c.E + 31) / 32;
    if (vpl <= 1) return launch_vpl<1>(c, logits, idx, w, s);
    if (vpl <= 2) return launch_vpl<2>(c, logits, idx, w, s);
    if (vpl <= 4) return launch_vpl<4>(c, logits, idx, w, s);
    if (vpl <= 8) return launch_vpl<8>(c, logits, idx, w, s);
    if (vpl <= 16) return launch_vpl<16>(c, logits, idx, w, s);
    return launch_vpl<32>(c, logits, idx, w, s);
}

}  // namespace ep

// route.cu -- router softmax + top-k (ep_route).
//
// What it computes is fixed by ep.h: top-k experts by raw logit (ties to the
// lower index, optionally restricted to the best groups by per-group maximum),
// and their softmax weights, renormalised over the k chosen when asked. The
// UBEP article only says each token goes to the device of its selected expert
// (opening section); the router itself is the plainest reading.
//
// One warp per token (route_token.cuh); 8 tokens per CTA.
#include "route_token.cuh"

namespace ep {
namespace {

constexpr int kRouteWarps = 8;  // tokens per CTA

template <int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const float *__restrict__ logits, int32_t T, int32_t E, int32_t k, int32_t n_groups,
             int32_t topk_groups, int32_t renormalize, int32_t *__restrict__ topk_idx,
             float *__restrict__ topk_w, unsigned *__restrict__ zero_a, int n_zero_a, unsigned *__restrict__ zero_b,
             int n_zero_b, int32_t *__restrict__ zero_c) {
    extern __shared__ float s_dyn[];  // [kRouteWarps][E] logits, group-limited routing only
    // A layout launched after this kernel may start now: it waits for this
    // grid before it reads anything this one writes.
    grid_launch_dependents();
    // Reset what later kernels of the same call sequence start from: zero_a
    // (the layout's count table) over all CTAs, the rest by the first.
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero_a; i += gridDim.x * blockDim.x) zero_a[i] = 0u;
    if (blockIdx.x == 0) {
        if ((int)threadIdx.x < n_zero_b) zero_b[threadIdx.x] = 0u;
        if (threadIdx.x == 0 && zero_c) *zero_c = 0;
    }
    __shared__ int2 s_cand[kRouteWarps][32];  // candidate (logit bits, expert)
    __shared__ int2 s_pick[kRouteWarps][32];  // the k picks in order
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * kRouteWarps + warp;
    if (t >= T) return;  // whole warp leaves together; no CTA-wide barrier follows
    int e;
    float w;
    route_token<VPL>(logits + t * E, E, k, n_groups, topk_groups, renormalize, lane, s_dyn + warp * E,
                     s_cand[warp], s_pick[warp], e, w);
    if (lane < k) {
        topk_idx[t * k + lane] = e;
        topk_w[t * k + lane] = w;
    }
}
template <int VPL>
cudaError_t launch_vpl(const ep_config &c, const float *logits, int32_t *idx, float *w, cudaStream_t s,
                       unsigned *za, int na, unsigned *zb, int nb, int32_t *zc) {
    const size_t smem = c.n_groups > 1 ? sizeof(float) * kRouteWarps * (size_t)c.E : 0;
    const unsigned grid = (unsigned)((c.T + kRouteWarps - 1) / kRouteWarps);
    route_kernel<VPL><<<grid, kRouteWarps * 32, smem, s>>>(logits, c.T, c.E, c.k, c.n_groups, c.topk_groups,
                                                         c.renormalize, idx, w, za, na, zb, nb, zc);
    return cudaGetLastError();
}

}  // namespace

bool route_one_wave(const ep_config &c) {
    const int vpl = (c.E + 31) / 32;
    const void *fn = vpl <= 1 ? reinterpret_cast<const void *>(route_kernel<1>)
                   : vpl <= 2 ? reinterpret_cast<const void *>(route_kernel<2>)
                   : vpl <= 4 ? reinterpret_cast<const void *>(route_kernel<4>)
                   : vpl <= 8 ? reinterpret_cast<const void *>(route_kernel<8>)
                   : vpl <= 16 ? reinterpret_cast<const void *>(route_kernel<16>)
                               : reinterpret_cast<const void *>(route_kernel<32>);
    const size_t smem = c.n_groups > 1 ? sizeof(float) * kRouteWarps * (size_t)c.E : 0;
    const int64_t ctas = ((int64_t)c.T + kRouteWarps - 1) / kRouteWarps;
    return ctas <= (int64_t)current_device_sm_count() * max_blocks_per_sm(fn, kRouteWarps * 32, smem);
}

cudaError_t launch_route(const ep_config &c, const float *logits, int32_t *idx, float *w, cudaStream_t s,
                         unsigned *za, int na, unsigned *zb, int nb, int32_t *zc) {
    if (c.T == 0) return cudaSuccess;
    const int vpl = (c.E + 31) / 32;
    if (vpl <= 1) return launch_vpl<1>(c, logits, idx, w, s, za, na, zb, nb, zc);
    if (vpl <= 2) return launch_vpl<2>(c, logits, idx, w, s, za, na, zb, nb, zc);
    if (vpl <= 4) return launch_vpl<4>(c, logits, idx, w, s, za, na, zb, nb, zc);
    if (vpl <= 8) return launch_vpl<8>(c, logits, idx, w, s, za, na, zb, nb, zc);
    if (vpl <= 16) return launch_vpl<16>(c, logits, idx, w, s, za, na, zb, nb, zc);
    return launch_vpl<32>(c, logits, idx, w, s, za, na, zb, nb, zc);
}

}  // namespace ep

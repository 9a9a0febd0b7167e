// dispatch.cu -- row scatter into the rank-partitioned send buffer (ep_dispatch).
//
// send[slot[t, j], :] = x[t, :] and slot_meta[slot[t, j]] = t k + j: each token
// row goes to the send-buffer row of every selected expert ("each token must
// be dispatched to the device hosting its selected expert", UBEP article,
// opening section). This is the data-movement half of the article's kernel
// decomposition; on one GPU it is a pure HBM copy: read x once, write k rows.
//
// Work unit = (token, segment of 32 * U 16-byte vectors). A warp loads its U
// vectors per lane once (non-allocating streaming loads) and stores them to
// the k destination rows, so each x byte is read once and each send byte
// written once. Units are spread over a grid sized to the resident capacity
// of the GPU, which keeps the load balanced when T is small relative to the
// SM count and rows are long (H = 7168: 7 segments per row).
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kDispatchThreads = 256;
constexpr int kDispatchU = 4;  // vectors per lane per unit: 4 x 16 B in flight

template <int K>
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ slot, uint4 *__restrict__ send,
                int32_t *__restrict__ meta, int32_t k_rt, int32_t hv, int32_t segs, int64_t units,
                int64_t rows) {
    const int k = K > 0 ? K : k_rt;
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;

    for (int64_t u = gwarp; u < units; u += nwarp) {
        const int64_t t = u / segs;
        const int seg = (int)(u - t * segs);

        int my_slot = -1;
        if (lane < k) {
            const int s = __ldg(slot + t * k + lane);
            my_slot = (s >= 0 && (int64_t)s < rows) ? s : -1;
            if (seg == 0 && my_slot >= 0) meta[my_slot] = (int32_t)(t * k + lane);
        }

        const int v0 = seg * (32 * kDispatchU) + lane;
        const uint4 *src = x + t * hv;
        uint4 val[kDispatchU];
#pragma unroll
        for (int q = 0; q < kDispatchU; ++q) {
            const int v = v0 + 32 * q;
            if (v < hv) val[q] = ld_stream_v4(src + v);
        }
        if (K > 0) {
#pragma unroll
            for (int j = 0; j < (K > 0 ? K : 1); ++j) {
                const int s = __shfl_sync(0xffffffffu, my_slot, j);
                if (s < 0) continue;
                uint4 *dst = send + (int64_t)s * hv;
#pragma unroll
                for (int q = 0; q < kDispatchU; ++q) {
                    const int v = v0 + 32 * q;
                    if (v < hv) st_v4(dst + v, val[q]);
                }
            }
        } else {
            for (int j = 0; j < k; ++j) {
                const int s = __shfl_sync(0xffffffffu, my_slot, j);
                if (s < 0) continue;
                uint4 *dst = send + (int64_t)s * hv;
#pragma unroll
                for (int q = 0; q < kDispatchU; ++q) {
                    const int v = v0 + 32 * q;
                    if (v < hv) st_v4(dst + v, val[q]);
                }
            }
        }
    }
}

template <int K>
cudaError_t launch_k(const ep_config &c, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send, int32_t *meta,
                     cudaStream_t s) {
    const int32_t hv = c.H / 8;
    const int32_t segs = (hv + 32 * kDispatchU - 1) / (32 * kDispatchU);
    const int64_t units = (int64_t)c.T * segs;
    const int64_t rows = (int64_t)c.T * c.k;
    int dev = 0;
    cudaGetDevice(&dev);
    const int occ = max_blocks_per_sm(reinterpret_cast<const void *>(dispatch_kernel<K>), kDispatchThreads, 0);
    const int64_t want = (units * 32 + kDispatchThreads - 1) / kDispatchThreads;
    const int64_t cap = (int64_t)sm_count(dev) * occ;
    const int64_t grid = want < cap ? want : cap;
    dispatch_kernel<K><<<(unsigned)grid, kDispatchThreads, 0, s>>>(
        reinterpret_cast<const uint4 *>(x), slot, reinterpret_cast<uint4 *>(send), meta, c.k, hv, segs, units,
        rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dispatch(const ep_config &c, const ep_bf16 *x, const int32_t *slot, ep_bf16 *send,
                            int32_t *meta, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    switch (c.k) {
        case 1: return launch_k<1>(c, x, slot, send, meta, s);
        case 2: return launch_k<2>(c, x, slot, send, meta, s);
        case 4: return launch_k<4>(c, x, slot, send, meta, s);
        case 6: return launch_k<6>(c, x, slot, send, meta, s);
        case 8: return launch_k<8>(c, x, slot, send, meta, s);
        default: return launch_k<0>(c, x, slot, send, meta, s);
    }
}

}  // namespace ep

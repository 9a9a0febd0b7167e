// combine.cu -- weighted top-k gather-reduce back to token order (ep_combine).
//
// out[t, h] = bf16_rne( fma(w[t,k-1], y[s_{k-1}, h], ... fma(w[t,0], y[s_0, h], 0) ) )
// with s_j = slot[t, j]: the k expert outputs of a token are brought back to
// it in the Combine step that follows the experts (UBEP article, opening
// section) and summed in fp32, one fused multiply-add per term, j = 0 .. k-1.
//
// Work unit = (token, segment of 32 * U 16-byte vectors). Each lane issues
// all k * U row loads of its unit before the first multiply-add, so a warp
// keeps k * U * 512 bytes in flight; y is read exactly once (streaming,
// non-allocating loads) and out written once.
//
// The kernel is launched as a programmatic dependent of whatever precedes it
// on the stream: its CTAs may become resident early, but each one waits on
// griddepcontrol.wait before its first memory access, so it sees every write
// of the previous kernel.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
    return *reinterpret_cast<const uint32_t *>(&p);
}

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4 &v) {
    acc[0] = __fmaf_rn(w, bf16_lo(v.x), acc[0]);
    acc[1] = __fmaf_rn(w, bf16_hi(v.x), acc[1]);
    acc[2] = __fmaf_rn(w, bf16_lo(v.y), acc[2]);
    acc[3] = __fmaf_rn(w, bf16_hi(v.y), acc[3]);
    acc[4] = __fmaf_rn(w, bf16_lo(v.z), acc[4]);
    acc[5] = __fmaf_rn(w, bf16_hi(v.z), acc[5]);
    acc[6] = __fmaf_rn(w, bf16_lo(v.w), acc[6]);
    acc[7] = __fmaf_rn(w, bf16_hi(v.w), acc[7]);
}

// K > 0: compile-time k (all K * U loads issued up front).
template <int K, int U>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ slot, const float *__restrict__ w,
               uint4 *__restrict__ out, int32_t hv, int32_t segs, int64_t units, int64_t rows) {
    grid_dependency_wait();  // launched as a programmatic dependent: nothing is touched before this
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;

    for (int64_t u = gwarp; u < units; u += nwarp) {
        const int64_t t = u / segs;
        const int seg = (int)(u - t * segs);
        int my_slot = -1;
        float my_w = 0.f;
        if (lane < K) {
            const int s = __ldg(slot + t * K + lane);
            my_slot = (s >= 0 && (int64_t)s < rows) ? s : -1;
            my_w = __ldg(w + t * K + lane);
        }
        int sj[K];
        float wj[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            sj[j] = __shfl_sync(0xffffffffu, my_slot, j);
            wj[j] = __shfl_sync(0xffffffffu, my_w, j);
        }
        const int v0 = seg * (32 * U) + lane;
        uint4 val[U][K];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int v = v0 + 32 * q;
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (v < hv && sj[j] >= 0) val[q][j] = ld_stream_v4(y + (int64_t)sj[j] * hv + v);
        }
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int v = v0 + 32 * q;
            if (v >= hv) continue;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (sj[j] >= 0) fma8(acc, wj[j], val[q][j]);
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            st_v4(out + t * hv + v, o);
        }
    }
}

// Runtime k (k > 8 or an uncommon k): loads and multiply-adds interleave per term.
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel_rt(const uint4 *__restrict__ y, const int32_t *__restrict__ slot, const float *__restrict__ w,
                  uint4 *__restrict__ out, int32_t k, int32_t hv, int32_t segs, int64_t units, int64_t rows) {
    grid_dependency_wait();
    constexpr int U = 2;
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t u = gwarp; u < units; u += nwarp) {
        const int64_t t = u / segs;
        const int seg = (int)(u - t * segs);
        int my_slot = -1;
        float my_w = 0.f;
        if (lane < k) {
            const int s = __ldg(slot + t * k + lane);
            my_slot = (s >= 0 && (int64_t)s < rows) ? s : -1;
            my_w = __ldg(w + t * k + lane);
        }
        const int v0 = seg * (32 * U) + lane;
        float acc[U][8];
#pragma unroll
        for (int q = 0; q < U; ++q)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
        for (int j = 0; j < k; ++j) {
            const int s = __shfl_sync(0xffffffffu, my_slot, j);
            const float wv = __shfl_sync(0xffffffffu, my_w, j);
            if (s < 0) continue;
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int v = v0 + 32 * q;
                if (v < hv) fma8(acc[q], wv, ld_stream_v4(y + (int64_t)s * hv + v));
            }
        }
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int v = v0 + 32 * q;
            if (v >= hv) continue;
            uint4 o;
            o.x = pack_bf16x2(acc[q][0], acc[q][1]);
            o.y = pack_bf16x2(acc[q][2], acc[q][3]);
            o.z = pack_bf16x2(acc[q][4], acc[q][5]);
            o.w = pack_bf16x2(acc[q][6], acc[q][7]);
            st_v4(out + t * hv + v, o);
        }
    }
}

int grid_for(const void *kern, int64_t units) {
    const int occ = max_blocks_per_sm(kern, kCombineThreads, 0);
    const int64_t want = (units * 32 + kCombineThreads - 1) / kCombineThreads;
    // 0 if the device query failed: the launch then reports the error
    const int64_t cap = (int64_t)current_device_sm_count() * occ;
    return (int)(want < cap ? want : cap);
}

template <int K, int U>
cudaError_t launch_ku(const ep_config &c, const ep_bf16 *y, const int32_t *slot, const float *w, ep_bf16 *out,
                      cudaStream_t s) {
    const int32_t hv = c.H / 8;
    const int32_t segs = (hv + 32 * U - 1) / (32 * U);
    const int64_t units = (int64_t)c.T * segs;
    const int grid = grid_for(reinterpret_cast<const void *>(combine_kernel<K, U>), units);
    return launch_dependent(combine_kernel<K, U>, dim3(grid), dim3(kCombineThreads), 0, s,
                            reinterpret_cast<const uint4 *>(y), slot, w, reinterpret_cast<uint4 *>(out), hv, segs,
                            units, (int64_t)c.T * c.k);
}

}  // namespace

cudaError_t launch_combine(const ep_config &c, const ep_bf16 *y, const int32_t *slot, const float *w,
                           ep_bf16 *out, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    switch (c.k) {
        case 1: return launch_ku<1, 4>(c, y, slot, w, out, s);
        case 2: return launch_ku<2, 4>(c, y, slot, w, out, s);
        case 4: return launch_ku<4, 2>(c, y, slot, w, out, s);
        case 6: return launch_ku<6, 1>(c, y, slot, w, out, s);
        case 8: return launch_ku<8, 1>(c, y, slot, w, out, s);
        default: break;
    }
    const int32_t hv = c.H / 8;
    const int32_t segs = (hv + 63) / 64;
    const int64_t units = (int64_t)c.T * segs;
    const int grid = grid_for(reinterpret_cast<const void *>(combine_kernel_rt), units);
    return launch_dependent(combine_kernel_rt, dim3(grid), dim3(kCombineThreads), 0, s,
                            reinterpret_cast<const uint4 *>(y), slot, w, reinterpret_cast<uint4 *>(out), c.k, hv,
                            segs, units, (int64_t)c.T * c.k);
}

}  // namespace ep

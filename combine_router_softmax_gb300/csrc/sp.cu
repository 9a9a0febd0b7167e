// sp.cu -- Data-as-Flag by Sentinel Polling (ep_sentinel_arm,
// ep_dispatch_expert_sp) and its bulk-synchronous counterpart
// (ep_expert_scale).
//
// The UBEP article ("Data-as-Flag", SP: Sentinel Polling) lets the receiver
// fill its destination buffer with a value no payload can take; the sender
// writes the raw payload with no flag or control message; the receiver polls
// until the value changes. Here sender and receiver are warps of one
// cooperative kernel (they wait on each other, so they may not be two
// launches, and every CTA must be resident):
//   * warp 0 of every CTA produces: it dispatches token rows into the send
//     buffer exactly as ep_dispatch does (TMA bulk loads of x rows, bulk
//     stores to the k slots);
//   * warps 1..7 consume: the rows of each worker of the chunk schedule are
//     spread over many warps; a lane polls each 16-byte vector until none of
//     its eight bf16 values is the sentinel 0xFFFF (a NaN bit pattern that
//     finite activations never take), applies the expert (a per-expert scale:
//     y = bf16_rne(float(send) * scale[e])) and writes the sentinel back,
//     which re-arms the buffer for the next call.
// A 32-bit word is written whole, so a vector with no sentinel half holds only
// new payload even while the bulk store that writes it is still in flight.
// Waits are bounded; a consumer that gives up sets ep_device_error bit 2 (4).
#include <cuda_bf16.h>

#include "ep_internal.cuh"
#include "flag_ops.cuh"

namespace ep {
namespace {

constexpr int kSpThreads = 256;          // warp 0 produces, warps 1..7 consume
constexpr int kSpConsumerWarps = kSpThreads / 32 - 1;
constexpr int kSpUnroll = 8;             // 16-byte polls in flight per consumer lane
constexpr bool kSpProbe = true;
constexpr int kSpStages = 2;             // x-row stages per producer
constexpr uint32_t kSpMaxPolls = 1u << 20;  // about a second of 64 ns sleeps and loads
constexpr uint32_t kSentinel2 = 0xFFFFFFFFu;  // two sentinel bf16 values

static __device__ int32_t g_sp_error;

__device__ __forceinline__ bool half_is_sentinel(uint32_t w) {
    return (w & 0xFFFFu) == 0xFFFFu || (w >> 16) == 0xFFFFu;
}

__device__ __forceinline__ bool has_sentinel(const uint4 &v) {
    return half_is_sentinel(v.x) || half_is_sentinel(v.y) || half_is_sentinel(v.z) || half_is_sentinel(v.w);
}

__device__ __forceinline__ uint32_t scale2(uint32_t w, float s) {
    const float lo = __uint_as_float(w << 16) * s;
    const float hi = __uint_as_float(w & 0xffff0000u) * s;
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

__device__ __forceinline__ uint4 scale8(const uint4 &v, float s) {
    uint4 o;
    o.x = scale2(v.x, s);
    o.y = scale2(v.y, s);
    o.z = scale2(v.z, s);
    o.w = scale2(v.w, s);
    return o;
}

__global__ void __launch_bounds__(256) sp_arm_kernel(uint4 *__restrict__ send, int64_t n_vec) {
    const uint4 s = make_uint4(kSentinel2, kSentinel2, kSentinel2, kSentinel2);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += stride) st_v4(send + i, s);
}

__global__ void __launch_bounds__(256) expert_scale_kernel(const uint4 *__restrict__ send,
                                                           const int32_t *__restrict__ expert_offset,
                                                           const float *__restrict__ scale, uint4 *__restrict__ y,
                                                           int32_t E, int64_t rows, int32_t hv) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t s = gw; s < rows; s += nw) {
        int lo = 0, hi = E;  // expert e with expert_offset[e] <= s < expert_offset[e + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if (__ldg(expert_offset + mid) <= s) lo = mid; else hi = mid;
        }
        const float sc = __ldg(scale + lo);
        for (int v = lane; v < hv; v += 32) st_v4(y + s * hv + v, scale8(ld_stream_v4(send + s * hv + v), sc));
    }
}

struct SpArgs {
    const char *x;
    const int32_t *slot;
    const int32_t *expert_offset;
    const float *scale;
    const ep_chunk *chunks;
    const int32_t *n_chunks;
    const int32_t *worker_begin;
    char *send;
    int32_t *meta;
    char *y;
    unsigned *row_flag;  // stop-and-wait only: [T k] epoch of each row's flag
    int32_t *err;
    int32_t T, H, E, k, W, row_pad;
    unsigned epoch;
};

// Expert that owns row s: the e with eoff[e] <= s < eoff[e + 1] (empty experts skipped).
__device__ __forceinline__ int owner_expert(const int32_t *eoff, int32_t E, int64_t s) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (eoff[mid] <= s) lo = mid; else hi = mid;
    }
    return lo;
}

// Every CTA: warp 0 produces (ep_dispatch's bulk path over tokens b, b + G,
// ...), warps 1..7 consume. Consumer warp g = 7 b + (warp - 1) serves worker
// g mod W; the nsub warps of one worker take the positions of that worker's
// concatenated chunk rows round-robin, so each worker's rows are polled by
// many warps at once and each warp walks its rows in the order they arrive
// (token order inside an expert's segment).
// kSW = false: Data-as-Flag by sentinel polling. kSW = true: the stop-and-wait
// baseline of the same section -- the producer lane waits until its row has
// landed, then releases the row's flag (the epoch); the consumer acquires the
// flag, then reads the row; nothing is re-armed.
template <bool kSW>
__global__ void __launch_bounds__(kSpThreads, 4) dispatch_expert_sp_kernel(SpArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int32_t row_bytes = a.H * 2;
    const int64_t rows = (int64_t)a.T * a.k;
    const size_t stage_bytes = (size_t)a.row_pad + 128;

    if (warp == 0) {
        // ---- producer
        uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kSpStages * stage_bytes);
        const int64_t first = blockIdx.x, G = gridDim.x;
        const int64_t n = first < a.T ? (a.T - first + G - 1) / G : 0;
        if (lane == 0) {
            for (int s = 0; s < kSpStages; ++s) mbar_init(&bar[s], 1);
            fence_mbar_init();
        }
        __syncwarp();
        auto load = [&](int s, int64_t t) {
            unsigned char *st = smem + (size_t)s * stage_bytes;
            mbar_arrive_expect_tx(&bar[s], (uint32_t)row_bytes + 4u * (uint32_t)a.k);
            bulk_g2s(st, a.x + t * row_bytes, (uint32_t)row_bytes, &bar[s]);
            bulk_g2s(st + a.row_pad, a.slot + t * a.k, 4u * (uint32_t)a.k, &bar[s]);
        };
        if (lane == 0)
            for (int s = 0; s < kSpStages && s < n; ++s) load(s, first + s * G);
        int64_t i = 0;
        bool ok = true;
        for (; i < n; ++i) {
            const int s = (int)(i % kSpStages);
            if (!mbar_wait_bounded(&bar[s], (uint32_t)((i / kSpStages) & 1), kSpMaxPolls)) {
                ok = false;
                break;
            }
            const int64_t t = first + i * G;
            const unsigned char *st = smem + (size_t)s * stage_bytes;
            if (lane < a.k) {
                const int sv = reinterpret_cast<const int32_t *>(st + a.row_pad)[lane];
                const bool valid = sv >= 0 && (int64_t)sv < rows;
                if (valid) {
                    bulk_s2g(a.send + (int64_t)sv * row_bytes, st, (uint32_t)row_bytes);
                    a.meta[sv] = (int32_t)(t * a.k + lane);
                }
                bulk_commit();
                if (kSW && valid) {
                    // the row has landed (writes done), is ordered before this
                    // thread's generic accesses, and only then is flagged
                    bulk_wait<0>();
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    st_release_u32(a.row_flag + sv, a.epoch);
                }
            }
            if (i >= 1 && i - 1 + kSpStages < n) {
                if (lane < a.k) bulk_wait_read<1>();
                __syncwarp();
                if (lane == 0) load((int)((i - 1) % kSpStages), first + (i - 1 + kSpStages) * G);
            }
        }
        if (!ok) {
            // Loads still in flight when the wait on token i gave up: token i,
            // and at i == 0 also the second initial load.
            if (lane == 0) atomicOr(a.err, kErrSpWait);
            const int64_t last = i == 0 ? (n < kSpStages ? n : kSpStages) : i + 1;
            for (int64_t j = i; j < last; ++j)
                mbar_wait_bounded(&bar[j % kSpStages], (uint32_t)((j / kSpStages) & 1), kSpMaxPolls);
        }
        if (lane < a.k) bulk_wait<0>();
        return;
    }

    // ---- consumers
    int32_t *s_eoff = reinterpret_cast<int32_t *>(smem + kSpStages * stage_bytes + 64);
    for (int e = threadIdx.x - 32; e <= a.E; e += kSpThreads - 32) s_eoff[e] = __ldg(a.expert_offset + e);
    asm volatile("bar.sync 1, %0;" ::"n"(kSpThreads - 32) : "memory");
    const int64_t g = (int64_t)blockIdx.x * kSpConsumerWarps + (warp - 1);
    const int64_t NG = (int64_t)gridDim.x * kSpConsumerWarps;
    const int w = (int)(g % a.W);
    const int64_t sub = g / a.W;
    const int64_t nsub = (NG - 1 - w) / a.W + 1;
    const int hv = a.H / 8;
    const uint4 *send4 = reinterpret_cast<const uint4 *>(a.send);
    uint4 *sendw = reinterpret_cast<uint4 *>(a.send);
    uint4 *y4 = reinterpret_cast<uint4 *>(a.y);
    const uint4 arm = make_uint4(kSentinel2, kSentinel2, kSentinel2, kSentinel2);

    // Tables that do not come from one ep_layout call on this cfg could name
    // chunks or rows outside the buffers: clamp to them and flag the error.
    const int nc = __ldg(a.n_chunks);
    int c0 = __ldg(a.worker_begin + w), c1 = __ldg(a.worker_begin + w + 1);
    bool ok = true;
    if (c0 < 0 || c1 > nc || c0 > c1) {
        ok = false;
        c1 = c0;
    }
    int64_t acc = 0;  // positions of the worker's rows before chunk ci
    for (int ci = c0; ci < c1 && ok; ++ci) {
        const int rb = __ldg(&a.chunks[ci].row_begin), rn = __ldg(&a.chunks[ci].row_count);
        if (rb < 0 || rn < 0 || (int64_t)rb + rn > rows) {
            ok = false;
            break;
        }
        int64_t p = acc + (((sub - acc) % nsub) + nsub) % nsub;  // first own position >= acc
        for (; p < acc + rn && ok; p += nsub) {
            const int64_t s = rb + (p - acc);
            const float sc = __ldg(a.scale + owner_expert(s_eoff, a.E, s));
            const uint4 *src = send4 + s * hv;
            if (kSW) {
                bool got = false;
                for (uint32_t polls = 0; polls <= kSpMaxPolls; ++polls) {
                    if (ld_acquire_u32(a.row_flag + s) == a.epoch) {
                        got = true;
                        break;
                    }
                    __nanosleep(64);
                }
                if (__all_sync(0xffffffffu, got)) {
                    for (int v0 = lane; v0 < hv; v0 += kSpUnroll * 32) {
                        uint4 val[kSpUnroll];
#pragma unroll
                        for (int u = 0; u < kSpUnroll; ++u)
                            if (v0 + 32 * u < hv) val[u] = ld_relaxed_v4(src + v0 + 32 * u);
#pragma unroll
                        for (int u = 0; u < kSpUnroll; ++u)
                            if (v0 + 32 * u < hv) st_v4(y4 + s * hv + v0 + 32 * u, scale8(val[u], sc));
                    }
                } else {
                    ok = false;
                }
                continue;
            }
            // Probe one vector (the row's last, which the bulk store writes
            // last or near it) until the payload shows: early polls then touch
            // one sector instead of pulling the whole sentinel row from HBM,
            // and the row is read once it sits in L2.
            if (kSpProbe) {
                uint32_t polls = 0;
                while (has_sentinel(ld_relaxed_v4(src + hv - 1)) && polls <= kSpMaxPolls) {
                    ++polls;
                    __nanosleep(128);
                }
            }
            for (int v0 = lane; v0 < hv; v0 += kSpUnroll * 32) {
                uint4 val[kSpUnroll];
#pragma unroll
                for (int u = 0; u < kSpUnroll; ++u)
                    if (v0 + 32 * u < hv) val[u] = ld_relaxed_v4(src + v0 + 32 * u);
#pragma unroll
                for (int u = 0; u < kSpUnroll; ++u) {
                    const int v = v0 + 32 * u;
                    if (v >= hv || !ok) continue;
                    uint32_t polls = 0;
                    while (has_sentinel(val[u])) {
                        if (++polls > kSpMaxPolls) break;
                        __nanosleep(64);
                        val[u] = ld_relaxed_v4(src + v);
                    }
                    if (polls > kSpMaxPolls) {
                        ok = false;
                        continue;
                    }
                    st_v4(y4 + s * hv + v, scale8(val[u], sc));
                    st_v4(sendw + s * hv + v, arm);
                }
            }
            ok = __all_sync(0xffffffffu, ok);
        }
        acc += rn;
    }
    if (!ok && lane == 0) atomicOr(a.err, kErrSpWait);
}

size_t sp_smem(int row_pad, int32_t E) {
    return (size_t)kSpStages * (row_pad + 128) + 64 + sizeof(int32_t) * ((size_t)E + 1);
}

}  // namespace

cudaError_t sp_error_word(int32_t **addr) {
    static std::atomic<int32_t *> cached[kMaxDevices_];  // zero-initialised: null
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices_) return cudaErrorInvalidDevice;
    if (!cached[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_sp_error);
        if (e != cudaSuccess) return e;
        cached[dev] = static_cast<int32_t *>(p);
    }
    *addr = cached[dev];
    return cudaSuccess;
}

cudaError_t launch_sentinel_arm(const ep_config &c, ep_bf16 *send, cudaStream_t s) {
    const int64_t n_vec = (int64_t)c.T * c.k * (c.H / 8);
    if (n_vec == 0) return cudaSuccess;
    int64_t grid = (n_vec + 255) / 256;
    const int64_t cap = (int64_t)current_device_sm_count() * 8;
    if (grid > cap) grid = cap;
    sp_arm_kernel<<<(unsigned)grid, 256, 0, s>>>(reinterpret_cast<uint4 *>(send), n_vec);
    return cudaGetLastError();
}

cudaError_t launch_expert_scale(const ep_config &c, const ep_bf16 *send, const int32_t *expert_offset,
                                const float *scale, ep_bf16 *y, cudaStream_t s) {
    const int64_t rows = (int64_t)c.T * c.k;
    if (rows == 0) return cudaSuccess;
    int64_t grid = (rows * 32 + 255) / 256;
    const int64_t cap = (int64_t)current_device_sm_count() * 8;
    if (grid > cap) grid = cap;
    expert_scale_kernel<<<(unsigned)grid, 256, 0, s>>>(reinterpret_cast<const uint4 *>(send), expert_offset, scale,
                                                       reinterpret_cast<uint4 *>(y), c.E, rows, c.H / 8);
    return cudaGetLastError();
}

namespace {

// EP_ERR_UNSUPPORTED-style refusal is signalled by cudaErrorNotSupported.

template <bool kSW>
cudaError_t launch_handoff(const ep_config &c, int32_t W, const ep_bf16 *x, const int32_t *slot,
                           const int32_t *expert_offset, const float *scale, const ep_chunk *chunks,
                           const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send, int32_t *meta,
                           ep_bf16 *y, unsigned *row_flag, unsigned epoch, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    const int32_t row_bytes = c.H * 2;
    if (c.k % 4 != 0 || row_bytes < 1024 || row_bytes > 48 * 1024) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> attr_set[kMaxDevices_];  // zero-initialised: false
    if (!attr_set[dev]) {
        if ((e = cudaFuncSetAttribute(dispatch_expert_sp_kernel<kSW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      110 * 1024)) != cudaSuccess)
            return e;
        attr_set[dev] = true;
    }
    const int row_pad = (row_bytes + 127) & ~127;
    const size_t smem = sp_smem(row_pad, c.E);
    const int occ =
        max_blocks_per_sm(reinterpret_cast<const void *>(dispatch_expert_sp_kernel<kSW>), kSpThreads, smem);
    const int64_t G = (int64_t)sm_count(dev) * occ;  // all co-resident: consumers wait on producers
    if (G < 1 || G * kSpConsumerWarps < W) return cudaErrorNotSupported;
    SpArgs a;
    a.x = reinterpret_cast<const char *>(x);
    a.slot = slot;
    a.expert_offset = expert_offset;
    a.scale = scale;
    a.chunks = chunks;
    a.n_chunks = n_chunks;
    a.worker_begin = worker_begin;
    a.send = reinterpret_cast<char *>(send);
    a.meta = meta;
    a.y = reinterpret_cast<char *>(y);
    a.row_flag = row_flag;
    a.epoch = epoch;
    if ((e = sp_error_word(&a.err)) != cudaSuccess) return e;
    a.T = c.T;
    a.H = c.H;
    a.E = c.E;
    a.k = c.k;
    a.W = W;
    a.row_pad = row_pad;
    void *args[] = {&a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(dispatch_expert_sp_kernel<kSW>),
                                       dim3((unsigned)G), dim3(kSpThreads), args, smem, s);
}

}  // namespace

cudaError_t launch_dispatch_expert_sp(const ep_config &c, int32_t W, const ep_bf16 *x, const int32_t *slot,
                                      const int32_t *expert_offset, const float *scale, const ep_chunk *chunks,
                                      const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send,
                                      int32_t *meta, ep_bf16 *y, cudaStream_t s) {
    return launch_handoff<false>(c, W, x, slot, expert_offset, scale, chunks, n_chunks, worker_begin, send, meta, y,
                                 nullptr, 0u, s);
}

cudaError_t launch_dispatch_expert_sw(const ep_config &c, int32_t W, const ep_bf16 *x, const int32_t *slot,
                                      const int32_t *expert_offset, const float *scale, const ep_chunk *chunks,
                                      const int32_t *n_chunks, const int32_t *worker_begin, ep_bf16 *send,
                                      int32_t *meta, ep_bf16 *y, unsigned *row_flag, unsigned epoch,
                                      cudaStream_t s) {
    return launch_handoff<true>(c, W, x, slot, expert_offset, scale, chunks, n_chunks, worker_begin, send, meta, y,
                                row_flag, epoch, s);
}

}  // namespace ep

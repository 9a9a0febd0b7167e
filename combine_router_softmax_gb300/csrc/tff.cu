// tff.cu -- Data-as-Flag by Token-Flag Fusion: the 512-byte block codec
// (ep_tff_encode, ep_tff_decode).
//
// The UBEP article ("Data-as-Flag", TFF) sends every token in 512-byte blocks
// of 32 bytes of synchronization metadata and 480 bytes of payload, written
// as one unit, so a receiver that sees the flag knows the payload is there.
// Block layout: [uint32 epoch, row, block, nbytes, 0, 0, 0, 0 | payload 480 B],
// payload zero beyond nbytes; row r of the send buffer takes
// ceil(row_bytes / 480) consecutive blocks.
//
// A GPU has no 512-byte atomic store, so the encoder orders the write instead:
// a warp takes 8 blocks at a time, stores their payload (8 vectors of 16 bytes
// per lane) and their metadata but the epoch word, and after a warp barrier
// lanes 0..7 release-store the 8 epochs. The decoder acquire-loads each
// block's epoch before it reads the rest, so a block whose flag matches is
// complete.
#include "ep_internal.cuh"
#include "flag_ops.cuh"

namespace ep {
namespace {

constexpr int kTffThreads = 256;
constexpr int kTffPayload = 480;
constexpr int kTffVecs = kTffPayload / 16;  // 30

// Blocks per warp step: 8 blocks = 240 payload vectors, 8 per lane in flight.
constexpr int kTffGroup = 8;

__global__ void __launch_bounds__(kTffThreads)
tff_encode_kernel(const uint4 *__restrict__ rows, uint4 *__restrict__ framed, int64_t n_rows, int32_t row_vecs,
                  int32_t nblk, unsigned epoch) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t total = n_rows * nblk;
    for (int64_t q0 = gw * kTffGroup; q0 < total; q0 += nw * kTffGroup) {
        uint4 val[kTffGroup];
#pragma unroll
        for (int u = 0; u < kTffGroup; ++u) {
            const int v = lane + 32 * u;  // vector v of the group: block v / 30, payload vector v % 30
            const int g = v / kTffVecs, j = v - g * kTffVecs;
            const int64_t q = q0 + g;
            val[u] = make_uint4(0, 0, 0, 0);
            if (g < kTffGroup && q < total) {
                const int64_t r = q / nblk;
                const int b = (int)(q - r * nblk);
                const int nv = row_vecs - b * kTffVecs < kTffVecs ? row_vecs - b * kTffVecs : kTffVecs;
                if (j < nv) val[u] = ld_stream_v4(rows + r * row_vecs + b * kTffVecs + j);
            }
        }
#pragma unroll
        for (int u = 0; u < kTffGroup; ++u) {
            const int v = lane + 32 * u;
            const int g = v / kTffVecs, j = v - g * kTffVecs;
            if (g < kTffGroup && q0 + g < total) st_v4(framed + (q0 + g) * 32 + 2 + j, val[u]);
        }
        // metadata of block q0 + lane (all but the epoch word), then the epochs
        const int64_t qm = q0 + lane;
        const bool mine = lane < kTffGroup && qm < total;
        if (mine) {
            const int64_t r = qm / nblk;
            const int b = (int)(qm - r * nblk);
            const int nv = row_vecs - b * kTffVecs < kTffVecs ? row_vecs - b * kTffVecs : kTffVecs;
            unsigned *m = reinterpret_cast<unsigned *>(framed + qm * 32);
            m[1] = (unsigned)r;
            m[2] = (unsigned)b;
            m[3] = (unsigned)(nv * 16);
            st_v4(framed + qm * 32 + 1, make_uint4(0, 0, 0, 0));
        }
        __syncwarp();  // the group's payload and metadata before any of its epochs
        if (mine) st_release_u32(reinterpret_cast<unsigned *>(framed + qm * 32), epoch);
    }
}

__global__ void __launch_bounds__(kTffThreads)
tff_decode_kernel(const uint4 *__restrict__ framed, uint4 *__restrict__ rows, int64_t n_rows, int32_t row_vecs,
                  int32_t nblk, unsigned epoch, unsigned *__restrict__ bad) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t total = n_rows * nblk;
    unsigned my_bad = 0;
    for (int64_t q0 = gw * kTffGroup; q0 < total; q0 += nw * kTffGroup) {
        // lane g < 8 checks block q0 + g: epoch (acquire) first, then the rest
        const int64_t qm = q0 + lane;
        bool good = false;
        if (lane < kTffGroup && qm < total) {
            const int64_t r = qm / nblk;
            const int b = (int)(qm - r * nblk);
            const int nv = row_vecs - b * kTffVecs < kTffVecs ? row_vecs - b * kTffVecs : kTffVecs;
            const unsigned *m = reinterpret_cast<const unsigned *>(framed + qm * 32);
            const unsigned e = ld_acquire_u32(m);
            good = e == epoch && m[1] == (unsigned)r && m[2] == (unsigned)b && m[3] == (unsigned)(nv * 16);
            my_bad += good ? 0u : 1u;
        }
        const unsigned ok = __ballot_sync(0xffffffffu, good);
        __syncwarp();  // orders every lane's payload loads after the acquires
        uint4 val[kTffGroup];
#pragma unroll
        for (int u = 0; u < kTffGroup; ++u) {
            const int v = lane + 32 * u;
            const int g = v / kTffVecs, j = v - g * kTffVecs;
            if (g < kTffGroup && ((ok >> g) & 1u)) val[u] = ld_relaxed_v4(framed + (q0 + g) * 32 + 2 + j);
        }
#pragma unroll
        for (int u = 0; u < kTffGroup; ++u) {
            const int v = lane + 32 * u;
            const int g = v / kTffVecs, j = v - g * kTffVecs;
            if (g < kTffGroup && ((ok >> g) & 1u)) {
                const int64_t q = q0 + g;
                const int64_t r = q / nblk;
                const int b = (int)(q - r * nblk);
                const int nv = row_vecs - b * kTffVecs < kTffVecs ? row_vecs - b * kTffVecs : kTffVecs;
                if (j < nv) st_v4(rows + r * row_vecs + b * kTffVecs + j, val[u]);
            }
        }
    }
    if (my_bad) atomicAdd(bad, my_bad);
}

int tff_grid(int64_t blocks) {
    const int64_t warps = (blocks + kTffGroup - 1) / kTffGroup;
    int64_t g = (warps * 32 + kTffThreads - 1) / kTffThreads;
    const int64_t cap = (int64_t)current_device_sm_count() * 8;
    if (g > cap) g = cap;
    return (int)(g > 0 ? g : 1);
}

}  // namespace

int64_t tff_blocks_per_row(const ep_config &c) { return ((int64_t)c.H * 2 + kTffPayload - 1) / kTffPayload; }

cudaError_t launch_tff_encode(const ep_config &c, const ep_bf16 *rows, void *framed, unsigned epoch,
                              cudaStream_t s) {
    const int64_t n_rows = (int64_t)c.T * c.k;
    const int32_t nblk = (int32_t)tff_blocks_per_row(c);
    if (n_rows == 0) return cudaSuccess;
    tff_encode_kernel<<<tff_grid(n_rows * nblk), kTffThreads, 0, s>>>(
        reinterpret_cast<const uint4 *>(rows), static_cast<uint4 *>(framed), n_rows, c.H / 8, nblk, epoch);
    return cudaGetLastError();
}

cudaError_t launch_tff_decode(const ep_config &c, const void *framed, unsigned epoch, ep_bf16 *rows,
                              unsigned *bad, cudaStream_t s) {
    const int64_t n_rows = (int64_t)c.T * c.k;
    const int32_t nblk = (int32_t)tff_blocks_per_row(c);
    if (n_rows == 0) return cudaSuccess;
    tff_decode_kernel<<<tff_grid(n_rows * nblk), kTffThreads, 0, s>>>(
        static_cast<const uint4 *>(framed), reinterpret_cast<uint4 *>(rows), n_rows, c.H / 8, nblk, epoch, bad);
    return cudaGetLastError();
}

}  // namespace ep

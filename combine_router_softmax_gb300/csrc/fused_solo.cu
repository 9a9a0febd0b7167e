// fused_solo.cu -- the split form of the small-batch dispatch kernel with a
// single tile (metadata) CTA, up to 4 tokens (fused_kernel.cuh), compiled in a
// module of its own: beside the other instances it slowed those down.
#include "fused_kernel.cuh"

namespace ep {

const void *fused_solo_kernel(int32_t E) {
    const int vpl = (E + 31) / 32;
    if (vpl <= 1) return reinterpret_cast<const void *>(dispatch_fused_kernel<1, true, true>);
    if (vpl <= 2) return reinterpret_cast<const void *>(dispatch_fused_kernel<2, true, true>);
    if (vpl <= 4) return reinterpret_cast<const void *>(dispatch_fused_kernel<4, true, true>);
    if (vpl <= 8) return reinterpret_cast<const void *>(dispatch_fused_kernel<8, true, true>);
    if (vpl <= 16) return reinterpret_cast<const void *>(dispatch_fused_kernel<16, true, true>);
    return reinterpret_cast<const void *>(dispatch_fused_kernel<32, true, true>);
}

}  // namespace ep

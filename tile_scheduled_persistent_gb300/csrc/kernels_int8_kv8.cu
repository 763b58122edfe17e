// Kernel instances with INT8 weights and the INT8 KV cache (smoothed keys,
// every attention chunk on the tensor cores).
#include "megakernel.cuh"

namespace tiles {

const void *megakernel_int8_kv8(int d, int G) {
#define TILES_KERNEL_CASE(DD, GG) \
    if (d == DD && G == GG) return (const void *)tiles_megakernel<DD, GG, true, 2>;
    TILES_KERNEL_CASE(64, 1) TILES_KERNEL_CASE(64, 2) TILES_KERNEL_CASE(64, 4) TILES_KERNEL_CASE(64, 8)
    TILES_KERNEL_CASE(128, 1) TILES_KERNEL_CASE(128, 2) TILES_KERNEL_CASE(128, 4) TILES_KERNEL_CASE(128, 8)
#undef TILES_KERNEL_CASE
    return nullptr;
}

}  // namespace tiles

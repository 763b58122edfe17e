// Kernel instances with INT8 weights: one per (head_dim, q heads per KV head),
// without the one-warp-per-chunk attention form.
#include "megakernel.cuh"

namespace tiles {

const void *megakernel_int8(int d, int G) {
#define TILES_KERNEL_CASE(DD, GG) \
    if (d == DD && G == GG) return (const void *)tiles_megakernel<DD, GG, true, 0>;
    TILES_KERNEL_CASE(64, 1) TILES_KERNEL_CASE(64, 2) TILES_KERNEL_CASE(64, 4) TILES_KERNEL_CASE(64, 8)
    TILES_KERNEL_CASE(128, 1) TILES_KERNEL_CASE(128, 2) TILES_KERNEL_CASE(128, 4) TILES_KERNEL_CASE(128, 8)
#undef TILES_KERNEL_CASE
    return nullptr;
}

}  // namespace tiles

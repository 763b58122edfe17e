// Kernel instances with BF16 weights and the one-warp-per-chunk attention
// form, for plans whose attention splits can hold 8 or more KV chunks (long
// contexts).
#include "megakernel.cuh"

namespace tiles {

const void *megakernel_bf16_mma(int d, int G) {
#define TILES_KERNEL_CASE(DD, GG) \
    if (d == DD && G == GG) return (const void *)tiles_megakernel<DD, GG, false, 1>;
    TILES_KERNEL_CASE(64, 1) TILES_KERNEL_CASE(64, 2) TILES_KERNEL_CASE(64, 4) TILES_KERNEL_CASE(64, 8)
    TILES_KERNEL_CASE(128, 1) TILES_KERNEL_CASE(128, 2) TILES_KERNEL_CASE(128, 4) TILES_KERNEL_CASE(128, 8)
#undef TILES_KERNEL_CASE
    return nullptr;
}

}  // namespace tiles

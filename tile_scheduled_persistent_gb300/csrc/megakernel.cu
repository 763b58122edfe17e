// Launchers of the persistent decode kernel and the measurement kernels (the
// device code is in megakernel.cuh; kernels_bf16.cu and kernels_int8.cu hold
// the kernel instances, compiled in parallel).
#include "megakernel.cuh"

namespace tiles {

const void *megakernel_bf16(int d, int G);      // kernels_bf16.cu
const void *megakernel_bf16_mma(int d, int G);  // kernels_bf16_mma.cu
const void *megakernel_int8(int d, int G);      // kernels_int8.cu
const void *megakernel_int8_mma(int d, int G);  // kernels_int8_mma.cu

static const void *megakernel_for(int d, int G, int wbytes, int mma) {
    if (wbytes == 1) return mma ? megakernel_int8_mma(d, G) : megakernel_int8(d, G);
    return mma ? megakernel_bf16_mma(d, G) : megakernel_bf16(d, G);
}

// ------------------------------------------------------------------ launchers
cudaError_t megakernel_configure(int d, int G, int wbytes, int mma, int smem_bytes) {
    const void *k = megakernel_for(d, G, wbytes, mma);
    if (!k) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t megakernel_occupancy(int d, int G, int wbytes, int mma, int smem_bytes, int *blocks_per_sm) {
    const void *k = megakernel_for(d, G, wbytes, mma);
    if (!k) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, kThreads, smem_bytes);
}

cudaError_t megakernel_launch(const KernelParams &p, int n_ctas, int smem_bytes, cudaStream_t st) {
    const void *k = megakernel_for(p.g.d, p.g.G, p.g.wbytes, p.g.attn_mma);
    if (!k) return cudaErrorInvalidValue;
    void *args[] = {const_cast<KernelParams *>(&p)};
    return cudaLaunchCooperativeKernel(k, dim3(n_ctas), dim3(kThreads), args, (size_t)smem_bytes, st);
}

// ------------------------------------------------------------------ INT8 weights
// Weight-only INT8 per output row ("History and roadmap", "Milestones":
// weight-only INT8 linear layers; the plainest scheme, as the pages give
// none): scale = max |w| / 127 and code = w / scale rounded to nearest even,
// clamped to +-127, all in FP32 (an all-zero row: scale 0, codes 0). One CTA
// per row. Source row r goes to destination row r * row_step + row0 (codes
// and scale), which writes the plan's packed layouts directly. With offset
// 128 a code is stored as the byte q + 128 (the plan's form: the GEMV then
// needs no sign flip); with 0, as the int8 q.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t *__restrict__ src, int rows,
                                                            int cols, uint8_t *__restrict__ dst,
                                                            float *__restrict__ scale, int row_step,
                                                            int row0, int offset) {
    const int r = blockIdx.x;
    if (r >= rows) return;
    const uint16_t *w = src + (size_t)r * cols;
    __shared__ float red[8];
    float amax = 0.f;
    for (int j = threadIdx.x; j < cols; j += blockDim.x) amax = fmaxf(amax, fabsf(bf2f(w[j])));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    const float sc = __fdiv_rn(amax, 127.0f);
    const size_t orow = (size_t)r * row_step + row0;
    if (threadIdx.x == 0) scale[orow] = sc;
    uint8_t *q = dst + orow * cols;
    for (int j = threadIdx.x; j < cols; j += blockDim.x) {
        float qf = sc > 0.f ? rintf(__fdiv_rn(bf2f(w[j]), sc)) : 0.f;
        qf = fminf(fmaxf(qf, -127.f), 127.f);
        q[j] = (uint8_t)((int)qf + offset);
    }
}

cudaError_t quantize_rows_launch(const void *src, int rows, int cols, void *dst, float *scale,
                                 int row_step, int row0, int offset, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    quantize_rows_kernel<<<rows, 256, 0, st>>>(reinterpret_cast<const uint16_t *>(src), rows, cols,
                                               reinterpret_cast<uint8_t *>(dst), scale, row_step, row0,
                                               offset);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ measurement kernels
__global__ void __launch_bounds__(512) copy_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                   size_t n) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
              d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

cudaError_t copy_launch(void *dst, const void *src, size_t bytes, int n_ctas, cudaStream_t st) {
    copy_kernel<<<n_ctas, 512, 0, st>>>(reinterpret_cast<uint4 *>(dst),
                                        reinterpret_cast<const uint4 *>(src), bytes / 16);
    return cudaGetLastError();
}

// rounds of grid barriers; CTA 0 reports the elapsed global-timer nanoseconds
__global__ void barrier_kernel(uint32_t *ctr, int rounds, unsigned long long *elapsed,
                               uint32_t *status, unsigned long long timeout_ns) {
    __shared__ int abort_flag;
    const uint32_t n = gridDim.x;
    unsigned long long t0 = 0;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) t0 = global_timer();
    for (int r = 0; r < rounds; ++r) {
        __syncthreads();
        if (threadIdx.x == 0) {
            red_release_add(ctr, 1u);
            const uint32_t target = n * (uint32_t)(r + 1);
            unsigned long long ts = global_timer();
            while (ld_relaxed(ctr) < target) {
                if (global_timer() - ts > timeout_ns) {
                    atomicOr(status, kDevTimeout);
                    abort_flag = 1;
                    break;
                }
            }
            fence_acquire_gpu();
        }
        __syncthreads();
        if (abort_flag) return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *elapsed = global_timer() - t0;
}

cudaError_t barrier_launch(uint32_t *ctr, int rounds, unsigned long long *elapsed, uint32_t *status,
                           int n_ctas, cudaStream_t st) {
    unsigned long long timeout = 2000000000ull;
    void *args[] = {&ctr, &rounds, &elapsed, &status, &timeout};
    return cudaLaunchCooperativeKernel((const void *)barrier_kernel, dim3(n_ctas), dim3(128), args, 0,
                                       st);
}

}  // namespace tiles

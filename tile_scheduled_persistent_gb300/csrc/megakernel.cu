// Launchers of the persistent decode kernel and the measurement kernels (the
// device code is in megakernel.cuh; kernels_bf16.cu and kernels_int8.cu hold
// the kernel instances, compiled in parallel).
#include "megakernel.cuh"

namespace tiles {

const void *megakernel_bf16(int d, int G);      // kernels_bf16.cu
const void *megakernel_bf16_mma(int d, int G);  // kernels_bf16_mma.cu
const void *megakernel_int8(int d, int G);      // kernels_int8.cu
const void *megakernel_int8_mma(int d, int G);  // kernels_int8_mma.cu
const void *megakernel_bf16_kv8(int d, int G);  // kernels_bf16_kv8.cu
const void *megakernel_int8_kv8(int d, int G);  // kernels_int8_kv8.cu

// ak: attention kind (attn_kind of the plan's geometry)
static const void *megakernel_for(int d, int G, int wbytes, int ak) {
    if (wbytes == 1) return ak == 2 ? megakernel_int8_kv8(d, G) : ak ? megakernel_int8_mma(d, G) : megakernel_int8(d, G);
    return ak == 2 ? megakernel_bf16_kv8(d, G) : ak ? megakernel_bf16_mma(d, G) : megakernel_bf16(d, G);
}

// ------------------------------------------------------------------ launchers
cudaError_t megakernel_configure(int d, int G, int wbytes, int ak, int smem_bytes) {
    const void *k = megakernel_for(d, G, wbytes, ak);
    if (!k) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t megakernel_occupancy(int d, int G, int wbytes, int ak, int smem_bytes, int *blocks_per_sm) {
    const void *k = megakernel_for(d, G, wbytes, ak);
    if (!k) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, kThreads, smem_bytes);
}

cudaError_t megakernel_launch(const KernelParams &p, int n_ctas, int smem_bytes, cudaStream_t st) {
    const void *k = megakernel_for(p.g.d, p.g.G, p.g.wbytes, attn_kind(p.g));
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

// ------------------------------------------------------------------ INT8 KV cache
// The INT8 cache of prefilled positions ("History and roadmap", M8: INT8 KV
// cache with smoothed keys; the plainest scheme, as the pages give none).
// Key shift of each (layer, KV head): mu_j = sum_t K[t][j] / n in FP64, in
// position order (one thread per channel), rounded to FP32; 0 when n = 0.
__global__ void kv8_mean_kernel(const uint16_t *__restrict__ K, int max_pos, int d, int n,
                                float *__restrict__ mu) {
    const int z = blockIdx.x, j = threadIdx.x;
    if (j >= d) return;
    const uint16_t *k = K + (size_t)z * max_pos * d + j;
    double acc = 0.0;
    for (int t = 0; t < n; ++t) acc += (double)bf2f(k[(size_t)t * d]);
    mu[(size_t)z * d + j] = n > 0 ? (float)(acc / n) : 0.f;
}

// Rows [t0, t0 + 64) of head z: one warp per row, keys minus mu and values
// quantized (s = max |x| / 127, codes x / s rounded to nearest even, clamped
// to +-127, FP32). Key codes go out row by row; value codes are staged and
// written transposed ([d][MP]) in 64-byte runs.
template <int D>
__global__ void __launch_bounds__(256) kv8_quant_kernel(const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
                                                        int max_pos, int mp, int n, const float *__restrict__ mu,
                                                        int8_t *__restrict__ kq, float *__restrict__ ks,
                                                        int8_t *__restrict__ vq, float *__restrict__ vs) {
    constexpr int E = D / 32;
    __shared__ int8_t vt[D][64];
    const int z = blockIdx.y, t0 = blockIdx.x * 64, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const float *m = mu + (size_t)z * D;
    for (int tt = w; tt < 64; tt += 8) {
        const int t = t0 + tt;
        if (t >= n) break;
        const size_t row = (size_t)z * max_pos + t;
        for (int kv = 0; kv < 2; ++kv) {
            float x[E], amax = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int j = lane + 32 * e;
                x[e] = kv == 0 ? __fsub_rn(bf2f(K[row * D + j]), m[j]) : bf2f(V[row * D + j]);
                amax = fmaxf(amax, fabsf(x[e]));
            }
            amax = warp_max(amax);
            const float sc = __fdiv_rn(amax, 127.0f);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                float qf = sc > 0.f ? rintf(__fdiv_rn(x[e], sc)) : 0.f;
                const int8_t c = (int8_t)fminf(fmaxf(qf, -127.f), 127.f);
                if (kv == 0)
                    kq[((size_t)z * mp + t) * D + lane + 32 * e] = c;
                else
                    vt[lane + 32 * e][tt] = c;
            }
            if (lane == 0) (kv == 0 ? ks : vs)[(size_t)z * mp + t] = sc;
        }
    }
    __syncthreads();
    const int nt = n - t0 < 64 ? n - t0 : 64;
    for (int i = threadIdx.x; i < D * 64; i += 256) {
        const int j = i / 64, tt = i % 64;
        if (tt < nt) vq[((size_t)z * D + j) * mp + t0 + tt] = vt[j][tt];
    }
}

cudaError_t kv8_from_bf16_launch(const uint16_t *k, const uint16_t *v, int Z, int max_pos, int mp, int d,
                                 int n_pos, int8_t *kq, float *ks, float *mu, int8_t *vq, float *vs,
                                 cudaStream_t st) {
    kv8_mean_kernel<<<Z, d, 0, st>>>(k, max_pos, d, n_pos, mu);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || n_pos == 0) return e;
    const dim3 grid((unsigned)((n_pos + 63) / 64), (unsigned)Z);
    if (d == 64)
        kv8_quant_kernel<64><<<grid, 256, 0, st>>>(k, v, max_pos, mp, n_pos, mu, kq, ks, vq, vs);
    else
        kv8_quant_kernel<128><<<grid, 256, 0, st>>>(k, v, max_pos, mp, n_pos, mu, kq, ks, vq, vs);
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

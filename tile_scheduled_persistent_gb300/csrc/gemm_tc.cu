// The projections of the multi-token pass on the fifth-generation tensor
// cores: C[z][t][m] = sum over k in split z of W[m][k] X[t][k], BF16 operands,
// FP32 accumulation ("History and roadmap", "Where it stands": prefill of a
// 512-token prompt, and "M8 so far": 16-token verify steps; with T tokens
// every weight row is used T times, so the projections are dense
// contractions).
//
// One CTA computes a tile of 128 weight rows (the MMA's M) against every token
// of the pass (N = T rounded up to 16, at most 256) over its split of K:
//   - warp 0, one lane: TMA copies of 64-element K slices of the weight tile
//     and of the activation tile (128-byte swizzle, K-major) into a ring of
//     shared-memory stages, each completing on its "full" mbarrier;
//   - warp 1, one lane: per stage four tcgen05.mma (M 128, N, K 16) with the
//     accumulator in tensor memory, then tcgen05.commit to the stage's
//     "empty" mbarrier (the copy of a later slice may reuse it) and, after
//     the last stage, to the "done" mbarrier;
//   - all four warps: tensor memory -> registers (tcgen05.ld, warp w owns
//     rows 32 w .. 32 w + 31) -> C, one token column at a time, so each warp
//     writes 32 consecutive m of one token. For the gate/up projection with
//     one split, the epilogue applies the SwiGLU instead: rows come in
//     (gate, up) pairs, so lane 2i pairs its gate sum with lane 2i + 1's up
//     sum and writes a[t][m / 2] = R(silu(g) u) in BF16, with the arithmetic
//     of the separate SwiGLU kernel (the split sum 0 + g first).
// Every wait is bounded: past the limit the CTA records a timeout in the
// status word, lets what it issued finish (bounded too), frees its tensor
// memory and returns.
#include <cuda_runtime.h>

#include <algorithm>

#include "megakernel.cuh"
#include "plan_internal.h"

namespace tiles {
namespace fwd {

// kTcM (plan_internal.h): weight rows per CTA, the MMA's M
constexpr int kTcBK = 64;        // K elements per stage: one 128-byte swizzle row
constexpr int kTcThreads = 128;
constexpr int kTcMaxStages = 12;
constexpr int kTcABytes = kTcM * kTcBK * 2;  // 16 KB weight slice per stage

struct TcCtl {
    uint64_t full[kTcMaxStages], empty[kTcMaxStages], done;
    uint32_t tmem_base, abort;
};

// Shared-memory matrix descriptor of a K-major tile written by the tiled copy
// with the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart
// (stride byte offset), start address in 16-byte units, descriptor version 1,
// layout code 2 (128-byte swizzle). The leading byte offset is unused for
// this layout and set to one unit.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: FP32 accumulator (bits 4-5 = 1), BF16
// A and B (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N / 8 at
// bit 17, M / 16 at bit 24.
__host__ __device__ __forceinline__ uint32_t tc_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive FP32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait on an mbarrier phase; false once the limit passed or another
// role of the CTA gave up.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, unsigned long long deadline,
                                        volatile uint32_t *abort) {
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 63u && (*abort || global_timer() > deadline)) return false;
    }
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ TensorMap mw, const __grid_constant__ TensorMap mx, int M, int T, int K,
                   int kps, int n_tile, int stages, float *__restrict__ C, uint16_t *__restrict__ act,
                   uint32_t *status, unsigned long long timeout_ns) {
    extern __shared__ __align__(1024) uint8_t tsm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t b_bytes = (uint32_t)n_tile * 128u;
    uint8_t *sa = tsm;                                   // [stages][128 rows][128 B]
    uint8_t *sb = tsm + (size_t)stages * kTcABytes;      // [stages][n_tile rows][128 B]
    TcCtl *ctl = reinterpret_cast<TcCtl *>(sb + (size_t)stages * b_bytes);
    // the swizzle atoms assume 1024-byte aligned tiles; never run otherwise
    if (smem_u32(tsm) & 1023u) {
        if (tid == 0) atomicOr(status, kDevBounds);
        return;
    }
    const int m0 = blockIdx.x * kTcM;
    const int k0 = blockIdx.z * kps, k1 = min(K, k0 + kps);
    const int nk = (k1 - k0 + kTcBK - 1) / kTcBK;
    const uint32_t ncols = n_tile <= 32 ? 32u : n_tile <= 64 ? 64u : n_tile <= 128 ? 128u : 256u;
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->done, 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ctl->tmem_base)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile uint32_t *abort = &ctl->abort;
    const unsigned long long deadline = global_timer() + timeout_ns;
    bool mma_issued = false;

    if (warp == 0 && lane == 0) {
        // producer: weight slice (x = k, y = m0) and activation slice (x = k, y = 0)
        for (int kc = 0; kc < nk; ++kc) {
            const int s = kc % stages, r = kc / stages;
            if (kc >= stages && !tc_wait(&ctl->empty[s], (uint32_t)(r - 1) & 1u, deadline, abort)) {
                *abort = 1;
                break;
            }
            mbar_expect_tx(&ctl->full[s], (uint32_t)kTcABytes + b_bytes);
            tensor_g2s_2d(sa + (size_t)s * kTcABytes, &mw, k0 + kc * kTcBK, m0, &ctl->full[s]);
            tensor_g2s_2d(sb + (size_t)s * b_bytes, &mx, k0 + kc * kTcBK, 0, &ctl->full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        const uint32_t idesc = tc_idesc(kTcM, n_tile);
        for (int kc = 0; kc < nk; ++kc) {
            const int s = kc % stages, r = kc / stages;
            if (!tc_wait(&ctl->full[s], (uint32_t)r & 1u, deadline, abort)) {
                *abort = 1;
                break;
            }
            tc_fence_after();
            const uint64_t ad = tc_desc_sw128(smem_u32(sa + (size_t)s * kTcABytes));
            const uint64_t bd = tc_desc_sw128(smem_u32(sb + (size_t)s * b_bytes));
#pragma unroll
            for (int ks = 0; ks < kTcBK / 16; ++ks)  // 16 elements = 32 bytes = 2 descriptor units
                tc_mma(tmem, ad + 2u * ks, bd + 2u * ks, idesc, (kc | ks) != 0 ? 1u : 0u);
            tc_commit(&ctl->empty[s]);
            mma_issued = true;
        }
        // the accumulator is complete when every MMA issued so far is
        tc_commit(&ctl->done);
    }
    __syncwarp();
    // epilogue: every warp waits for the accumulator
    const bool ok = tc_wait(&ctl->done, 0u, deadline, abort) && !*abort;
    tc_fence_after();
    if (ok) {
        const int m = m0 + 32 * warp + lane;
        float *Cz = C + (size_t)blockIdx.z * T * M;
        const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
        for (int c0 = 0; c0 < n_tile; c0 += 16) {
            float v[16];
            if (nk > 0) {
                tc_ld16(trow + (uint32_t)c0, v);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.f;  // an empty split adds zeros
            }
            if constexpr (SWIGLU) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = c0 + j;
                    const float up = __shfl_down_sync(0xFFFFFFFFu, v[j], 1);
                    if (!(lane & 1) && m < M && t < T) {
                        const float gt = __fadd_rn(0.f, v[j]), u = __fadd_rn(0.f, up);
                        const float silu = __fdiv_rn(gt, __fadd_rn(1.0f, expf(-gt)));
                        act[(size_t)t * (M / 2) + m / 2] = f2bf(__fmul_rn(silu, u));
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = c0 + j;
                    if (m < M && t < T) Cz[(size_t)t * M + m] = v[j];
                }
            }
        }
    } else if (!ok && tid == 0) {
        atomicOr(status, kDevTimeout);
    }
    if (!ok && warp == 1 && lane == 0 && mma_issued) {
        // the MMAs issued depend on nothing but shared memory: let them finish
        // before the tensor memory goes (bounded as well)
        const unsigned long long d2 = global_timer() + timeout_ns;
        volatile uint32_t never = 0;
        tc_wait(&ctl->done, 0u, d2, &never);
    }
    if (!ok && warp == 0 && lane == 0) {
        // and the copies in flight into the stages, likewise
        const unsigned long long d2 = global_timer() + timeout_ns;
        volatile uint32_t never = 0;
        for (int kc = nk - stages > 0 ? nk - stages : 0; kc < nk; ++kc)
            tc_wait(&ctl->full[kc % stages], (uint32_t)(kc / stages) & 1u, d2, &never);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

// ------------------------------------------------------------------ host side
TcShape tc_shape(int M, int T, int K, int sms, int max_sk) {
    TcShape s;
    s.n_tile = (T + 15) / 16 * 16;
    s.mt = (M + kTcM - 1) / kTcM;
    const int nkc = (K + kTcBK - 1) / kTcBK;
    // splits: as many as keep the grid within one wave (one CTA per SM: a
    // second wave of a few CTAs would double the projection's time)
    int sk = std::max(1, std::min(nkc, sms / s.mt));
    sk = std::max(1, std::min(sk, max_sk));
    s.kps = ((nkc + sk - 1) / sk) * kTcBK;
    s.sk = (K + s.kps - 1) / s.kps;
    const int stage = kTcABytes + s.n_tile * 128;
    s.stages = std::min(kTcMaxStages, (200 * 1024) / stage);  // 4 stages at 256 tokens, 11 at 16
    // at least 116 KB of shared memory: one CTA per SM, so no CTA ever waits for tensor memory
    s.smem = std::max((size_t)116 * 1024, (size_t)s.stages * stage + sizeof(TcCtl));
    return s;
}

cudaError_t gemm_tc_configure() {
    const int bytes = 200 * 1024 + (int)sizeof(TcCtl) + 1024;
    cudaError_t e = cudaFuncSetAttribute((const void *)gemm_tc_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute((const void *)gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bytes);
    return e;
}

cudaError_t gemm_tc_launch(const TensorMap &mw, const TensorMap &mx, const TcShape &s, int M, int T, int K,
                           float *C, uint16_t *act, uint32_t *status, unsigned long long timeout_ns,
                           cudaStream_t st) {
    if (act && (s.sk != 1 || M % 2)) return cudaErrorInvalidValue;
    if (act)
        gemm_tc_kernel<true><<<dim3(s.mt, 1, s.sk), kTcThreads, s.smem, st>>>(mw, mx, M, T, K, s.kps, s.n_tile,
                                                                              s.stages, C, act, status, timeout_ns);
    else
        gemm_tc_kernel<false><<<dim3(s.mt, 1, s.sk), kTcThreads, s.smem, st>>>(mw, mx, M, T, K, s.kps, s.n_tile,
                                                                               s.stages, C, act, status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace fwd
}  // namespace tiles

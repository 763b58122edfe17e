// Multi-token forward pass: T tokens at positions P0 .. P0 + T - 1 through the
// whole model in one pass, every layer processing all of them at once. It
// computes exactly what T decode steps with those input tokens compute (each
// token attends to every cached position up to its own, the K/V rows of the
// earlier tokens of the pass included), and it is the substrate of two rows of
// the roadmap: a verify step over k draft tokens ("History and roadmap", "M8
// so far": 16-token verify steps on the split-KV decode kernels) and batched
// prompt prefill ("Tiles", "Scope and code release": prefill still runs one
// token per step; "History and roadmap", "Where it stands": prefill of a
// 512-token prompt).
//
// With T columns every weight row is used T times, so the projections are
// dense contractions: they run on the fifth-generation tensor cores
// (gemm_tc.cu: TMA-staged operands, tcgen05.mma with the accumulator in
// tensor memory, split along K across CTAs when the output alone would not
// fill the GPU, and the split partial sums added in a fixed order by the
// kernel that consumes them). Attention is a causal,
// split-KV, multi-query kernel on the same MMAs (scores in FP32, the softmax
// weights split into a BF16 high part and a BF16 remainder for the p V
// product, as in the decode kernel), followed by an ordered combine. Norms,
// RoPE, the KV write, SwiGLU, residual adds and the greedy choice are fused
// into small per-token kernels. Rounding points are the decode kernel's: the
// residual stream, every GEMM input, q and the cached K/V are BF16.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "megakernel.cuh"
#include "plan_internal.h"

namespace tiles {
namespace fwd {

constexpr int kMaxTokens = 256;  // tokens per pass

// c += A B, A 16x16 (row), B 16x8 (col), BF16 in, FP32 accumulate. Fragments
// for lane (g, t) = (lane / 4, lane % 4): a = {(g, 2t..2t+1), (g+8, 2t..),
// (g, 2t+8..), (g+8, 2t+8..)}, b = {(k 2t..2t+1, n g), (k 2t+8.., n g)},
// c = {(g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)}.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9},"
        " {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

// ------------------------------------------------------------------ per-token kernels
// Block-wide sum of NT threads in a fixed order (warp trees, then warps in order).
template <int NT>
__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) t += red[w];
    __syncthreads();
    return t;
}
__device__ __forceinline__ float block_sum256(float v, float *red) { return block_sum<256>(v, red); }

// h[t] = R(rmsnorm(x[t]) * gain), x[t] a bf16 row of n; r = 1 / sqrt(mean(x^2) + eps)
__device__ __forceinline__ void norm_row(const uint16_t *x, const uint16_t *gain, int n, float eps, uint16_t *h,
                                         float *red) {
    float ss = 0.f;
    for (int j = threadIdx.x; j < n; j += 256) {
        const float v = bf2f(x[j]);
        ss = fmaf(v, v, ss);
    }
    const float tot = block_sum256(ss, red);
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)n), eps)));
    for (int j = threadIdx.x; j < n; j += 256)
        h[j] = f2bf(__fmul_rn(__fmul_rn(bf2f(x[j]), r), bf2f(gain[j])));
}

// x[t] = E[token t]; h[t] = R(rmsnorm(x[t]) * gain). A token id out of range
// is recorded in the status word (and row 0 used).
__global__ void __launch_bounds__(256) embed_norm_kernel(const int32_t *tokens, const uint16_t *embed, int V,
                                                         int H, const uint16_t *gain, float eps, uint16_t *x,
                                                         uint16_t *h, uint32_t *status) {
    __shared__ float red[8];
    const int t = blockIdx.x;
    int tok = tokens[t];
    if (tok < 0 || tok >= V) {
        if (threadIdx.x == 0) atomicOr(status, kDevBounds);
        tok = 0;
    }
    uint16_t *xt = x + (size_t)t * H;
    for (int j = threadIdx.x; j < H; j += 256) xt[j] = embed[(size_t)tok * H + j];
    __syncthreads();
    norm_row(xt, gain, H, eps, h + (size_t)t * H, red);
}

// Sum over the sk split partials of 4 consecutive floats at p (split stride
// zs), in split order, with up to four splits' loads in flight.
__device__ __forceinline__ float4 split_sum4(const float *__restrict__ p, size_t zs, int sk) {
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [](float4 &a, const float4 &b) {
        a.x = __fadd_rn(a.x, b.x);
        a.y = __fadd_rn(a.y, b.y);
        a.z = __fadd_rn(a.z, b.z);
        a.w = __fadd_rn(a.w, b.w);
    };
    for (int s0 = 0; s0 < sk; s0 += 8) {
        float4 a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (s0 + i < sk) a[i] = __ldg(reinterpret_cast<const float4 *>(p + (size_t)(s0 + i) * zs));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (s0 + i < sk) add(y, a[i]);
    }
    return y;
}

// x[t] = R(x[t] + sum_s part[s][t]) (the split partial sums in order), then
// h[t] = R(rmsnorm(x[t]) * gain). 512 threads, four elements per thread and
// step (H is a multiple of 8).
__global__ void __launch_bounds__(512) resid_norm_kernel(const float *__restrict__ part, int sk, int T, int H,
                                                         uint16_t *__restrict__ x, const uint16_t *__restrict__ gain,
                                                         float eps, uint16_t *__restrict__ h) {
    __shared__ float red[16];
    const int t = blockIdx.x;
    uint16_t *xt = x + (size_t)t * H;
    const float *pt = part + (size_t)t * H;
    float ss = 0.f;
    for (int j = threadIdx.x * 4; j < H; j += 2048) {
        const float4 y = split_sum4(pt + j, (size_t)T * H, sk);
        const uint2 xv = *reinterpret_cast<const uint2 *>(xt + j);
        const float r0 = round_bf(__fadd_rn(bf_lo(xv.x), y.x)), r1 = round_bf(__fadd_rn(bf_hi(xv.x), y.y));
        const float r2 = round_bf(__fadd_rn(bf_lo(xv.y), y.z)), r3 = round_bf(__fadd_rn(bf_hi(xv.y), y.w));
        *reinterpret_cast<uint2 *>(xt + j) = make_uint2(pack_bf2(r0, r1), pack_bf2(r2, r3));
        ss = fmaf(r0, r0, ss);
        ss = fmaf(r1, r1, ss);
        ss = fmaf(r2, r2, ss);
        ss = fmaf(r3, r3, ss);
    }
    const float tot = block_sum<512>(ss, red);
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)H), eps)));
    uint16_t *ht = h + (size_t)t * H;
    for (int j = threadIdx.x * 4; j < H; j += 2048) {
        const uint2 xv = *reinterpret_cast<const uint2 *>(xt + j);
        const uint2 gv = *reinterpret_cast<const uint2 *>(gain + j);
        const float h0 = __fmul_rn(__fmul_rn(bf_lo(xv.x), r), bf_lo(gv.x));
        const float h1 = __fmul_rn(__fmul_rn(bf_hi(xv.x), r), bf_hi(gv.x));
        const float h2 = __fmul_rn(__fmul_rn(bf_lo(xv.y), r), bf_lo(gv.y));
        const float h3 = __fmul_rn(__fmul_rn(bf_hi(xv.y), r), bf_hi(gv.y));
        *reinterpret_cast<uint2 *>(ht + j) = make_uint2(pack_bf2(h0, h1), pack_bf2(h2, h3));
    }
}

// a[t][r] = R(silu(g) * u), g and u the split sums of packed rows 2r and 2r + 1;
// two rows per thread (F is a multiple of 8).
__global__ void __launch_bounds__(256) swiglu_kernel(const float *__restrict__ part, int sk, int T, int F,
                                                     uint16_t *__restrict__ a) {
    const size_t n2 = (size_t)T * F / 2;
    for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n2; i += (size_t)gridDim.x * 256) {
        const size_t e = 2 * i;  // output element: token e / F, rows r, r + 1
        const int t = (int)(e / F), r = (int)(e % F);
        const float4 y = split_sum4(part + (size_t)t * 2 * F + 2 * (size_t)r, (size_t)T * 2 * F, sk);
        const float s0 = __fdiv_rn(y.x, __fadd_rn(1.0f, expf(-y.x)));
        const float s1 = __fdiv_rn(y.z, __fadd_rn(1.0f, expf(-y.z)));
        *reinterpret_cast<uint32_t *>(a + e) = pack_bf2(__fmul_rn(s0, y.y), __fmul_rn(s1, y.w));
    }
}

// Per token and head (grid T x (nq + 2 nkv), one warp each, D / 32 elements a
// lane): the split sums of the Q/K/V rows, per-head RMSNorm (q_norm / k_norm)
// when enabled, RoPE at position P0 + t, q -> the q buffer (bf16), k and v ->
// the caches at P0 + t (bf16).
template <int D>
__global__ void __launch_bounds__(32) qkv_post_kernel(const float *part, int sk, int T, int rows, int nq, int nkv,
                                                      int max_pos, int layer, int P0, int qk_norm, float eps,
                                                      const uint16_t *q_norm, const uint16_t *k_norm,
                                                      const float *rope_cos, const float *rope_sin, uint16_t *q,
                                                      uint16_t *kc, uint16_t *vc) {
    constexpr int E = D / 32;
    const int t = blockIdx.x, hh = blockIdx.y, lane = threadIdx.x;
    const bool is_q = hh < nq, is_k = !is_q && hh < nq + nkv;
    const int kvh = is_q ? 0 : (is_k ? hh - nq : hh - nq - nkv);
    const int row0 = is_q ? hh * D : (is_k ? nq * D + kvh * D : nq * D + nkv * D + kvh * D);
    float v[E];
    const float *pt = part + (size_t)t * rows + row0 + lane;
    const size_t zs = (size_t)T * rows;
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = 0.f;
    int s = 0;
    for (; s + 2 <= sk; s += 2) {  // split sums in order, 2 E loads in flight
        float a0[E], a1[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            a0[e] = __ldg(pt + (size_t)s * zs + 32 * e);
            a1[e] = __ldg(pt + (size_t)(s + 1) * zs + 32 * e);
        }
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __fadd_rn(__fadd_rn(v[e], a0[e]), a1[e]);
    }
    for (; s < sk; ++s)
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __fadd_rn(v[e], __ldg(pt + (size_t)s * zs + 32 * e));
    const int P = P0 + t;
    const size_t crow = (((size_t)layer * nkv + kvh) * max_pos + P) * D;
    if (!is_q && !is_k) {
#pragma unroll
        for (int e = 0; e < E; ++e) vc[crow + lane + 32 * e] = f2bf(v[e]);
        return;
    }
    if (qk_norm) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
        ss = warp_sum(ss);
        const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)D), eps)));
        const uint16_t *gn = is_q ? q_norm : k_norm;
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], r), bf2f(gn[lane + 32 * e]));
    }
    const float *cs = rope_cos + (size_t)P * (D / 2);
    const float *sn = rope_sin + (size_t)P * (D / 2);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {  // rotate-half: element j pairs with j + D/2
        const int jx = lane + 32 * e;
        const float c = cs[jx], s = sn[jx];
        const float x0 = v[e], x1 = v[e + E / 2];
        v[e] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
        v[e + E / 2] = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
    }
    if (is_q) {
        uint16_t *qt = q + ((size_t)t * nq + hh) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) qt[lane + 32 * e] = f2bf(v[e]);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) kc[crow + lane + 32 * e] = f2bf(v[e]);
    }
}

// ------------------------------------------------------------------ attention
// Causal multi-query attention of KV head h over one split of the positions.
// Query rows r of the head are (token t, q head h G + i) with r = t G + i; a
// CTA takes 64 rows (4 warps x 16) and positions [p_lo, p_hi) of split z, in
// blocks of 64 staged in shared memory. Row r sees positions p <= P0 + t.
// Per block: s = q K^T d^-1/2 on m16n8k16 MMAs, online softmax per row,
// o += p V with p as a BF16 high part plus a BF16 remainder. Writes the
// split's partial (m, l, o[d]) of every row: part[(t nq + q head)][z][2 + d].
template <int D>
__global__ void __launch_bounds__(128) attn_mt_kernel(const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                                                      int layer, int nq, int nkv, int G, int max_pos, int P0, int T,
                                                      int split_len, float scale, float *part, int S) {
    constexpr int LD = D + 8;
    constexpr int NJ = D / 8;  // output n-tiles
    extern __shared__ __align__(128) uint16_t asm_[];
    uint16_t *sQ = asm_, *sK = asm_ + 64 * LD, *sV = asm_ + 2 * 64 * LD;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int h = blockIdx.y, z = blockIdx.z;
    const int R = T * G, r0 = blockIdx.x * 64;
    const int p_lo = z * split_len, p_hi = min((z + 1) * split_len, P0 + T);
    // Q rows of this CTA
    for (int i = tid; i < 64 * (D / 8); i += 128) {
        const int rr = i / (D / 8), c = (i % (D / 8)) * 8, r = r0 + rr;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < R) val = *reinterpret_cast<const uint4 *>(q + ((size_t)(r / G) * nq + h * G + r % G) * D + c);
        *reinterpret_cast<uint4 *>(sQ + rr * LD + c) = val;
    }
    // this lane's two rows and the last position each may see
    const int ra = r0 + warp * 16 + g, rb = ra + 8;
    const int lim_a = ra < R ? P0 + ra / G : -1, lim_b = rb < R ? P0 + rb / G : -1;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[NJ][4];
#pragma unroll
    for (int j = 0; j < NJ; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    const size_t head_base = ((size_t)layer * nkv + h) * max_pos;
    for (int pb = p_lo; pb < p_hi; pb += 64) {
        __syncthreads();  // previous block fully read
        for (int i = tid; i < 64 * (D / 8); i += 128) {
            const int pp = i / (D / 8), c = (i % (D / 8)) * 8, pos = pb + pp;
            uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
            if (pos < p_hi) {
                kv = *reinterpret_cast<const uint4 *>(kc + (head_base + pos) * D + c);
                vv = *reinterpret_cast<const uint4 *>(vc + (head_base + pos) * D + c);
            }
            *reinterpret_cast<uint4 *>(sK + pp * LD + c) = kv;
            *reinterpret_cast<uint4 *>(sV + pp * LD + c) = vv;
        }
        __syncthreads();
        // scores: 16 rows x 64 positions (8 n-tiles)
        float sc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        const uint16_t *qw = sQ + warp * 16 * LD;
#pragma unroll
        for (int kk = 0; kk < D; kk += 16) {
            uint32_t a[4];
            ldsm_x4(smem_u32(qw + (lane & 15) * LD + kk + (lane >> 4) * 8), a);
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t b[4];  // positions 8j .. 8j + 15
                ldsm_x4(smem_u32(sK + (8 * j + (lane & 7) + (lane >> 4) * 8) * LD + kk + ((lane >> 3) & 1) * 8), b);
                mma16816(sc[j], a, b[0], b[1]);
                mma16816(sc[j + 1], a, b[2], b[3]);
            }
        }
        // mask and scale; online softmax per row (rows g and g + 8 of the warp)
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int pos = pb + 8 * j + 2 * t4 + (e & 1);
                const int lim = (e >> 1) ? lim_b : lim_a;
                const float v = (pos < p_hi && pos <= lim) ? sc[j][e] * scale : -INFINITY;
                sc[j][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        float corr[2], mn[2];
#pragma unroll
        for (int rI = 0; rI < 2; ++rI) {
            mx[rI] = fmaxf(mx[rI], __shfl_xor_sync(0xFFFFFFFFu, mx[rI], 1));
            mx[rI] = fmaxf(mx[rI], __shfl_xor_sync(0xFFFFFFFFu, mx[rI], 2));
            mn[rI] = fmaxf(m[rI], mx[rI]);
            const float base = mn[rI] == -INFINITY ? 0.f : mn[rI];  // nothing seen yet: keep zeros
            corr[rI] = expf(m[rI] - base);
            mn[rI] = base;
        }
        float ls[2] = {0.f, 0.f};
        uint32_t phi[4][4], plo[4][4];  // A fragments of p for the 4 k-steps of 16 positions
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pv[e] = expf(sc[j][e] - mn[e >> 1]);
                ls[e >> 1] += pv[e];
            }
            const float h0 = bf2f(f2bf(pv[0])), h1 = bf2f(f2bf(pv[1])), h2 = bf2f(f2bf(pv[2])), h3 = bf2f(f2bf(pv[3]));
            // k-step j / 2: tile 2 kk holds a0 (row g) and a1 (row g + 8), tile 2 kk + 1 a2 and a3
            const int ks = j >> 1, hi = j & 1;
            phi[ks][2 * hi + 0] = pack_bf2(h0, h1);
            phi[ks][2 * hi + 1] = pack_bf2(h2, h3);
            plo[ks][2 * hi + 0] = pack_bf2(__fsub_rn(pv[0], h0), __fsub_rn(pv[1], h1));
            plo[ks][2 * hi + 1] = pack_bf2(__fsub_rn(pv[2], h2), __fsub_rn(pv[3], h3));
        }
#pragma unroll
        for (int rI = 0; rI < 2; ++rI) {
            ls[rI] += __shfl_xor_sync(0xFFFFFFFFu, ls[rI], 1);
            ls[rI] += __shfl_xor_sync(0xFFFFFFFFu, ls[rI], 2);
            l[rI] = fmaf(l[rI], corr[rI], ls[rI]);
            m[rI] = mx[rI] == -INFINITY && m[rI] == -INFINITY ? -INFINITY : mn[rI];
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            o[j][0] *= corr[0];
            o[j][1] *= corr[0];
            o[j][2] *= corr[1];
            o[j][3] *= corr[1];
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            // mma A order {a0, a1, a2, a3} = {(g, k 2t..), (g + 8, k 2t..), (g, k 2t + 8..), (g + 8, k 2t + 8..)}
            const uint32_t ah[4] = {phi[ks][0], phi[ks][1], phi[ks][2], phi[ks][3]};
            const uint32_t al[4] = {plo[ks][0], plo[ks][1], plo[ks][2], plo[ks][3]};
#pragma unroll
            for (int j = 0; j < NJ; j += 2) {
                uint32_t b[4];  // positions 16 ks (+8), dims 8j and 8j + 8, transposed
                ldsm_x4_t(smem_u32(sV + (16 * ks + ((lane >> 3) & 1) * 8 + (lane & 7)) * LD + 8 * j + (lane >> 4) * 8), b);
                mma16816(o[j], ah, b[0], b[1]);
                mma16816(o[j], al, b[0], b[1]);
                mma16816(o[j + 1], ah, b[2], b[3]);
                mma16816(o[j + 1], al, b[2], b[3]);
            }
        }
    }
    // partials of this lane's two rows
#pragma unroll
    for (int rI = 0; rI < 2; ++rI) {
        const int r = rI ? rb : ra;
        if (r >= R) continue;
        float *dst = part + (((size_t)(r / G) * nq + h * G + r % G) * S + z) * (2 + D);
        if (t4 == 0) {
            dst[0] = m[rI];
            dst[1] = l[rI];
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            dst[2 + 8 * j + 2 * t4] = o[j][2 * rI];
            dst[2 + 8 * j + 2 * t4 + 1] = o[j][2 * rI + 1];
        }
    }
}

// o[t][i][dd] = R(sum_z w_z o_z / sum_z w_z l_z), w_z = e^(m_z - max m), over
// the splits in order (grid T x nq, D threads).
__global__ void attn_combine_kernel(const float *part, int S, int nq, int D, uint16_t *o) {
    const int t = blockIdx.x, i = blockIdx.y, dd = threadIdx.x;
    const float *pr = part + ((size_t)t * nq + i) * S * (2 + D);
    float M = -INFINITY;
    for (int z = 0; z < S; ++z) M = fmaxf(M, pr[(size_t)z * (2 + D)]);
    float L = 0.f, O = 0.f;
    for (int z = 0; z < S; ++z) {
        const float mz = pr[(size_t)z * (2 + D)];
        if (mz == -INFINITY) continue;
        const float w = expf(mz - M);
        L = fmaf(w, pr[(size_t)z * (2 + D) + 1], L);
        O = fmaf(w, pr[(size_t)z * (2 + D) + 2 + dd], O);
    }
    o[((size_t)t * nq + i) * D + dd] = f2bf(__fdiv_rn(O, L));
}

// Greedy choice per token: the largest logit, lowest index on ties. Grid
// (T, kArgBlocks): each block reduces a slice of the row to the packed key
// (ordered logit, inverted row) and raises keys[t] to it; the last block of
// the token (a per-token ticket) writes the row and resets keys[t] and the
// ticket for the next pass. The maximum does not depend on the order of the
// atomics.
constexpr int kArgBlocks = 16;
__global__ void __launch_bounds__(256) argmax_kernel(const float *__restrict__ logits, int V,
                                                     unsigned long long *keys, uint32_t *tickets, int32_t *out) {
    __shared__ unsigned long long best[8];
    const int t = blockIdx.x;
    const float *lt = logits + (size_t)t * V;
    const int per = (V + kArgBlocks - 1) / kArgBlocks;
    const int r0 = blockIdx.y * per, r1 = min(V, r0 + per);
    unsigned long long k = 0;
    for (int r = r0 + threadIdx.x; r < r1; r += 256) {
        const unsigned long long kk = argmax_key(lt[r], (uint32_t)r);
        k = kk > k ? kk : k;
    }
    k = warp_max_u64(k);
    if ((threadIdx.x & 31) == 0) best[threadIdx.x >> 5] = k;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long b = 0;
        for (int w = 0; w < 8; ++w) b = best[w] > b ? best[w] : b;
        atomicMax(&keys[t], b);
        __threadfence();
        if (atomicAdd(&tickets[t], 1u) == kArgBlocks - 1) {
            __threadfence();
            const unsigned long long m = atomicMax(&keys[t], 0ull);
            out[t] = key_row(m);
            keys[t] = 0ull;
            tickets[t] = 0u;
        }
    }
}

// Greedy acceptance of a verify step: inputs = last token, d_1 .. d_k; a_i =
// argmax after input i. n = the longest prefix with d_{i+1} == a_i; emits
// d_1 .. d_n, then a_n.
__global__ void accept_kernel(const int32_t *inputs, const int32_t *argmax, int k, int32_t *tokens,
                              int32_t *n_accepted) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int n = 0;
    while (n < k && inputs[n + 1] == argmax[n]) ++n;
    for (int i = 0; i < n; ++i) tokens[i] = inputs[i + 1];
    tokens[n] = argmax[n];
    *n_accepted = n;
}

// ------------------------------------------------------------------ host side
// The 2-D BF16 tensor map of an operand, made once per (base, shape, box).
const TensorMap *operand_map(ForwardScratch &f, const void *base, int inner, int rows, int ld, int box_rows) {
    const std::array<uint64_t, 5> key = {(uint64_t)(uintptr_t)base, (uint64_t)inner, (uint64_t)rows,
                                         (uint64_t)ld, (uint64_t)box_rows};
    for (auto &e : f.maps)
        if (e.first == key) return &e.second;
    if (f.maps.size() >= 4096) f.maps.clear();
    TensorMap m;
    if (!encode_bf16_2d(&m, base, (uint64_t)inner, (uint64_t)rows, (uint64_t)ld * 2, 64, (uint32_t)box_rows))
        return nullptr;
    f.maps.emplace_back(key, m);
    return &f.maps.back().second;
}

// Launches C = W X^T (split partial sums) on the tensor cores and returns the
// split count: W [M][K] (ldw elements per row), X [T][K] (ldx). With act
// (gate/up rows in pairs) and a single split, the SwiGLU output goes to act
// instead of C and *sk_out is 0.
cudaError_t gemm(tiles_plan_s *plan, const void *W, int ldw, const uint16_t *X, int ldx, int M, int T, int K,
                 float *C, int max_sk, int *sk_out, cudaStream_t st, uint16_t *act = nullptr) {
    const TcShape s = tc_shape(M, T, K, plan->sm_count, max_sk);
    ForwardScratch &f = plan->fwd;
    const TensorMap *mw = operand_map(f, W, K, M, ldw, kTcM);
    const TensorMap *mx = mw ? operand_map(f, X, K, T, ldx, s.n_tile) : nullptr;
    if (!mw || !mx) return cudaErrorInvalidValue;
    if (s.sk != 1) act = nullptr;
    *sk_out = act ? 0 : s.sk;
    return gemm_tc_launch(*mw, *mx, s, M, T, K, C, act, plan->base.status, plan->base.timeout_ns, st);
}

// splits of the attention: about two CTAs per SM over the (query block, KV
// head, split) grid, each split a multiple of 64 positions
int attn_splits_wanted(const Geom &g, int T, int sms) {
    const int qb = (T * g.G + 63) / 64;
    return std::max(1, (2 * sms + qb * g.nkv - 1) / (qb * g.nkv));
}
int attn_split_len(const Geom &g, int P0, int T, int sms) {
    const int want = attn_splits_wanted(g, T, sms);
    int len = ((P0 + T + want - 1) / want + 63) / 64 * 64;
    return std::max(64, len);
}
size_t attn_smem(int d) { return (size_t)3 * 64 * (d + 8) * 2; }

}  // namespace fwd
}  // namespace tiles

using namespace tiles;
using namespace tiles::fwd;

namespace {

template <typename T>
cudaError_t falloc(tiles_plan_s *p, T **ptr, size_t bytes) {
    void *v = nullptr;
    cudaError_t e = cudaMalloc(&v, bytes ? bytes : 16);
    if (e != cudaSuccess) return e;
    p->fwd.allocs.push_back(v);
    *ptr = reinterpret_cast<T *>(v);
    return cudaSuccess;
}

// Working memory for passes of up to kMaxTokens tokens (first use).
tiles_status_t forward_setup(tiles_plan_s *plan) {
    ForwardScratch &f = plan->fwd;
    if (f.ready) return TILES_OK;
    const Geom &g = plan->sched.geom;
    const int Tm = kMaxTokens;
    size_t part = 0;
    for (int T = 1; T <= Tm; ++T) {
        const int shapes[4][2] = {{g.qkv_rows, g.H}, {g.H, g.qd}, {2 * g.F, g.H}, {g.H, g.F}};
        for (auto &mk : shapes) {
            const TcShape s = tc_shape(mk[0], T, mk[1], plan->sm_count, 1 << 30);
            part = std::max(part, (size_t)s.sk * T * mk[0]);
        }
    }
    // (token, split) pairs of the attention partials: a pass of T tokens has at
    // most min(ceil(max_pos / 64), wanted(T)) splits
    size_t pairs = 0;
    for (int T = 1; T <= Tm; ++T)
        pairs = std::max(pairs, (size_t)T * std::min((g.max_pos + 63) / 64,
                                                     attn_splits_wanted(g, T, plan->sm_count)));
    if (falloc(plan, &f.x, (size_t)Tm * g.H * 2) != cudaSuccess ||
        falloc(plan, &f.h, (size_t)Tm * g.H * 2) != cudaSuccess ||
        falloc(plan, &f.q, (size_t)Tm * g.qd * 2) != cudaSuccess ||
        falloc(plan, &f.o, (size_t)Tm * g.qd * 2) != cudaSuccess ||
        falloc(plan, &f.a, (size_t)Tm * g.F * 2) != cudaSuccess ||
        falloc(plan, &f.part, part * 4) != cudaSuccess ||
        falloc(plan, &f.apart, pairs * g.nq * (2 + g.d) * 4) != cudaSuccess ||
        falloc(plan, &f.logits, (size_t)Tm * g.V * 4) != cudaSuccess ||
        falloc(plan, &f.argmax, (size_t)Tm * 4) != cudaSuccess ||
        falloc(plan, &f.tokens, (size_t)(Tm + 1) * 4) != cudaSuccess ||
        falloc(plan, &f.arg_keys, (size_t)Tm * 8) != cudaSuccess ||
        falloc(plan, &f.arg_tickets, (size_t)Tm * 4) != cudaSuccess)
        return TILES_ERR_CUDA;
    // the argmax kernel leaves them at zero after every pass
    if (cudaMemset(f.arg_keys, 0, (size_t)Tm * 8) != cudaSuccess ||
        cudaMemset(f.arg_tickets, 0, (size_t)Tm * 4) != cudaSuccess)
        return TILES_ERR_CUDA;
    f.part_elems = part;
    f.attn_pairs = pairs;
    for (int d : {64, 128}) {
        const void *k = d == 64 ? (const void *)attn_mt_kernel<64> : (const void *)attn_mt_kernel<128>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem(d)) != cudaSuccess)
            return TILES_ERR_CUDA;
    }
    if (gemm_tc_configure() != cudaSuccess) return TILES_ERR_CUDA;
    f.ready = true;
    return TILES_OK;
}

// One pass of T <= kMaxTokens tokens at positions P0 .. P0 + T - 1.
tiles_status_t forward_pass(tiles_plan_s *plan, uint16_t *kc, uint16_t *vc, const int32_t *tokens, int T, int P0,
                            cudaStream_t st, int32_t *argmax, float *logits) {
    const Geom &g = plan->sched.geom;
    const KernelParams &kp = plan->base;
    ForwardScratch &f = plan->fwd;
    const int sms = plan->sm_count;
    const float eps = kp.eps;
    std::vector<LayerPtrs> &lp = plan->layers_host;
    int sk = 1;
    embed_norm_kernel<<<T, 256, 0, st>>>(tokens, kp.embed, g.V, g.H, lp[0].attn_norm, eps, f.x, f.h, kp.status);
    const int split = attn_split_len(g, P0, T, sms);
    const int S = (P0 + T + split - 1) / split;
    if ((size_t)T * S > f.attn_pairs) return TILES_ERR_CAPACITY;
    const dim3 agrid((T * g.G + 63) / 64, g.nkv, S);
    for (int l = 0; l < g.L; ++l) {
        const LayerPtrs &L = lp[l];
        if (gemm(plan, L.qkv, g.H, f.h, g.H, g.qkv_rows, T, g.H, f.part, 1 << 30, &sk, st) != cudaSuccess)
            return TILES_ERR_CUDA;
        const dim3 qgrid(T, g.nq + 2 * g.nkv);
        if (g.d == 64)
            qkv_post_kernel<64><<<qgrid, 32, 0, st>>>(f.part, sk, T, g.qkv_rows, g.nq, g.nkv, g.max_pos, l, P0,
                                                      kp.qk_norm, eps, L.q_norm, L.k_norm, kp.rope_cos,
                                                      kp.rope_sin, f.q, kc, vc);
        else
            qkv_post_kernel<128><<<qgrid, 32, 0, st>>>(f.part, sk, T, g.qkv_rows, g.nq, g.nkv, g.max_pos, l, P0,
                                                       kp.qk_norm, eps, L.q_norm, L.k_norm, kp.rope_cos,
                                                       kp.rope_sin, f.q, kc, vc);
        if (g.d == 64)
            attn_mt_kernel<64><<<agrid, 128, attn_smem(64), st>>>(f.q, kc, vc, l, g.nq, g.nkv, g.G, g.max_pos, P0, T, split,
                                                      kp.attn_scale, f.apart, S);
        else
            attn_mt_kernel<128><<<agrid, 128, attn_smem(128), st>>>(f.q, kc, vc, l, g.nq, g.nkv, g.G, g.max_pos, P0, T, split,
                                                       kp.attn_scale, f.apart, S);
        attn_combine_kernel<<<dim3(T, g.nq), g.d, 0, st>>>(f.apart, S, g.nq, g.d, f.o);
        if (gemm(plan, L.o, g.qd, f.o, g.qd, g.H, T, g.qd, f.part, 1 << 30, &sk, st) != cudaSuccess)
            return TILES_ERR_CUDA;
        resid_norm_kernel<<<T, 512, 0, st>>>(f.part, sk, T, g.H, f.x, L.ffn_norm, eps, f.h);
        // Short passes with one gate/up split run the SwiGLU in the projection's
        // epilogue. Measured on GB300, Llama-1B shape: 17-token verify steps
        // 1.45 -> 1.42 ms; a 256-token prefill pass 4.20 -> 5.27 ms, as four
        // warps per SM then spend ~30 us on the divisions the separate kernel
        // spreads over the whole GPU.
        if (gemm(plan, L.gu, g.H, f.h, g.H, 2 * g.F, T, g.H, f.part, 1 << 30, &sk, st, T <= 32 ? f.a : nullptr) !=
            cudaSuccess)
            return TILES_ERR_CUDA;
        if (sk > 0)
            swiglu_kernel<<<std::min(4096, (T * g.F / 2 + 255) / 256), 256, 0, st>>>(f.part, sk, T, g.F, f.a);
        if (gemm(plan, L.down, g.F, f.a, g.F, g.H, T, g.F, f.part, 1 << 30, &sk, st) != cudaSuccess)
            return TILES_ERR_CUDA;
        const uint16_t *next_gain = l + 1 < g.L ? lp[l + 1].attn_norm : kp.final_norm;
        resid_norm_kernel<<<T, 512, 0, st>>>(f.part, sk, T, g.H, f.x, next_gain, eps, f.h);
    }
    // LM head (tied embedding), one split: the partial sums are the logits
    float *lg = logits ? logits : f.logits;
    if (gemm(plan, kp.embed, g.H, f.h, g.H, g.V, T, g.H, lg, 1, &sk, st) != cudaSuccess) return TILES_ERR_CUDA;
    argmax_kernel<<<dim3(T, kArgBlocks), 256, 0, st>>>(lg, g.V, f.arg_keys, f.arg_tickets, argmax);
    return cudaGetLastError() == cudaSuccess ? TILES_OK : TILES_ERR_CUDA;
}

tiles_status_t forward_check(tiles_plan_t plan, void *k_cache, void *v_cache, int32_t n, int32_t start_pos) {
    if (!plan || !k_cache || !v_cache || n < 1 || start_pos < 0) return TILES_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
        return TILES_ERR_INVALID_ARG;
    const Geom &g = plan->sched.geom;
    if (g.wbytes != 2 || g.kv8) return TILES_ERR_UNSUPPORTED;  // BF16 weights and cache only
    if ((long long)start_pos + n > g.max_pos) return TILES_ERR_CAPACITY;
    tiles_status_t st = plan_check_device(plan);
    if (st != TILES_OK) return st;
    return forward_setup(plan);
}

}  // namespace

extern "C" {

tiles_status_t tiles_forward(tiles_plan_t plan, void *k_cache, void *v_cache, const int32_t *tokens,
                             int32_t n_tokens, int32_t start_pos, void *stream, int32_t *out_argmax,
                             float *out_logits) {
    if (!tokens || !out_argmax) return TILES_ERR_INVALID_ARG;
    tiles_status_t st = forward_check(plan, k_cache, v_cache, n_tokens, start_pos);
    if (st != TILES_OK) return st;
    const Geom &g = plan->sched.geom;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    for (int t0 = 0; t0 < n_tokens; t0 += kMaxTokens) {
        const int T = std::min(kMaxTokens, n_tokens - t0);
        st = forward_pass(plan, reinterpret_cast<uint16_t *>(k_cache), reinterpret_cast<uint16_t *>(v_cache),
                          tokens + t0, T, start_pos + t0, cs, out_argmax + t0,
                          out_logits ? out_logits + (size_t)t0 * g.V : nullptr);
        if (st != TILES_OK) return st;
    }
    return TILES_OK;
}

tiles_status_t tiles_verify(tiles_plan_t plan, void *k_cache, void *v_cache, const int32_t *inputs, int32_t k,
                            int32_t start_pos, void *stream, int32_t *out_tokens, int32_t *out_n_accepted,
                            float *out_logits) {
    if (!inputs || !out_tokens || !out_n_accepted || k < 0 || k + 1 > kMaxTokens) return TILES_ERR_INVALID_ARG;
    tiles_status_t st = forward_check(plan, k_cache, v_cache, k + 1, start_pos);
    if (st != TILES_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    st = forward_pass(plan, reinterpret_cast<uint16_t *>(k_cache), reinterpret_cast<uint16_t *>(v_cache), inputs,
                      k + 1, start_pos, cs, plan->fwd.argmax, out_logits);
    if (st != TILES_OK) return st;
    accept_kernel<<<1, 32, 0, cs>>>(inputs, plan->fwd.argmax, k, out_tokens, out_n_accepted);
    return cudaGetLastError() == cudaSuccess ? TILES_OK : TILES_ERR_CUDA;
}

}  // extern "C"

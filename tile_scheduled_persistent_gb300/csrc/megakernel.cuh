// The persistent decode kernel for sm_103a.
//
// One CTA per SM runs its static task list once per step, for up to 64 steps
// per cooperative launch ("Tiles: Scheduling LLM Decoding as a Graph of
// Tiles", intro and "What the code contains": a fixed worker per SM executes a
// planned schedule, greedy selection inside the kernel, up to 64 tokens per
// launch). Each CTA has
//   - one producer warp: a single lane walks the same task list as the
//     consumers and streams every tile's weight rows (or K/V positions) into a
//     shared-memory ring with cp.async.bulk (TMA) copies, completing on per-slot
//     mbarriers. Weights never depend on activations, so the stream runs ahead
//     across phase boundaries and keeps HBM busy while the consumers wait
//     (the megakernel paragraph of the same page: load the next weights while
//     the current work finishes).
//   - eight consumer warps: chunk j of the CTA's stream goes to ring slot
//     j % slots, and each slot has one owning warp, (j % slots) % 8. GEMV chunks: 16-byte bf16 loads from shared memory,
//     FP32 FMA, warp-shuffle reductions. Attention chunks: split-KV online
//     softmax over up to kv_block positions per chunk.
// Phases are ordered by counters in global memory (one grid barrier per phase
// in the wave schedule, or per-phase dependency counters): release-add after a
// task, acquire-spin before one. Every spin is bounded by the global timer;
// on expiry the CTA records an error in the status word, drains its copies in
// flight and returns, and every other CTA leaves at its next wait.
//
// Fused work (same page, intro: norms and activations fold into the tiles
// next to them; "History and roadmap", "M8 so far": q/k norm + RoPE + KV
// write, residual + RMSNorm and SwiGLU-in-GEMV fusions):
//   QKV tiles     RMSNorm of the residual in the prologue
//   ATTN tiles    per-head q/k RMSNorm, RoPE, KV write at the new position
//   O / DOWN      residual add in the epilogue
//   GATE/UP       RMSNorm prologue, SwiGLU epilogue
//   LM head       final RMSNorm prologue, argmax epilogue (packed 64-bit
//                 atomicMax: ordered logit bits high, inverted row low, so the
//                 lowest row wins ties)
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tiles_internal.h"

namespace tiles {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// One box of a 3-D tiled tensor map (coordinates innermost first) into shared
// memory, completing on an mbarrier. `map` is the address of a tensor map in
// kernel-parameter space; the innermost coordinate is a multiple of 64
// elements (128 bytes), as the tiled copy requires 16-byte alignment there.
__device__ __forceinline__ void tensor_g2s_3d(void *dst, const TensorMap *map, int x, int y, int z,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tensor_g2s_2d(void *dst, const TensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Tensor-core helpers of the attention tiles: four 8x8 BF16 matrices from
// shared memory (lanes 8i..8i+7 give the row addresses of matrix i), plain or
// transposed, and one m16n8k16 BF16 MMA with FP32 accumulation.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// c += A B for A 16x16 and B 16x8 when only rows 0..7 of A are nonzero:
// a0 = (row g, k 2t..2t+1) and a2 = (row g, k 2t+8..2t+9) for lane (g, t) =
// (lane / 4, lane % 4), b0 = (k 2t..2t+1, n g), b1 = (k 2t+8..2t+9, n g), and
// the accumulator of row g, columns 2t and 2t+1, in c0, c1 (rows 8..15 of
// the result are zero and are not kept).
__device__ __forceinline__ void mma_rows8(float &c0, float &c1, uint32_t a0, uint32_t a2, uint32_t b0,
                                          uint32_t b1) {
    asm volatile("{\n\t.reg .f32 z2, z3;\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, z2, z3}, {%2, %6, %3, %6}, {%4, %5},"
        " {%0, %1, %7, %7};\n\t}"
        : "+f"(c0), "+f"(c1)
        : "r"(a0), "r"(a2), "r"(b0), "r"(b1), "r"(0u), "f"(0.f));
}

// c += A B, A 16x16 and B 16x8 in full: a = {(g, 2t..2t+1), (g+8, 2t..2t+1),
// (g, 2t+8..2t+9), (g+8, 2t+8..2t+9)}, b = {(k 2t..2t+1, n g), (k 2t+8..2t+9,
// n g)}, c = {(g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)} for lane (g, t).
__device__ __forceinline__ void mma_m16n8k16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9},"
        " {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The transpose of an 8x8 matrix of 16-bit elements held as lane (g, t):
// row g, columns 2t and 2t+1; returns the same lane's pair of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Byte offset of 16-byte unit u (elements 8u..8u+7) of row r in a chunk region
// written by the tiled copy with the 128-byte swizzle: boxes of kvb rows x 128
// bytes one after another (unit u lives in box u / 8), and inside each
// 1024-byte-aligned group of 8 rows the unit index is XORed with the row
// index mod 8.
__device__ __forceinline__ uint32_t swz_off(int kvb, int r, int u) {
    return ((uint32_t)(u >> 3) * (uint32_t)kvb + (uint32_t)r) * 128u + ((uint32_t)((u & 7) ^ (r & 7)) << 4);
}

// Byte offset of 16-byte unit u of row r in an INT8 cache tile written by the
// tiled copy with rows of RB bytes (64 or 128) and the swizzle of that width:
// the unit index is XORed with bits 7.. of the row's offset (128-byte rows:
// r mod 8; 64-byte rows: (r / 2) mod 4). Tiles start 1024-byte aligned.
template <int RB>
__device__ __forceinline__ uint32_t swz8_off(int r, int u) {
    static_assert(RB == 64 || RB == 128, "swizzled rows are 64 or 128 bytes");
    if (RB == 128) return (uint32_t)r * 128u + ((uint32_t)(u ^ (r & 7)) << 4);
    return (uint32_t)r * 64u + ((uint32_t)(u ^ ((r >> 1) & 3)) << 4);
}

// Four INT8 codes (bytes c0..c3 of w) as two BF16 pairs (c0, c1) and (c2, c3),
// exactly. With the byte 0x43 above it, a byte b is the BF16 number whose
// exponent carries b's top bit: 128 + (b & 127) when that bit is clear; so
// (0x43, c & 127) - (0x43, c & 128) is 128 + (c & 127) - 128 = c for c >= 0
// and 128 + (c + 128) - 256 = c for c < 0. One exact BF16 subtraction per pair.
__device__ __forceinline__ void codes_bf16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x0 = __byte_perm(w, 0x43434343u, 0x4140);  // [c0, 0x43, c1, 0x43]
    const uint32_t x1 = __byte_perm(w, 0x43434343u, 0x4342);  // [c2, 0x43, c3, 0x43]
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(x0 & 0xFF7FFF7Fu), "r"(x0 & 0xFF80FF80u));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(x1 & 0xFF7FFF7Fu), "r"(x1 & 0xFF80FF80u));
}

__device__ __forceinline__ void bulk_g2s_nohint(void *dst, const void *src, uint32_t bytes,
                                                uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *src) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
}
__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.volatile.shared.u64 %0, [%1];" : "=l"(v) : "r"((uint32_t)__cvta_generic_to_shared(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_volatile_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.volatile.shared.u64 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint32_t *p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile(const uint32_t *p) {
    return *(const volatile uint32_t *)p;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_release_cta(int *p, int v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta(const int *p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Consumer barrier that also ORs a flag over all consumer threads: every thread
// gets the same answer, so leaving on it keeps the barrier sequence aligned.
__device__ __forceinline__ bool consumer_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kConsumerWarps * 32)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ numerics
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// float -> bfloat16, round to nearest even (finite inputs; NaN kept as NaN)
__device__ __forceinline__ uint16_t f2bf(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
__device__ __forceinline__ float round_bf(float f) { return bf2f(f2bf(f)); }

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

__device__ __forceinline__ float dot8(const uint4 &w, const float (&x)[8], float acc) {
    acc = fmaf(bf_lo(w.x), x[0], acc); acc = fmaf(bf_hi(w.x), x[1], acc);
    acc = fmaf(bf_lo(w.y), x[2], acc); acc = fmaf(bf_hi(w.y), x[3], acc);
    acc = fmaf(bf_lo(w.z), x[4], acc); acc = fmaf(bf_hi(w.z), x[5], acc);
    acc = fmaf(bf_lo(w.w), x[6], acc); acc = fmaf(bf_hi(w.w), x[7], acc);
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// order-preserving key of (logit, row): bigger logit first, lower row on ties
__device__ __forceinline__ unsigned long long argmax_key(float f, uint32_t row) {
    uint32_t u = __float_as_uint(f);
    uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - row);
}
__device__ __forceinline__ int key_row(unsigned long long k) {
    return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

// ------------------------------------------------------------------ shared state
struct Ctl {
    int unused;
    int token;
    int step_ready;  // consumers passed the first wait of this step (KV of earlier steps visible)
    float red[kConsumerWarps];
    unsigned long long warp_key[kConsumerWarps];
    unsigned long long stream_pos;  // weight bytes the producers have handed to the ring
};

static_assert(2 * kMaxSlots * 8 + sizeof(Ctl) <= (size_t)kCtlBytes, "control block overflows its region");

struct Smem {
    uint64_t *full, *empty;
    Ctl *ctl;
    uint8_t *ring;
    uint8_t *vec;
};

__device__ __forceinline__ Smem smem_layout(uint8_t *base, const KernelParams &p) {
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(base);
    s.empty = s.full + kMaxSlots;
    s.ctl = reinterpret_cast<Ctl *>(base + 2 * kMaxSlots * 8);
    s.ring = base + p.ring_off;
    s.vec = base + p.vec_off;
    return s;
}

__device__ __forceinline__ bool failed(const KernelParams &p) { return ld_volatile(p.status) != 0; }

// ------------------------------------------------------------------ tagged activations
// Activation words carry the tag of the phase that wrote them:
// 1 + 6 (step L + layer) + kind, with kind 0 for the Q/K/V rows, 1 for x after
// the O-projection, 2 for the SwiGLU output a, 3 for x after the down
// projection, 4 for the split partials, 5 for the merged attention output o.
// The step is the launch's own (< 64), so within a launch no tag repeats (at
// most 384 L < 2^16), and every launch starts from zeroed words, so 0 never
// matches and nothing of an earlier launch reads as ready.
enum { kTagQKV = 0, kTagXAttn = 1, kTagA = 2, kTagXFfn = 3, kTagPart = 4, kTagO = 5 };
__device__ __forceinline__ uint32_t act_tag(const KernelParams &p, int step, int layer, int kind) {
    return 1u + 6u * ((uint32_t)step * (uint32_t)p.g.L + (uint32_t)layer) + (uint32_t)kind;
}

// Bounded polling of tagged words, like every other wait: the global timer
// limits it, and a failure elsewhere ends it.
struct Poll {
    unsigned long long t0 = 0;
    uint32_t spins = 0;
    // false: stop polling (timeout recorded in the status word, or the run is aborting)
    __device__ bool again(const KernelParams &p) {
        if (t0 == 0) t0 = global_timer();
        if ((++spins & 31u) == 0) {
            if (failed(p)) return false;
            if (global_timer() - t0 > p.timeout_ns) {
                atomicOr(p.status, kDevTimeout);
                return false;
            }
        }
        return true;
    }
};

__device__ __forceinline__ bool tags_ok4(const uint4 &w, uint32_t tag) {
    return ((w.x >> 16) == tag) & ((w.y >> 16) == tag) & ((w.z >> 16) == tag) & ((w.w >> 16) == tag);
}
// the bf16 halves of 8 tagged words, packed as 8 consecutive bf16
__device__ __forceinline__ uint4 untag8(const uint4 &lo, const uint4 &hi) {
    return make_uint4(__byte_perm(lo.x, lo.y, 0x5410), __byte_perm(lo.z, lo.w, 0x5410),
                      __byte_perm(hi.x, hi.y, 0x5410), __byte_perm(hi.z, hi.w, 0x5410));
}

__device__ __forceinline__ unsigned long long *trace_rec(const KernelParams &p, int cta, int step,
                                                         int task) {
    if (!p.trace || step >= p.trace_steps) return nullptr;
    return p.trace + (((size_t)cta * p.trace_steps + step) * p.trace_tasks + task) * kTraceWords;
}

// Bounded spin until counter >= target. false when the run is aborting.
// Acquire side of a dependency counter: relaxed polls, one acquire fence once
// the target is seen (the signal side is a release reduction after a CTA
// barrier, which orders every thread's writes of the tile before it).
static __device__ bool wait_counter(const KernelParams &p, const uint32_t *ctr, uint32_t target) {
    if (ld_relaxed(ctr) >= target) {
        fence_acquire_gpu();
        return true;
    }
    unsigned long long t0 = global_timer();
    for (uint32_t spin = 1;; ++spin) {
        if (ld_relaxed(ctr) >= target) {
            fence_acquire_gpu();
            return true;
        }
        if ((spin & 31u) == 0) {
            if (failed(p)) return false;
            if (global_timer() - t0 > p.timeout_ns) {
                atomicOr(p.status, kDevTimeout);
                return false;
            }
        }
    }
}

// Bounded mbarrier wait. false on timeout or when the run is aborting.
static __device__ bool wait_mbar(const KernelParams &p, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = global_timer();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 15u) == 0) {
            if (failed(p)) return false;
            if (global_timer() - t0 > p.timeout_ns) {
                atomicOr(p.status, kDevTimeout);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ producer
struct Producer {
    const KernelParams &p;
    Smem &s;
    uint32_t j = 0;  // chunks issued
    bool ok = true;
    unsigned long long pol_weights;  // L2 evict-first: weights are streamed once per step
    unsigned long long stall = 0;    // ns spent waiting for a free slot (traced runs)
    bool tracing = false;
    int pid = 0;                     // this producer issues chunks of slots with slot % 2 == pid

    __device__ Producer(const KernelParams &p_, Smem &s_, int pid_) : p(p_), s(s_), pid(pid_) {
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_weights));
    }

    // Weight rows [r0, ...) of a GEMV tile (BF16 or INT8 codes): where they
    // start in HBM. A gate/up row is the pair of packed rows (gate, up).
    __device__ const uint8_t *gemv_src(int op, int layer, uint32_t r0) const {
        const LayerPtrs &lw = p.layers[layer];
        const size_t rb = (size_t)op_in_dim(p.g, op) * p.g.wbytes * op_mats(op);
        switch (op) {
            case TILES_OP_QKV: return lw.qkv + r0 * rb;
            case TILES_OP_OPROJ: return lw.o + r0 * rb;
            case TILES_OP_GATEUP: return lw.gu + r0 * rb;
            case TILES_OP_DOWN: return lw.down + r0 * rb;
            default: return p.lm + r0 * rb;
        }
    }

    unsigned long long stream_bytes = 0;  // weight bytes of every chunk passed so far

    // Chunk j's slot belongs to this producer?
    __device__ bool owns(uint32_t jj) const {
        return (int)((jj % (uint32_t)p.g.ring_slots) % kProducerWarps) == pid;
    }

    // Reserve the next slot: wait until its previous chunk was consumed.
    __device__ uint8_t *acquire(uint64_t **bar) {
        const uint32_t ns = (uint32_t)p.g.ring_slots;
        uint32_t slot = j % ns;
        if (j >= ns) {
            unsigned long long t0 = tracing ? global_timer() : 0;
            const uint32_t par = ((j / ns) - 1u) & 1u;
            if (!wait_mbar(p, &s.empty[slot], par)) {
                ok = false;
                return nullptr;
            }
            if (tracing) stall += global_timer() - t0;
        }
        *bar = &s.full[slot];
        return s.ring + (size_t)slot * p.g.slot_bytes;
    }

    __device__ void gemv_chunk(int op, int layer, uint32_t r0, uint32_t nr) {
        stream_bytes += (unsigned long long)nr * op_in_dim(p.g, op) * p.g.wbytes * op_mats(op);
        if (pid == 0) st_volatile_u64(&s.ctl->stream_pos, stream_bytes);
        if (!owns(j)) {
            ++j;
            return;
        }
        uint64_t *bar;
        uint8_t *dst = acquire(&bar);
        if (!dst) return;
        // the chunk's rows are contiguous (Q/K/V and gate/up are plan-packed): one copy
        const uint32_t bytes = nr * (uint32_t)op_in_dim(p.g, op) * (uint32_t)p.g.wbytes * (uint32_t)op_mats(op);
        mbar_expect_tx(bar, bytes);
        bulk_g2s(dst, gemv_src(op, layer, r0), bytes, bar, pol_weights);
        ++j;
    }

    // The whole block of kv_block positions from q0 (a multiple of kv_block)
    // of kv head `h`, as swizzled tiles of the K and V tensor maps: one box
    // per 64 dims, K boxes then V boxes. Rows past max_pos arrive as zeros;
    // rows from position P on are overwritten or zeroed by the consumer.
    __device__ void kv_chunk_tensor(int layer, int h, int q0) {
        if (!owns(j)) {
            ++j;
            return;
        }
        uint64_t *bar;
        uint8_t *dst = acquire(&bar);
        if (!dst) return;
        // the swizzle pattern assumes 1024-byte aligned boxes; never issue otherwise
        if (smem_u32(dst) & 1023u) {
            atomicOr(p.status, kDevBounds);
            ok = false;
            return;
        }
        const Geom &g = p.g;
        const int nb = g.d / 64;
        const uint32_t box = (uint32_t)g.kv_block * 128u;
        mbar_expect_tx(bar, 2u * (uint32_t)nb * box);
        const int z = layer * g.nkv + h;
        for (int i = 0; i < nb; ++i) {
            tensor_g2s_3d(dst + (size_t)i * box, &p.kv_map[0], 64 * i, q0, z, bar);
            tensor_g2s_3d(dst + (size_t)(nb + i) * box, &p.kv_map[1], 64 * i, q0, z, bar);
        }
        ++j;
    }

    // INT8 cache: the kv_block positions from q0 of kv head `h` as four tiles
    // (key codes [kv_block][d], value codes [d][kv_block], key scales, value
    // scales). Rows past the tensor arrive as zeros; positions from P on are
    // stale and are masked or overwritten by the consumer.
    __device__ void kv_chunk_q8(int layer, int h, int q0) {
        if (!owns(j)) {
            ++j;
            return;
        }
        uint64_t *bar;
        uint8_t *dst = acquire(&bar);
        if (!dst) return;
        if (smem_u32(dst) & 1023u) {
            atomicOr(p.status, kDevBounds);
            ok = false;
            return;
        }
        const Geom &g = p.g;
        const int z = layer * g.nkv + h;
        mbar_expect_tx(bar, (uint32_t)kv8_chunk_bytes(g.d));
        tensor_g2s_3d(dst, &p.kv_map[0], 0, q0, z, bar);
        tensor_g2s_3d(dst + 8192, &p.kv_map[1], q0, 0, z, bar);
        tensor_g2s_2d(dst + 16384, &p.kv_map[2], q0, z, bar);
        tensor_g2s_2d(dst + 16384 + g.kv_block * 4, &p.kv_map[3], q0, z, bar);
        ++j;
    }

    // K/V of positions written by step st-1 may be read only after this CTA's
    // consumers acquired the end of step st-1 (they publish that in step_ready).
    int ready = 0;
    __device__ bool kv_ready(int st) {
        if (ready >= st) return true;
        unsigned long long t0 = global_timer();
        for (uint32_t spin = 0;; ++spin) {
            ready = ld_acquire_cta(&s.ctl->step_ready);
            if (ready >= st) break;
            if ((spin & 15u) == 15u) {
                if (failed(p)) return false;
                if (global_timer() - t0 > p.timeout_ns) {
                    atomicOr(p.status, kDevTimeout);
                    return false;
                }
            }
        }
        // generic-proxy K/V writes of earlier steps, then async-proxy reads
        fence_proxy_async_global();
        return true;
    }

    // AK: attention kind of the kernel instance (0 shared chunks only, 1 also
    // one warp per chunk for long splits, 2 INT8 cache)
    template <int AK>
    __device__ __forceinline__ void run(int cta) {
        const Geom &g = p.g;
        const int t0 = p.offsets[cta], t1 = p.offsets[cta + 1];
        fence_proxy_async_global();
        for (int st = 0; st < p.n_steps && ok; ++st) {
            const int P = p.pos0 + st;
            for (int ti = t0; ti < t1 && ok; ++ti) {
                const tiles_task t = p.tasks[ti];
                unsigned long long *tr = pid == 0 ? trace_rec(p, cta, st, ti - t0) : nullptr;
                tracing = tr != nullptr;
                stall = 0;
                if (tr) tr[kTrProdFirst] = global_timer();
                if (op_is_gemv(t.op)) {
                    const uint32_t rpc = (uint32_t)op_rows_per_chunk(g, t.op);
                    for (uint32_t r = t.begin; r < t.end && ok; r += rpc) {
                        uint32_t nr = t.end - r < rpc ? t.end - r : rpc;
                        gemv_chunk(t.op, t.layer, r, nr);
                    }
                } else if (t.op == TILES_OP_ATTN) {
                    if (!kv_ready(st)) { ok = false; break; }
                    for (uint32_t it = t.begin; it < t.end && ok; ++it) {
                        const int h = (int)(it / (uint32_t)g.kv_splits);
                        const int c = (int)(it % (uint32_t)g.kv_splits);
                        int b0, b1;
                        attn_split_blocks(g, P + 1, c, &b0, &b1);
                        // whole blocks: positions from P on are overwritten,
                        // zeroed or masked by the consumer
                        for (int b = b0; b < b1 && ok; ++b) {
                            if (AK == 2)
                                kv_chunk_q8(t.layer, h, b * g.kv_block);
                            else
                                kv_chunk_tensor(t.layer, h, b * g.kv_block);
                        }
                    }
                }
                if (tr) {
                    tr[kTrProdLast] = global_timer();
                    tr[kTrProdStall] = stall;
                    tr[kTrOpInfo] = (unsigned long long)t.op | ((unsigned long long)t.layer << 8) |
                                    ((unsigned long long)task_chunks(g, t, P) << 32);
                }
            }
        }
        if (pid == 0) st_volatile_u64(&s.ctl->stream_pos, ~0ull);  // releases the prefetch warp
        // drain: wait for every copy still in flight so no bulk copy outlives the
        // CTA. An issued copy completes on its own (it waits on nothing but
        // memory), so this wait ends; it is bounded all the same, and running
        // out is reported like any other timeout.
        const uint32_t ns = (uint32_t)g.ring_slots;
        uint32_t first = j > ns ? j - ns : 0;
        for (uint32_t k = first; k < j; ++k) {
            if (!owns(k)) continue;
            unsigned long long t0n = global_timer();
            while (!mbar_try_wait(&s.full[k % ns], (k / ns) & 1u)) {
                if (global_timer() - t0n > p.timeout_ns) {
                    atomicOr(p.status, kDevTimeout);
                    break;
                }
            }
        }
    }
};

// ------------------------------------------------------------------ L2 prefetch warp
// Warms L2 with the loads of the dependency chain. While the weight stream
// saturates HBM, a copy the ring issues waits behind every copy in flight on
// the GPU (the rings alone hold about 3 us of HBM traffic), and on the chain
// Q/K/V -> attention -> O-projection that wait is pure latency. So the warp
// walks this CTA's tasks in the producers' order and prefetches into L2, one
// 128-byte line per lane, only the weight rows of the Q/K/V and O-projection
// tiles and the cached K/V of the attention tiles, once the producers are
// within l2_prefetch_bytes of weights of them: about one FFN phase ahead, so
// they are in L2 when the ring asks. Gate/up, down and LM-head rows are left
// to the ring (prefetching them too only adds DRAM traffic and congestion).
// Issue may be paced (a token bucket in global-timer nanoseconds). The warp
// never makes the kernel wait: when the producers finish or anything fails,
// it stops.
struct Prefetcher {
    const KernelParams &p;
    Smem &s;
    const int lane;
    unsigned long long next_ns = 0;

    __device__ Prefetcher(const KernelParams &p_, Smem &s_) : p(p_), s(s_), lane(threadIdx.x & 31) {}

    // false: stop prefetching (failure, or the producers stopped moving)
    __device__ bool wait_window(unsigned long long pos) {
        if (pos < ld_volatile_u64(&s.ctl->stream_pos) + p.l2_prefetch_bytes) return true;
        const unsigned long long t0 = global_timer();
        for (uint32_t spin = 1;; ++spin) {
            __nanosleep(64);
            const unsigned long long sp = ld_volatile_u64(&s.ctl->stream_pos);
            if (sp == ~0ull) return false;
            if (pos < sp + p.l2_prefetch_bytes) return true;
            if ((spin & 63u) == 0 && (failed(p) || global_timer() - t0 > p.timeout_ns)) return false;
        }
    }

    // lines [a, a + bytes) of one range, 4 KB per warp instruction
    __device__ bool range(const uint8_t *a, unsigned long long bytes, unsigned long long pos) {
        for (unsigned long long off = 0; off < bytes; off += 4096) {
            if (!wait_window(pos + off)) return false;
            if (p.l2_prefetch_ns_per_4k) {
                unsigned long long now = global_timer();
                const unsigned long long floor = now > 8ull * p.l2_prefetch_ns_per_4k ? now - 8ull * p.l2_prefetch_ns_per_4k : 0ull;
                if (next_ns < floor) next_ns = floor;  // at most 32 KB of burst credit
                while (now < next_ns) now = global_timer();
                next_ns += p.l2_prefetch_ns_per_4k;
            }
            const unsigned long long o = off + (unsigned long long)lane * 128u;
            if (o < bytes) prefetch_l2(a + o);
        }
        return true;
    }

    __device__ void run(int cta) {
        const Geom &g = p.g;
        const int t0 = p.offsets[cta], t1 = p.offsets[cta + 1];
        unsigned long long pos = 0;  // weight bytes of the tasks walked so far
        for (int st = 0; st < p.n_steps; ++st) {
            const int P = p.pos0 + st;
            for (int ti = t0; ti < t1; ++ti) {
                const tiles_task t = p.tasks[ti];
                if (failed(p)) return;
                if (op_is_gemv(t.op)) {
                    const unsigned long long rb = (unsigned long long)op_in_dim(g, t.op) * g.wbytes * op_mats(t.op);
                    const unsigned long long bytes = (unsigned long long)(t.end - t.begin) * rb;
                    if (t.op != TILES_OP_QKV && t.op != TILES_OP_OPROJ) {
                        pos += bytes;  // streaming tiles: left to the ring
                        continue;
                    }
                    const unsigned long long sp = ld_volatile_u64(&s.ctl->stream_pos);
                    if (sp == ~0ull) return;
                    // skip what the producers already handed to the ring
                    unsigned long long skip = sp > pos ? (sp - pos) & ~4095ull : 0ull;
                    if (skip < bytes) {
                        const LayerPtrs &lw = p.layers[t.layer];
                        const uint8_t *a = (t.op == TILES_OP_QKV ? lw.qkv : lw.o) + (size_t)t.begin * rb;
                        if (!range(a + skip, bytes - skip, pos + skip)) return;
                    }
                    pos += bytes;
                } else if (t.op == TILES_OP_ATTN && !g.kv8) {
                    // cached positions only: position P is written in this step
                    for (uint32_t it = t.begin; it < t.end; ++it) {
                        const int h = (int)(it / (uint32_t)g.kv_splits);
                        int b0, b1;
                        attn_split_blocks(g, P + 1, (int)(it % (uint32_t)g.kv_splits), &b0, &b1);
                        int q0 = b0 * g.kv_block, q1 = b1 * g.kv_block;
                        if (q1 > P) q1 = P;
                        if (q1 <= q0) continue;
                        const size_t off = ((size_t)(t.layer * g.nkv + h) * g.max_pos + q0) * g.d;
                        const unsigned long long n = (unsigned long long)(q1 - q0) * g.d * 2u;
                        if (!range(reinterpret_cast<const uint8_t *>(p.k_cache + off), n, pos)) return;
                        if (!range(reinterpret_cast<const uint8_t *>(p.v_cache + off), n, pos)) return;
                    }
                }
            }
        }
    }
};

// ------------------------------------------------------------------ GEMV rows
// NR rows (x MATS matrices) of one chunk against the input vector in shared
// memory: lane c reads 16-byte columns c, c+32, ... of every row, FP32 FMA,
// then an xor-shuffle reduction; lane r returns row r's sums. The row count is
// a compile-time constant so no predicated-off rows are issued.
template <int MATS, int NR>
__device__ __forceinline__ void gemv_rows(const uint8_t *slot, const uint4 *vec, int nu4,
                                          size_t row_bytes, int rpc, float (&res)[MATS]) {
    const int lane = threadIdx.x & 31;
    float acc[NR][MATS];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int m = 0; m < MATS; ++m) acc[r][m] = 0.f;
    for (int c = lane; c < nu4; c += 32) {
        float xf[8];
        unpack8(vec[c], xf);
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int m = 0; m < MATS; ++m) {
                // MATS == 2: gate row r at 2r, up row r at 2r + 1 (packed layout)
                const uint4 w = reinterpret_cast<const uint4 *>(slot + ((size_t)r * MATS + m) * row_bytes)[c];
                acc[r][m] = dot8(w, xf, acc[r][m]);
            }
    }
#pragma unroll
    for (int m = 0; m < MATS; ++m) res[m] = 0.f;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int m = 0; m < MATS; ++m) {
            const float v = warp_sum(acc[r][m]);
            if (lane == r) res[m] = v;
        }
}

template <int MATS>
__device__ __forceinline__ void gemv_rows_n(uint32_t nr, const uint8_t *slot, const uint4 *vec, int nu4,
                                            size_t row_bytes, int rpc, float (&res)[MATS]) {
    switch (nr) {
        case 1: gemv_rows<MATS, 1>(slot, vec, nu4, row_bytes, rpc, res); break;
        case 2: gemv_rows<MATS, 2>(slot, vec, nu4, row_bytes, rpc, res); break;
        case 3: gemv_rows<MATS, 3>(slot, vec, nu4, row_bytes, rpc, res); break;
        case 4: gemv_rows<MATS, 4>(slot, vec, nu4, row_bytes, rpc, res); break;
        case 5: gemv_rows<MATS, 5>(slot, vec, nu4, row_bytes, rpc, res); break;
        case 6: gemv_rows<MATS, 6>(slot, vec, nu4, row_bytes, rpc, res); break;
        case 7: gemv_rows<MATS, 7>(slot, vec, nu4, row_bytes, rpc, res); break;
        default: gemv_rows<MATS, 8>(slot, vec, nu4, row_bytes, rpc, res); break;
    }
}

// ------------------------------------------------------------------ INT8 GEMV rows
// Two FP32 lanes in one 64-bit register (low word first), for the paired
// FP32 instructions of sm_100 and later (one issue does two adds or FMAs).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ unsigned long long f2_pack_bits(uint32_t lo, uint32_t hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float f2_sum(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return __fadd_rn(lo, hi);
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Four INT8 codes of a word to exact floats, as two pairs: the plan stores
// each code q as the byte u = q + 128, the byte placed under the exponent of
// 2^23 is the float 2^23 + u, and subtracting 2^23 + 128 leaves q (both steps
// exact). Then 16 codes times 16 inputs (8 pairs), accumulated in FP32 on two
// lanes (even and odd elements); each product is exact.
__device__ __forceinline__ unsigned long long dot16_q8(const uint4 &w, const unsigned long long (&x)[8],
                                                       unsigned long long acc) {
    const unsigned long long bias = f2_pack(8388736.0f, 8388736.0f);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t u = ws[k];
        const unsigned long long f01 =
            f2_sub(f2_pack_bits(__byte_perm(u, 0x4B000000u, 0x7540), __byte_perm(u, 0x4B000000u, 0x7541)), bias);
        const unsigned long long f23 =
            f2_sub(f2_pack_bits(__byte_perm(u, 0x4B000000u, 0x7542), __byte_perm(u, 0x4B000000u, 0x7543)), bias);
        acc = f2_fma(f01, x[2 * k], acc);
        acc = f2_fma(f23, x[2 * k + 1], acc);
    }
    return acc;
}

// The INT8 form of gemv_rows: lane c reads the 16-code pieces c, c+32, ... of
// every row (16 bytes each) and the 16 matching BF16 inputs; lane r returns
// row r's unscaled sums (the epilogue applies the row scale).
template <int MATS, int NR>
__device__ __forceinline__ void gemv_rows_q8(const uint8_t *slot, const uint4 *vec, int n16,
                                             size_t row_bytes, float (&res)[MATS]) {
    const int lane = threadIdx.x & 31;
    unsigned long long acc[NR][MATS];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int m = 0; m < MATS; ++m) acc[r][m] = 0ull;
    for (int c = lane; c < n16; c += 32) {
        unsigned long long xp[8];
        {
            const uint4 a = vec[2 * c], b = vec[2 * c + 1];
            const uint32_t xs[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) xp[e] = f2_pack(bf_lo(xs[e]), bf_hi(xs[e]));
        }
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int m = 0; m < MATS; ++m) {
                const uint4 w = reinterpret_cast<const uint4 *>(slot + ((size_t)r * MATS + m) * row_bytes)[c];
                acc[r][m] = dot16_q8(w, xp, acc[r][m]);
            }
    }
#pragma unroll
    for (int m = 0; m < MATS; ++m) res[m] = 0.f;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int m = 0; m < MATS; ++m) {
            const float v = warp_sum(f2_sum(acc[r][m]));
            if (lane == r) res[m] = v;
        }
}

template <int MATS>
__device__ __forceinline__ void gemv_rows_q8_n(uint32_t nr, const uint8_t *slot, const uint4 *vec, int n16,
                                               size_t row_bytes, float (&res)[MATS]) {
    switch (nr) {
        case 1: gemv_rows_q8<MATS, 1>(slot, vec, n16, row_bytes, res); break;
        case 2: gemv_rows_q8<MATS, 2>(slot, vec, n16, row_bytes, res); break;
        case 3: gemv_rows_q8<MATS, 3>(slot, vec, n16, row_bytes, res); break;
        case 4: gemv_rows_q8<MATS, 4>(slot, vec, n16, row_bytes, res); break;
        case 5: gemv_rows_q8<MATS, 5>(slot, vec, n16, row_bytes, res); break;
        case 6: gemv_rows_q8<MATS, 6>(slot, vec, n16, row_bytes, res); break;
        case 7: gemv_rows_q8<MATS, 7>(slot, vec, n16, row_bytes, res); break;
        default: gemv_rows_q8<MATS, 8>(slot, vec, n16, row_bytes, res); break;
    }
}

// ------------------------------------------------------------------ consumers
struct Consumer {
    const KernelParams &p;
    Smem &s;
    const int tid, warp, lane;
    uint32_t j = 0;  // chunks consumed by the CTA (all warps keep the same count)
    int step = 0, P = 0;
    bool bad = false;  // this thread saw a timeout, an abort or a bad index

    __device__ Consumer(const KernelParams &p_, Smem &s_, int tid_)
        : p(p_), s(s_), tid(tid_), warp(tid_ >> 5), lane(tid_ & 31) {}

    // Chunk k lives in ring slot k % slots and is consumed by the warp that owns
    // that slot, (k % slots) % 8. One owner per slot means a warp only waits on
    // a slot after it released the slot's previous chunk itself, so the
    // mbarrier parity can never alias a chunk two ring laps ahead.
    __device__ bool mine(uint32_t k) const {
        return (int)((k % (uint32_t)p.g.ring_slots) % kConsumerWarps) == warp;
    }

    // slot of CTA chunk k, after its data landed; nullptr when aborting
    __device__ uint8_t *wait_chunk(uint32_t k) {
        const uint32_t ns = (uint32_t)p.g.ring_slots;
        uint32_t slot = k % ns;
        const bool ok = wait_mbar(p, &s.full[slot], (k / ns) & 1u);
        if (!__all_sync(0xFFFFFFFFu, ok)) {  // warp-uniform decision
            bad = true;
            return nullptr;
        }
        return s.ring + (size_t)slot * p.g.slot_bytes;
    }
    __device__ void release_chunk(uint32_t k) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[k % (uint32_t)p.g.ring_slots]);
    }

    __device__ int token_of_step(int st) {
        const int sg = p.step0 + st;
        int tok;
        if (sg < p.n_prompt) tok = p.prompt[sg];
        else if (st > 0) tok = key_row(__ldcg(&p.keys[st - 1]));
        else tok = __ldcg(&p.out_tokens[sg - p.n_prompt]);
        return tok;
    }

    // ---------------------------------------------------------- prologues
    // vec <- bf16(rmsnorm(src) * gain), src bf16 [n <= 8192] in global memory,
    // or (src null) already in vec; sum of squares in a fixed order, so every
    // CTA computes the same scale. One pass over src: each thread keeps its (at
    // most four) 16-byte pieces in registers.
    __device__ void rmsnorm_to_vec(const uint16_t *src, const uint16_t *gain, int n) {
        constexpr int kMaxU = 4;
        const int nu4 = n >> 3;
        uint4 v[kMaxU];
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxU; ++k) {
            const int c = tid + k * kConsumerWarps * 32;
            if (c < nu4) {
                v[k] = src ? __ldcg(reinterpret_cast<const uint4 *>(src) + c) : reinterpret_cast<const uint4 *>(s.vec)[c];
                float f[8];
                unpack8(v[k], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) s.ctl->red[warp] = ss;
        consumer_sync();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += s.ctl->red[w];
        const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)n), p.eps)));
        uint4 *dst = reinterpret_cast<uint4 *>(s.vec);
#pragma unroll
        for (int k = 0; k < kMaxU; ++k) {
            const int c = tid + k * kConsumerWarps * 32;
            if (c < nu4) {
                const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(gain) + c);
                float f[8], gf[8];
                unpack8(v[k], f);
                unpack8(gv, gf);
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint16_t lo = f2bf(__fmul_rn(__fmul_rn(f[2 * e], r), gf[2 * e]));
                    const uint16_t hi = f2bf(__fmul_rn(__fmul_rn(f[2 * e + 1], r), gf[2 * e + 1]));
                    o[e] = (uint32_t)lo | ((uint32_t)hi << 16);
                }
                dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }

    // residual rows [begin, end) into shared memory, for the epilogue: of the
    // embedding row (first layer), else of the tagged x words carrying `tag`
    __device__ void load_residual(const uint16_t *embed_row, uint32_t tag, uint32_t begin, uint32_t end) {
        uint16_t *res = reinterpret_cast<uint16_t *>(s.vec + p.res_off);
        for (uint32_t r = begin + tid; r < end; r += kConsumerWarps * 32) {
            if (embed_row) {
                res[r - begin] = __ldcg(&embed_row[r]);
                continue;
            }
            uint32_t w = ld_relaxed_u32(p.xw + r);
            Poll pl;
            while ((w >> 16) != tag) {
                if (bad || !pl.again(p)) {
                    bad = true;
                    break;
                }
                w = ld_relaxed_u32(p.xw + r);
            }
            res[r - begin] = (uint16_t)(w & 0xFFFFu);
        }
    }

    __device__ uint32_t tag(int layer, int kind) const { return act_tag(p, step, layer, kind); }

    // vec[0, n) (bf16) <- the tagged words src[0, n), n a multiple of 8, each
    // polled until it carries `tg`. First pass: four 8-word pieces per thread
    // in flight, the ready ones stored; then the stale ones are polled.
    __device__ void gather_tagged(const uint32_t *src, int n, uint32_t tg) {
        constexpr int B = 4;
        const int n8 = n >> 3;
        uint4 *dst = reinterpret_cast<uint4 *>(s.vec);
        for (int c0 = tid; c0 < n8; c0 += B * kConsumerWarps * 32) {
            uint32_t stale = 0;
#pragma unroll
            for (int k = 0; k < B; ++k) {
                const int c = c0 + k * kConsumerWarps * 32;
                if (c < n8) {
                    const uint4 lo = ld_relaxed_v4(src + 8 * c), hi = ld_relaxed_v4(src + 8 * c + 4);
                    if (tags_ok4(lo, tg) && tags_ok4(hi, tg)) dst[c] = untag8(lo, hi);
                    else stale |= 1u << k;
                }
            }
            for (int k = 0; stale != 0; ++k, stale >>= 1) {
                if (!(stale & 1u)) continue;
                const int c = c0 + k * kConsumerWarps * 32;
                Poll pl;
                uint4 lo, hi;
                do {
                    if (bad || !pl.again(p)) {
                        bad = true;
                        break;
                    }
                    lo = ld_relaxed_v4(src + 8 * c);
                    hi = ld_relaxed_v4(src + 8 * c + 4);
                } while (!(tags_ok4(lo, tg) && tags_ok4(hi, tg)));
                if (!bad) dst[c] = untag8(lo, hi);
            }
        }
    }

    // One output row of a GEMV task, from its MATS dot products: the fused
    // epilogue of the op (residual add, SwiGLU, logits store).
    template <int MATS>
    __device__ void emit_row(int op, const tiles_task &t, uint32_t row, const float (&v)[MATS]) {
        switch (op) {
            case TILES_OP_QKV:
                st_relaxed_u64(p.qkvw + row, ((unsigned long long)tag(t.layer, kTagQKV) << 32) | __float_as_uint(v[0]));
                break;
            case TILES_OP_OPROJ:
            case TILES_OP_DOWN: {  // residual rows were loaded in the prologue
                const uint16_t xb = reinterpret_cast<const uint16_t *>(s.vec + p.res_off)[row - t.begin];
                const uint32_t tg = tag(t.layer, op == TILES_OP_OPROJ ? kTagXAttn : kTagXFfn);
                st_relaxed_u32(p.xw + row, (tg << 16) | f2bf(__fadd_rn(bf2f(xb), v[0])));
                break;
            }
            case TILES_OP_GATEUP: {
                const float gt = v[0];
                const float silu = __fdiv_rn(gt, __fadd_rn(1.0f, expf(-gt)));
                st_relaxed_u32(p.aw + row, (tag(t.layer, kTagA) << 16) | f2bf(__fmul_rn(silu, v[MATS - 1])));
                break;
            }
            case TILES_OP_LMHEAD:
                if (p.out_logits) __stcg(&p.out_logits[(size_t)(p.step0 + step) * p.g.V + row], v[0]);
                break;
        }
    }

    // Chunk k goes to the warp that owns its slot, which reduces it alone; the
    // warps work on different chunks at once.
    template <int MATS, bool Q8>
    __device__ void gemv_task(const tiles_task &t) {
        const Geom &g = p.g;
        const int op = t.op;
        const int in = op_in_dim(g, op);
        const int nu4 = in >> 3;
        const float *scale = nullptr;  // INT8: one FP32 scale per streamed row
        if constexpr (Q8) {
            const LayerPtrs &lw = p.layers[t.layer];
            scale = op == TILES_OP_QKV ? lw.s_qkv : op == TILES_OP_OPROJ ? lw.s_o
                  : op == TILES_OP_GATEUP ? lw.s_gu : op == TILES_OP_DOWN ? lw.s_down : p.lm_s;
        }
        const uint32_t rpc = (uint32_t)op_rows_per_chunk(g, op);
        const uint32_t nchunks = (t.end - t.begin + rpc - 1) / rpc;
        const uint4 *vec = reinterpret_cast<const uint4 *>(s.vec);
        unsigned long long best = 0;
        for (uint32_t k = 0; k < nchunks; ++k) {
            const uint32_t jj = j + k;
            if (!mine(jj)) continue;
            const uint32_t r0 = t.begin + k * rpc;
            const uint32_t nr = t.end - r0 < rpc ? t.end - r0 : rpc;
            float sc[MATS];  // INT8: the row scales load while the chunk arrives
            if constexpr (Q8) {
                const uint32_t row = r0 + ((uint32_t)lane < nr ? lane : 0);
#pragma unroll
                for (int m = 0; m < MATS; ++m)  // gate/up: packed rows 2 row, 2 row + 1
                    sc[m] = __ldg(scale + (MATS == 2 ? 2 * row + m : row));
            }
            const uint8_t *slot = wait_chunk(jj);
            if (!slot) break;
            if (k == 0 && cur_tr && lane == 0) cur_tr[kTrFirstChunk] = global_timer();
            float mine[MATS];
            if constexpr (Q8) {
                gemv_rows_q8_n<MATS>(nr, slot, vec, in >> 4, (size_t)in, mine);
            } else {
                gemv_rows_n<MATS>(nr, slot, vec, nu4, (size_t)in * 2, (int)rpc, mine);
            }
            release_chunk(jj);
            if constexpr (Q8) {
#pragma unroll
                for (int m = 0; m < MATS; ++m) mine[m] = __fmul_rn(mine[m], sc[m]);
            }
            if ((uint32_t)lane < nr) emit_row<MATS>(op, t, r0 + lane, mine);
            if (op == TILES_OP_LMHEAD) {
                unsigned long long key = (uint32_t)lane < nr ? argmax_key(mine[0], r0 + lane) : 0ull;
                key = warp_max_u64(key);
                best = key > best ? key : best;
            }
        }
        j += nchunks;
        if (op == TILES_OP_LMHEAD) {
            if (lane == 0) s.ctl->warp_key[warp] = best;
            consumer_sync();
            if (tid == 0) {
                unsigned long long b = 0;
                for (int w = 0; w < kConsumerWarps; ++w) b = s.ctl->warp_key[w] > b ? s.ctl->warp_key[w] : b;
                atomicMax(&p.keys[step], b);
            }
        }
    }

    // ---------------------------------------------------------- attention
    // Layout of the vec region during attention tasks.
    struct AttnSmem {
        uint16_t *knew;    // [d]
        uint16_t *vnew;    // [d]
        float *wstate;     // [warps][G][4 + d]
        uint16_t *qh;      // [G][d + 8] bf16 q (rows padded: conflict-free MMA fragment loads)
        int8_t *k8, *v8;   // INT8 cache: codes of the new key (minus mu) and value rows [d]
        float *s8;         // and their scales [2]
    };
    __device__ AttnSmem attn_smem() const {
        const Geom &g = p.g;
        AttnSmem a;
        uint8_t *b = s.vec;
        a.knew = reinterpret_cast<uint16_t *>(b);
        b += (size_t)g.d * 2;
        a.vnew = reinterpret_cast<uint16_t *>(b);
        b += (size_t)g.d * 2;
        a.wstate = reinterpret_cast<float *>(b);
        b += (size_t)kConsumerWarps * g.G * (kPartialPad + g.d) * 4;
        a.qh = reinterpret_cast<uint16_t *>(b);
        b += (size_t)g.G * (g.d + 8) * 2;
        a.k8 = reinterpret_cast<int8_t *>(b);
        a.v8 = a.k8 + g.d;
        a.s8 = reinterpret_cast<float *>(b + 2 * g.d);
        return a;
    }

    // q heads of kv head h (and k, v of head h): optional RMSNorm over the head,
    // RoPE at position P, rounding to bf16. One warp per head.
    // One row of the INT8 cache from its FP32 values x (lane holds elements
    // lane + 32 e): s = max |x| / 127, codes x / s rounded to nearest even and
    // clamped to +-127, all FP32 (an all-zero row: s = 0, codes 0).
    template <int E>
    __device__ __forceinline__ void quantize_row8(const float (&x)[E], int8_t *codes, float *scale) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
        amax = warp_max(amax);
        const float sc = __fdiv_rn(amax, 127.0f);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float qf = sc > 0.f ? rintf(__fdiv_rn(x[e], sc)) : 0.f;
            qf = fminf(fmaxf(qf, -127.f), 127.f);
            codes[lane + 32 * e] = (int8_t)qf;
        }
        if (lane == 0) *scale = sc;
    }

    template <int D, int AK>
    __device__ void prep_qkv(int h, const AttnSmem &a) {
        constexpr bool KV8 = AK == 2;
        const Geom &g = p.g;
        const LayerPtrs &lw = p.layers[cur_layer];
        const float *cs = p.rope_cos + (size_t)P * (D / 2);
        const float *sn = p.rope_sin + (size_t)P * (D / 2);
        constexpr int E = D / 32;  // elements per lane: lane, lane+32, ...
        for (int hh = warp; hh < g.G + 2; hh += kConsumerWarps) {
            const bool is_q = hh < g.G, is_k = hh == g.G;
            const int row0 = is_q ? (h * g.G + hh) * D
                                  : (is_k ? g.qd + h * D : g.qd + g.kvd + h * D);
            float v[E];
            {
                const uint32_t tg = tag(cur_layer, kTagQKV);
                unsigned long long w[E];
#pragma unroll
                for (int e = 0; e < E; ++e) w[e] = ld_relaxed_u64(p.qkvw + row0 + lane + 32 * e);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    Poll pl;
                    while ((uint32_t)(w[e] >> 32) != tg) {
                        if (bad || !pl.again(p)) {
                            bad = true;
                            break;
                        }
                        w[e] = ld_relaxed_u64(p.qkvw + row0 + lane + 32 * e);
                    }
                    v[e] = __uint_as_float((uint32_t)w[e]);
                }
            }
            if (!is_q && !is_k) {
#pragma unroll
                for (int e = 0; e < E; ++e) a.vnew[lane + 32 * e] = f2bf(v[e]);
                if (KV8) {
#pragma unroll
                    for (int e = 0; e < E; ++e) v[e] = round_bf(v[e]);
                    quantize_row8<E>(v, a.v8, &a.s8[1]);
                }
                continue;
            }
            if (p.qk_norm) {
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
                ss = warp_sum(ss);
                const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)D), p.eps)));
                const uint16_t *gn = is_q ? lw.q_norm : lw.k_norm;
#pragma unroll
                for (int e = 0; e < E; ++e) v[e] = __fmul_rn(__fmul_rn(v[e], r), bf2f(gn[lane + 32 * e]));
            }
            // rotate-half: element j pairs with j + D/2 (both held by this lane)
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                const int jx = lane + 32 * e;
                const float c = cs[jx], sv = sn[jx];
                const float x0 = v[e], x1 = v[e + E / 2];
                v[e] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sv));
                v[e + E / 2] = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, sv));
            }
            if (is_q) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    a.qh[hh * (D + 8) + lane + 32 * e] = f2bf(v[e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) a.knew[lane + 32 * e] = f2bf(v[e]);
                if (KV8) {
                    // the cached key is the rounded key minus this head's shift mu
                    const float *mu = p.mu8 + (size_t)(cur_layer * g.nkv + h) * D;
#pragma unroll
                    for (int e = 0; e < E; ++e) v[e] = __fsub_rn(round_bf(v[e]), mu[lane + 32 * e]);
                    quantize_row8<E>(v, a.k8, &a.s8[0]);
                }
            }
        }
    }

    int cur_layer = 0;
    unsigned long long *cur_tr = nullptr;  // trace record of the running task, or null

    // One chunk of positions [q0, q0 + npos) for the G q heads of one kv head,
    // on the tensor cores (the chunk arrived as swizzled K and V tiles), with
    // positions as the 16 rows of the m16n8k16 A operand and the q heads as
    // the 8 columns of B (columns >= G are zero). A 16-position block takes
    // d/16 MMAs for s^T = K q^T and 2 d/16 for o^T += V^T p^T: half of what
    // q heads as A rows take, since G <= 8 rows of 16 would be used there.
    // Lane (g, t) = (lane / 4, lane % 4) holds the scores of positions g and
    // g + 8 of each block for heads 2t and 2t + 1, and their running m and l
    // (l summed over this lane's positions only, reduced over g at the end).
    // A round takes NP blocks from block grp0 on, and the next round starts
    // grp_step rounds later: (NP, 0, 1) walks the whole chunk (2048 / D
    // positions a round), (1, w, 8) gives warp w every eighth block. Per round:
    //   s = K q^T (FP32, exact BF16 products), masked past npos, times d^-1/2;
    //   m' = max(m, max over positions), c = e^(m - m'), p = e^(s - m'),
    //   l' = c l + sum p, o' = c o;
    //   p^T becomes B fragments by one movmatrix.trans per 8 x 8 block, as a
    //   BF16 high part and a BF16 remainder (two MMAs, ~16 bits kept);
    //   o^T += V^T p^T with V^T's fragments from transposed ldmatrix of V.
    // o[mt] holds (dims 16 mt + g and 16 mt + g + 8) x (heads 2t, 2t + 1).
    template <int D, int G, int NP>
    __device__ __forceinline__ void attn_chunk_mma(const uint8_t *slot, int npos, const uint32_t *qcol, bool qcol_ok,
                                                   float (&m)[2], float (&l)[2], float (&o)[D / 16][4], int grp0,
                                                   int grp_step) {
        constexpr int SUB = 16 * NP;  // positions per round (NP 16-position blocks)
        constexpr int KS = D / 16;     // k-steps of the scores
        constexpr int MT = D / 16;     // 16-dim row tiles of o^T
        const int kvb = p.g.kv_block;
        const uint32_t kb = smem_u32(slot), vb = kb + (uint32_t)kvb * D * 2;
        const int g8 = lane >> 2;
        const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix and row this lane points at
        for (int p0 = grp0 * SUB; p0 < npos; p0 += grp_step * SUB) {
            float s[NP][4];
#pragma unroll
            for (int pt = 0; pt < NP; ++pt) {
                s[pt][0] = s[pt][1] = s[pt][2] = s[pt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    // rows 0-7 / 8-15 of the block, dims 16 ks .. + 7 / + 8 .. + 15
                    uint32_t a[4];
                    ldsm_x4(kb + swz_off(kvb, p0 + 16 * pt + 8 * (mi & 1) + ri, 2 * ks + (mi >> 1)), a);
                    const uint32_t b0 = qcol_ok ? qcol[8 * ks] : 0u, b1 = qcol_ok ? qcol[8 * ks + 4] : 0u;
                    mma_m16n8k16(s[pt], a[0], a[1], a[2], a[3], b0, b1);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int pt = 0; pt < NP; ++pt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const bool ok = p0 + 16 * pt + 8 * hr + g8 < npos;
                    s[pt][2 * hr] = ok ? s[pt][2 * hr] * p.attn_scale : -INFINITY;
                    s[pt][2 * hr + 1] = ok ? s[pt][2 * hr + 1] * p.attn_scale : -INFINITY;
                    mx0 = fmaxf(mx0, s[pt][2 * hr]);
                    mx1 = fmaxf(mx1, s[pt][2 * hr + 1]);
                }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
            }
            const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
            const float c0 = expf(m[0] - mn0), c1 = expf(m[1] - mn1);
            float ls0 = 0.f, ls1 = 0.f;
            uint32_t bh[NP][2], bl[NP][2];
#pragma unroll
            for (int pt = 0; pt < NP; ++pt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const float pa = expf(s[pt][2 * hr] - mn0), pb = expf(s[pt][2 * hr + 1] - mn1);
                    ls0 += pa;
                    ls1 += pb;
                    const uint16_t ha = f2bf(pa), hb = f2bf(pb);
                    const uint16_t ra = f2bf(__fsub_rn(pa, bf2f(ha))), rb = f2bf(__fsub_rn(pb, bf2f(hb)));
                    bh[pt][hr] = movmatrix_t((uint32_t)ha | ((uint32_t)hb << 16));
                    bl[pt][hr] = movmatrix_t((uint32_t)ra | ((uint32_t)rb << 16));
                }
            l[0] = fmaf(l[0], c0, ls0);
            l[1] = fmaf(l[1], c1, ls1);
            m[0] = mn0;
            m[1] = mn1;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[mt][0] *= c0;
                o[mt][1] *= c1;
                o[mt][2] *= c0;
                o[mt][3] *= c1;
            }
#pragma unroll
            for (int pt = 0; pt < NP; ++pt)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    // V^T (dims 16 mt.., positions 16 pt..): transposed loads of V blocks
                    // (positions block mi >> 1, dims block mi & 1)
                    uint32_t a[4];
                    ldsm_x4_t(vb + swz_off(kvb, p0 + 16 * pt + 8 * (mi >> 1) + ri, 2 * mt + (mi & 1)), a);
                    mma_m16n8k16(o[mt], a[0], a[1], a[2], a[3], bh[pt][0], bh[pt][1]);
                    mma_m16n8k16(o[mt], a[0], a[1], a[2], a[3], bl[pt][0], bl[pt][1]);
                }
        }
    }

    // The INT8-cache form of attn_chunk_mma (positions as A rows, q heads as B
    // columns). The chunk holds key codes [kvb][D] and value codes transposed
    // [D][kvb] (swizzled tiles), then the key and value scales. A 32-bit
    // ldmatrix word is four codes: of four consecutive dims of one position
    // (keys) or four consecutive positions of one dim (values). They become
    // the A fragment's k slots 2t, 2t+1, 2t+8, 2t+9, so:
    //   - q's B fragment takes dims 4t..4t+3 of each 16 in the same slots
    //     (words 2t and 2t+1 of the k-step: a consistent permutation of the
    //     summed dims);
    //   - row r of a 16-position score block is position 4 (r mod 8 / 2) +
    //     (r & 1) + 2 (r / 8) (the ldmatrix row addresses choose it), so that
    //     after movmatrix.trans a lane's p fragment covers exactly the four
    //     positions 4t..4t+3 its value words hold.
    // Key scales multiply the score rows after the MMA; value scales fold into
    // p (masked positions get exact zeros, so stale codes and scales past npos
    // never reach the sums); l sums the unscaled p.
    // A round is NP 16-position blocks; this warp takes rounds grp0,
    // grp0 + grp_step, ... of the chunk (all of them when it owns the chunk;
    // one block in eight when all warps share a chunk of a short split).
    template <int D, int G, int NP>
    __device__ __forceinline__ void attn_chunk_mma_q8(const uint8_t *slot, int npos, const uint32_t *qcol,
                                                      bool qcol_ok, float (&m)[2], float (&l)[2],
                                                      float (&o)[D / 16][4], int grp0, int grp_step) {
        constexpr int KVB = 8192 / D;  // positions per chunk; also the value tile's row bytes
        constexpr int SUB = 16 * NP;   // positions per round
        constexpr int KU = D / 16;     // 16-byte units of a key row (= k-steps)
        constexpr int MT = D / 16;     // 16-dim row tiles of o^T
        const uint32_t kb = smem_u32(slot), vb = kb + 8192u;
        const float *ksc = reinterpret_cast<const float *>(slot + 16384);
        const float *vsc = ksc + KVB;
        const int g8 = lane >> 2;
        const int mi = lane >> 3, ri = lane & 7;
        const int kr_off = 4 * (ri >> 1) + (ri & 1) + 2 * (mi & 1);  // position of the row this lane addresses
        const int my_off = 4 * (g8 >> 1) + (g8 & 1);                 // position of this lane's row g (+2: row g + 8)
        for (int p0 = grp0 * SUB; p0 < npos; p0 += grp_step * SUB) {
            float s[NP][4];
#pragma unroll
            for (int pt = 0; pt < NP; ++pt) {
                s[pt][0] = s[pt][1] = s[pt][2] = s[pt][3] = 0.f;
#pragma unroll
                for (int u0 = 0; u0 < KU; u0 += 2) {
                    // words: rows 0-7 / 8-15 of the block, units u0 and u0 + 1
                    uint32_t w[4];
                    ldsm_x4(kb + swz8_off<D>(p0 + 16 * pt + kr_off, u0 + (mi >> 1)), w);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int ks = u0 + i;
                        uint32_t a0, a1, a2, a3;
                        codes_bf16x2(w[2 * i], a0, a2);
                        codes_bf16x2(w[2 * i + 1], a1, a3);
                        const uint32_t b0 = qcol_ok ? qcol[8 * ks] : 0u, b1 = qcol_ok ? qcol[8 * ks + 1] : 0u;
                        mma_m16n8k16(s[pt], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
            float vs[NP][2];
#pragma unroll
            for (int pt = 0; pt < NP; ++pt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int pos = p0 + 16 * pt + my_off + 2 * hr;
                    const bool ok = pos < npos;
                    const float kscale = ksc[pos];
                    vs[pt][hr] = ok ? vsc[pos] : 0.f;
                    s[pt][2 * hr] = ok ? (s[pt][2 * hr] * kscale) * p.attn_scale : -INFINITY;
                    s[pt][2 * hr + 1] = ok ? (s[pt][2 * hr + 1] * kscale) * p.attn_scale : -INFINITY;
                    mx0 = fmaxf(mx0, s[pt][2 * hr]);
                    mx1 = fmaxf(mx1, s[pt][2 * hr + 1]);
                }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
            }
            const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
            const float c0 = expf(m[0] - mn0), c1 = expf(m[1] - mn1);
            float ls0 = 0.f, ls1 = 0.f;
            uint32_t bh[NP][2], bl[NP][2];
#pragma unroll
            for (int pt = 0; pt < NP; ++pt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const float pa = expf(s[pt][2 * hr] - mn0), pb = expf(s[pt][2 * hr + 1] - mn1);
                    ls0 += pa;
                    ls1 += pb;
                    const float wa = pa * vs[pt][hr], wb = pb * vs[pt][hr];
                    const uint16_t ha = f2bf(wa), hb = f2bf(wb);
                    const uint16_t ra = f2bf(__fsub_rn(wa, bf2f(ha))), rb = f2bf(__fsub_rn(wb, bf2f(hb)));
                    bh[pt][hr] = movmatrix_t((uint32_t)ha | ((uint32_t)hb << 16));
                    bl[pt][hr] = movmatrix_t((uint32_t)ra | ((uint32_t)rb << 16));
                }
            l[0] = fmaf(l[0], c0, ls0);
            l[1] = fmaf(l[1], c1, ls1);
            m[0] = mn0;
            m[1] = mn1;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[mt][0] *= c0;
                o[mt][1] *= c1;
                o[mt][2] *= c0;
                o[mt][3] *= c1;
            }
#pragma unroll
            for (int pt = 0; pt < NP; ++pt)
#pragma unroll
                for (int mt = 0; mt < MT; mt += 2) {
                    // words: dims 16 mt + 0..7, + 8..15, 16 (mt + 1) + 0..7, + 8..15; positions 16 pt ..
                    uint32_t w[4];
                    ldsm_x4(vb + swz8_off<KVB>(16 * mt + 8 * mi + ri, (p0 >> 4) + pt), w);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        uint32_t a0, a1, a2, a3;
                        codes_bf16x2(w[2 * i], a0, a2);
                        codes_bf16x2(w[2 * i + 1], a1, a3);
                        mma_m16n8k16(o[mt + i], a0, a1, a2, a3, bh[pt][0], bh[pt][1]);
                        mma_m16n8k16(o[mt + i], a0, a1, a2, a3, bl[pt][0], bl[pt][1]);
                    }
                }
        }
    }

    // The swizzled form: row r = P - q0 of the chunk gets the new K and V, and
    // the V rows after it (stale cache memory, which may hold any bits) become
    // zeros, so the masked positions add exact zeros to p V.
    template <int D>
    __device__ __forceinline__ void place_new_kv_swz(uint8_t *slot, int q0) {
        const int kvb = p.g.kv_block;
        const AttnSmem a = attn_smem();
        const int r = P - q0;
        uint8_t *vs = slot + (size_t)kvb * D * 2;
        for (int e = lane; e < D; e += 32) {
            const uint32_t off = swz_off(kvb, r, e >> 3) + (uint32_t)(e & 7) * 2u;
            *reinterpret_cast<uint16_t *>(slot + off) = a.knew[e];
            *reinterpret_cast<uint16_t *>(vs + off) = a.vnew[e];
        }
        const int nz = (kvb - r - 1) * (D / 8);  // 16-byte units of the rows after r
        for (int i = lane; i < nz; i += 32) {
            const int rr = r + 1 + i / (D / 8), u = i % (D / 8);
            *reinterpret_cast<uint4 *>(vs + swz_off(kvb, rr, u)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
    }

    // The INT8 form: row r = P - q0 of the chunk gets the new key codes (one
    // row of the key tile), value codes (one column of the transposed value
    // tile) and both scales. The other stale rows stay: they are masked.
    template <int D>
    __device__ __forceinline__ void place_new_kv_q8(uint8_t *slot, int q0) {
        constexpr int KVB = 8192 / D;
        const AttnSmem a = attn_smem();
        const int r = P - q0;
        uint8_t *vt = slot + 8192;
        float *ksc = reinterpret_cast<float *>(slot + 16384);
        for (int e = lane; e < D; e += 32) {
            slot[swz8_off<D>(r, e >> 4) + (e & 15)] = (uint8_t)a.k8[e];
            vt[swz8_off<KVB>(e, r >> 4) + (r & 15)] = (uint8_t)a.v8[e];
        }
        if (lane == 0) {
            ksc[r] = a.s8[0];
            ksc[KVB + r] = a.s8[1];
        }
        fence_proxy_async_smem();
        __syncwarp();
    }

    template <int D, int G, int AK>
    __device__ void attn_task(const tiles_task &t) {
        constexpr bool MMA = AK >= 1, KV8 = AK == 2;
        const Geom &g = p.g;
        const AttnSmem a = attn_smem();
        int prepared = -1;
        for (uint32_t it = t.begin; it < t.end; ++it) {
            const int h = (int)(it / (uint32_t)g.kv_splits);
            const int c = (int)(it % (uint32_t)g.kv_splits);
            if (h != prepared) {
                consumer_sync();  // previous item finished reading q / knew / vnew
                prep_qkv<D, AK>(h, a);
                consumer_sync();
                if (cur_tr && tid == 0 && prepared < 0) cur_tr[kTrPrologue] = global_timer();
                prepared = h;
            }
            int b0, b1;
            attn_split_blocks(g, P + 1, c, &b0, &b1);
            const int pb = P / g.kv_block;
            const bool has_new = pb >= b0 && pb < b1;
            if (has_new && tid < D) {
                // the one tile whose range holds position P writes the new K/V
                if (KV8) {
                    const size_t z = (size_t)(cur_layer * g.nkv + h);
                    p.kq8[(z * g.kv_mp + P) * D + tid] = a.k8[tid];
                    p.vq8[(z * D + tid) * g.kv_mp + P] = a.v8[tid];
                    if (tid == 0) {
                        p.ks8[z * g.kv_mp + P] = a.s8[0];
                        p.vs8[z * g.kv_mp + P] = a.s8[1];
                    }
                } else {
                    const size_t off = ((size_t)(cur_layer * g.nkv + h) * g.max_pos + P) * D + tid;
                    p.k_cache[off] = a.knew[tid];
                    p.v_cache[off] = a.vnew[tid];
                }
                fence_proxy_async_global();
            }
            const uint32_t nch = (uint32_t)(b1 - b0);
            {
                // tensor cores: every q head of the group as a B column
                const int g8 = lane >> 2, t4 = lane & 3;
                // q head g8 as BF16 pairs (dims 2t4 + 16ks (+8) in word t4 + 8ks (+4))
                // (the INT8 form reads words 2 t4 and 2 t4 + 1 of each k-step instead)
                const uint32_t *qcol = reinterpret_cast<const uint32_t *>(a.qh + (size_t)(g8 < G ? g8 : 0) * (D + 8)) +
                                       (KV8 ? 2 * t4 : t4);
                float mm[2] = {-INFINITY, -INFINITY}, ll[2] = {0.f, 0.f}, oo[D / 16][4];
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) oo[mt][0] = oo[mt][1] = oo[mt][2] = oo[mt][3] = 0.f;
                if (KV8 && nch < (uint32_t)kConsumerWarps) {
                    // a short split (INT8 cache): every warp works on every chunk,
                    // one 16-position block in eight each; the chunk is released
                    // once all warps are done with it
                    for (uint32_t k = 0; k < nch; ++k) {
                        const uint32_t jj = j + k;
                        uint8_t *slot = wait_chunk(jj);
                        const int q0 = (b0 + (int)k) * g.kv_block;
                        int q1 = q0 + g.kv_block;
                        if (q1 > P + 1) q1 = P + 1;
                        if (slot && warp == 0 && q0 <= P && P < q1) place_new_kv_q8<D>(slot, q0);
                        if (consumer_sync_or(bad)) break;
                        attn_chunk_mma_q8<D, G, 1>(slot, q1 - q0, qcol, g8 < G, mm, ll, oo, warp, kConsumerWarps);
                        consumer_sync();
                        if (tid == 0) mbar_arrive(&s.empty[jj % (uint32_t)g.ring_slots]);
                    }
                } else if (!KV8 && !(MMA && attn_owner(g, (int)nch))) {
                    // a short split (BF16 cache): all warps work on each group of
                    // resident chunks (at most a ring's worth), one 16-position
                    // block per warp and round, the group's blocks numbered across
                    // its chunks; the group is released once all warps are done
                    const uint32_t ns = (uint32_t)g.ring_slots;
                    const int nb = g.kv_block / 16;
                    for (uint32_t k0 = 0; k0 < nch; k0 += ns) {
                        const uint32_t kn = nch - k0 < ns ? nch - k0 : ns;
                        for (uint32_t k = k0; k < k0 + kn; ++k) {
                            uint8_t *slot = wait_chunk(j + k);
                            if (k == 0 && cur_tr && tid == 0 && it == t.begin) cur_tr[kTrFirstChunk] = global_timer();
                            const int q0 = (b0 + (int)k) * g.kv_block;
                            if (slot && warp == 0 && q0 <= P && P < q0 + g.kv_block) place_new_kv_swz<D>(slot, q0);
                        }
                        if (consumer_sync_or(bad)) break;
                        for (uint32_t k = k0; k < k0 + kn; ++k) {
                            const uint8_t *slot = s.ring + (size_t)((j + k) % ns) * g.slot_bytes;
                            const int q0 = (b0 + (int)k) * g.kv_block;
                            int q1 = q0 + g.kv_block;
                            if (q1 > P + 1) q1 = P + 1;
                            // group block (k - k0) nb + b goes to warp (k - k0) nb + b mod 8
                            const int first = ((warp - (int)(k - k0) * nb) % kConsumerWarps + kConsumerWarps) %
                                              kConsumerWarps;
                            attn_chunk_mma<D, G, 1>(slot, q1 - q0, qcol, g8 < G, mm, ll, oo, first, kConsumerWarps);
                        }
                        consumer_sync();
                        if (tid == 0)
                            for (uint32_t k = k0; k < k0 + kn; ++k) mbar_arrive(&s.empty[(j + k) % ns]);
                    }
                } else if constexpr (MMA) {
                    // a long split: each chunk to its slot's owner warp
                    for (uint32_t k = 0; k < nch; ++k) {
                        const uint32_t jj = j + k;
                        if (!mine(jj)) continue;
                        uint8_t *slot = wait_chunk(jj);
                        if (!slot) break;
                        const int q0 = (b0 + (int)k) * g.kv_block;
                        int q1 = q0 + g.kv_block;
                        if (q1 > P + 1) q1 = P + 1;
                        if (KV8) {
                            if (q0 <= P && P < q1) place_new_kv_q8<D>(slot, q0);
                            attn_chunk_mma_q8<D, G, 2048 / D / 16>(slot, q1 - q0, qcol, g8 < G, mm, ll, oo, 0, 1);
                        } else {
                            if (q0 <= P && P < q1) place_new_kv_swz<D>(slot, q0);
                            attn_chunk_mma<D, G, 2048 / D / 16>(slot, q1 - q0, qcol, g8 < G, mm, ll, oo, 0, 1);
                        }
                        release_chunk(jj);
                    }
                }
                // per-warp states -> shared memory: l summed over the lanes of a
                // head (lanes with the same t), then heads 2 t4 and 2 t4 + 1
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    ll[0] += __shfl_xor_sync(0xFFFFFFFFu, ll[0], off);
                    ll[1] += __shfl_xor_sync(0xFFFFFFFFu, ll[1], off);
                }
                float *ws = a.wstate + (size_t)warp * G * (kPartialPad + D);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int hh = 2 * t4 + e;
                    if (hh >= G) continue;
                    float *w = ws + (size_t)hh * (kPartialPad + D);
                    if (g8 == 0) {
                        w[0] = mm[e];
                        w[1] = ll[e];
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        w[kPartialPad + 16 * mt + g8] = oo[mt][e];
                        w[kPartialPad + 16 * mt + g8 + 8] = oo[mt][2 + e];
                    }
                }
            }
            j += nch;
            // per-warp states -> one partial for (q heads, split c): first each
            // (head, warp) state's weight e^(m_w - M) into word 2 of the state
            // (0 for a head no warp saw), then the outputs
            consumer_sync();
            if (tid < G * kConsumerWarps) {
                const int i = tid / kConsumerWarps, w = tid % kConsumerWarps;
                float M = -INFINITY;
                for (int v = 0; v < kConsumerWarps; ++v)
                    M = fmaxf(M, a.wstate[((size_t)v * G + i) * (kPartialPad + D)]);
                float *st = a.wstate + ((size_t)w * G + i) * (kPartialPad + D);
                st[2] = M == -INFINITY ? 0.f : expf(st[0] - M);
                st[3] = M;
            }
            consumer_sync();
            for (int idx = tid; idx < G * D; idx += kConsumerWarps * 32) {
                const int i = idx / D, dd = idx % D;
                const float M = a.wstate[(size_t)i * (kPartialPad + D) + 3];
                float L = 0.f, O = 0.f;
                if (M != -INFINITY) {
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float *st = a.wstate + ((size_t)w * G + i) * (kPartialPad + D);
                        const float sc = st[2];
                        L = fmaf(sc, st[1], L);
                        O = fmaf(sc, st[kPartialPad + dd], O);
                    }
                }
                unsigned long long *dst = p.partw + ((size_t)(h * G + i) * g.kv_splits + c) * (2 + D);
                const unsigned long long tg = (unsigned long long)tag(cur_layer, kTagPart) << 32;
                if (dd == 0) {
                    st_relaxed_u64(&dst[0], tg | __float_as_uint(M));
                    st_relaxed_u64(&dst[1], tg | __float_as_uint(L));
                }
                st_relaxed_u64(&dst[2 + dd], tg | __float_as_uint(O));
            }
            // wstate is reused by the next item; leave together on any failure
            if (consumer_sync_or(bad)) return;
            if (cur_tr && tid == 0) cur_tr[kTrPartials] = global_timer();
        }
        // Every partial of this task is out; now merge. (A merge polls the other
        // splits of its head, so no merge may come before a partial of the same
        // task: a CTA holding two splits of one head would wait on itself.)
        for (uint32_t it = t.begin; it < t.end; ++it) {
            merge_slice<D, G>((int)(it / (uint32_t)g.kv_splits), (int)(it % (uint32_t)g.kv_splits));
            if (consumer_sync_or(bad)) return;
        }
    }

    // Slice c of KV head h's merged attention output: elements [e0, e1) of its
    // G d outputs, S-th of them per split, from the S partials in split order:
    //   M = max_c m_c, w_c = e^(m_c - M), o = sum_c w_c o_c / sum_c w_c l_c.
    // One thread per (element, split) pair polls that pair's tagged m, l and o
    // into shared memory; then one thread per element merges and writes the
    // tagged bf16 output, which the O-projection tiles gather.
    template <int D, int G>
    __device__ void merge_slice(int h, int c) {
        const Geom &g = p.g;
        const int S = g.kv_splits, n = G * D, per = (n + S - 1) / S;
        const int e0 = c * per, e1 = e0 + per < n ? e0 + per : n;
        if (e0 >= e1) return;
        const int ne = e1 - e0;
        float *st = reinterpret_cast<float *>(s.vec);  // [ne][S][3]: m, l, o
        float *wt = st + (size_t)ne * S * 3;           // [heads of the slice][S]: e^(m_c - M)
        const uint32_t tg = tag(cur_layer, kTagPart);
        for (int q = tid; q < ne * S; q += kConsumerWarps * 32) {
            const int e = e0 + q / S, cc = q % S;
            const unsigned long long *pw = p.partw + ((size_t)(h * G + e / D) * S + cc) * (2 + D);
            unsigned long long wm = ld_relaxed_u64(pw), wl = ld_relaxed_u64(pw + 1),
                               wo = ld_relaxed_u64(pw + 2 + e % D);
            Poll pl;
            while ((uint32_t)(wm >> 32) != tg || (uint32_t)(wl >> 32) != tg || (uint32_t)(wo >> 32) != tg) {
                if (bad || !pl.again(p)) {
                    bad = true;
                    break;
                }
                wm = ld_relaxed_u64(pw);
                wl = ld_relaxed_u64(pw + 1);
                wo = ld_relaxed_u64(pw + 2 + e % D);
            }
            st[q * 3 + 0] = __uint_as_float((uint32_t)wm);
            st[q * 3 + 1] = __uint_as_float((uint32_t)wl);
            st[q * 3 + 2] = __uint_as_float((uint32_t)wo);
        }
        consumer_sync();
        if (cur_tr && tid == 0) cur_tr[kTrMergeIn] = global_timer();
        // m and l belong to a (q head, split), so the weights are taken once per
        // head of the slice, from its first element's staged copies
        const int hq0 = e0 / D, nhq = (e1 - 1) / D - hq0 + 1;
        for (int q = tid; q < nhq * S; q += kConsumerWarps * 32) {
            const int hl = q / S, cc = q % S;
            const int ef = (hq0 + hl) * D > e0 ? (hq0 + hl) * D : e0;
            const float *sq = st + (size_t)(ef - e0) * S * 3;
            float M = -INFINITY;
            for (int c2 = 0; c2 < S; ++c2) M = fmaxf(M, sq[c2 * 3]);
            const float mc = sq[cc * 3];
            wt[q] = mc == -INFINITY ? 0.f : expf(mc - M);
        }
        consumer_sync();
        const uint32_t to = tag(cur_layer, kTagO) << 16;
        for (int q = tid; q < ne; q += kConsumerWarps * 32) {
            const float *sq = st + (size_t)q * S * 3;
            const float *wq = wt + (size_t)((e0 + q) / D - hq0) * S;
            float L = 0.f, O = 0.f;
            for (int cc = 0; cc < S; ++cc) {
                const float w = wq[cc];
                L = fmaf(w, sq[cc * 3 + 1], L);
                O = fmaf(w, sq[cc * 3 + 2], O);
            }
            st_relaxed_u32(p.ow + (size_t)h * n + e0 + q, to | f2bf(__fdiv_rn(O, L)));
        }
    }

    // ---------------------------------------------------------- main loop
    // D (head_dim), G (q heads per KV head) and the weight format (Q8: INT8
    // codes) are compile-time: each kernel instance carries only its own code.
    template <int D, int G, bool Q8, int AK>
    __device__ __forceinline__ void run(int cta) {
        const Geom &g = p.g;
        const int t0 = p.offsets[cta], t1 = p.offsets[cta + 1];
        for (step = 0; step < p.n_steps; ++step) {
            P = p.pos0 + step;
            for (int ti = t0; ti < t1; ++ti) {
                const tiles_task t = p.tasks[ti];
                cur_layer = t.layer;
                // ---- wait for the inputs
                cur_tr = trace_rec(p, cta, step, ti - t0);
                unsigned long long *tr = tid == 0 ? cur_tr : nullptr;
                if (tr) tr[kTrWaitStart] = global_timer();
                if (tid == 0) {
                    const uint32_t target = t.wait_mul * (uint32_t)step + t.wait_add;
                    if (t.wait_ctr != TILES_NO_COUNTER &&
                        !wait_counter(p, p.counters + (size_t)t.wait_ctr * kCounterStride, target))
                        bad = true;
                    if (ti == t0 && !bad) st_release_cta(&s.ctl->step_ready, step);
                    if (!bad && (t.op == TILES_OP_QKV || t.op == TILES_OP_OPROJ) && t.layer == 0) {
                        int tok = token_of_step(step);
                        if (tok < 0 || tok >= g.V) {
                            atomicOr(p.status, kDevBounds);
                            bad = true;
                            tok = 0;
                        }
                        s.ctl->token = tok;
                    }
                }
                if (consumer_sync_or(bad)) return;
                if (tr) tr[kTrWaitEnd] = global_timer();
                // ---- work
                switch (t.op) {
                    case TILES_OP_QKV:
                        if (t.layer > 0) {
                            gather_tagged(p.xw, g.H, tag(t.layer - 1, kTagXFfn));
                            consumer_sync();
                        }
                        rmsnorm_to_vec(t.layer == 0 ? p.embed + (size_t)s.ctl->token * g.H : nullptr,
                                       p.layers[t.layer].attn_norm, g.H);
                        consumer_sync();
                        if (tr) tr[kTrPrologue] = global_timer();
                        gemv_task<1, Q8>(t);
                        break;
                    case TILES_OP_ATTN:
                        attn_task<D, G, AK>(t);
                        break;
                    case TILES_OP_OPROJ:
                        gather_tagged(p.ow, g.qd, tag(t.layer, kTagO));
                        load_residual(t.layer == 0 ? p.embed + (size_t)s.ctl->token * g.H : nullptr,
                                      t.layer == 0 ? 0u : tag(t.layer - 1, kTagXFfn), t.begin, t.end);
                        consumer_sync();
                        if (tr) tr[kTrPrologue] = global_timer();
                        gemv_task<1, Q8>(t);
                        break;
                    case TILES_OP_GATEUP:
                        gather_tagged(p.xw, g.H, tag(t.layer, kTagXAttn));
                        consumer_sync();
                        rmsnorm_to_vec(nullptr, p.layers[t.layer].ffn_norm, g.H);
                        consumer_sync();
                        if (tr) tr[kTrPrologue] = global_timer();
                        gemv_task<2, Q8>(t);
                        break;
                    case TILES_OP_DOWN:
                        gather_tagged(p.aw, g.F, tag(t.layer, kTagA));
                        load_residual(nullptr, tag(t.layer, kTagXAttn), t.begin, t.end);
                        consumer_sync();
                        if (tr) tr[kTrPrologue] = global_timer();
                        gemv_task<1, Q8>(t);
                        break;
                    case TILES_OP_LMHEAD:
                        gather_tagged(p.xw, g.H, tag(g.L - 1, kTagXFfn));
                        consumer_sync();
                        rmsnorm_to_vec(nullptr, p.final_norm, g.H);
                        consumer_sync();
                        if (tr) tr[kTrPrologue] = global_timer();
                        gemv_task<1, Q8>(t);
                        break;
                    default:
                        break;
                }
                // ---- publish
                if (consumer_sync_or(bad)) return;
                if (tr) tr[kTrTaskEnd] = global_timer();
                if (tid == 0 && t.signal_ctr != TILES_NO_COUNTER) {
                    red_release_add(p.counters + (size_t)t.signal_ctr * kCounterStride, 1u);
                }
            }
        }
        // the chosen tokens of this launch
        if (cta == 0 && tid == 0) {
            const uint32_t target = p.final_mul * (uint32_t)p.n_steps;
            if (wait_counter(p, p.counters + (size_t)p.final_ctr * kCounterStride, target)) {
                for (int st = 0; st < p.n_steps; ++st) {
                    const int sg = p.step0 + st;
                    if (sg >= p.n_prompt - 1)
                        p.out_tokens[sg - (p.n_prompt - 1)] = key_row(__ldcg(&p.keys[st]));
                }
            }
        }
    }
};

// AK, the attention kind: 0 shared chunks only; 1 also one warp per chunk for
// long splits; 2 INT8 KV cache. Every form runs on the tensor cores.
template <int D, int G, bool Q8, int AK>
__global__ void __launch_bounds__(kThreads, 1) tiles_megakernel(const __grid_constant__ KernelParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem s = smem_layout(smem_raw, p);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int i = 0; i < p.g.ring_slots; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        s.ctl->unused = 0;
        s.ctl->token = 0;
        s.ctl->step_ready = 0;
        s.ctl->stream_pos = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid >= (kConsumerWarps + kProducerWarps) * 32) {
        if (p.l2_prefetch_bytes) {
            Prefetcher pf(p, s);
            pf.run(blockIdx.x);
        }
        return;
    }
    if (tid >= kConsumerWarps * 32) {
        if ((tid & 31) == 0) {
            Producer prod(p, s, (tid >> 5) - kConsumerWarps);
            prod.template run<AK>(blockIdx.x);
        }
        return;
    }
    Consumer cons(p, s, tid);
    cons.template run<D, G, Q8, AK>(blockIdx.x);
}

}  // namespace tiles

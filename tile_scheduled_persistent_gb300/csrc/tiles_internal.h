// Internal definitions shared by the host planner and the persistent kernel:
// chunk geometry (which bytes a task streams, in which ring slot), the kernel
// parameter block and device-side status codes. Everything here is computed
// identically on the host (planner, validator, byte counts) and the device
// (producer and consumer warps), so both sides agree on the chunk sequence.
#pragma once

#include <stdint.h>

#include "../../include/tiles.h"

#ifdef __CUDACC__
#define TILES_HD __host__ __device__ __forceinline__
#else
#define TILES_HD inline
#endif

namespace tiles {

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarps = 2;  // lane 0 of each issues the copies of every other ring slot
constexpr int kPrefetchWarps = 1;
constexpr int kThreads = (kConsumerWarps + kProducerWarps + kPrefetchWarps) * 32;
constexpr int kMaxRowsPerChunk = 8;                   // GEMV rows a warp handles per chunk
constexpr int kMaxSlots = 32;
constexpr int kSmemLimit = 232448;                    // 227 KB dynamic shared memory per CTA
constexpr int kCtlBytes = 1024;                       // mbarriers + control block
constexpr int kPhaseKinds = 6;                        // QKV, ATTN, COMBINE, O, GATEUP, DOWN
constexpr int kMaxStepsPerLaunch = 64;
constexpr int kCodeOffset = 128;                      // a plan stores INT8 code q as the byte q + 128
constexpr int kCounterStride = 32;                    // u32 words: one 128-byte line per counter
constexpr int kPartialPad = 4;                        // (m, l, -, -) ahead of o[d] in a partial

// device status word bits
constexpr uint32_t kDevTimeout = 1u;
constexpr uint32_t kDevBounds = 2u;

// Shapes derived from the model description and the resolved options.
struct Geom {
    int L, H, nq, nkv, d, F, V, max_pos, G, qd, kvd, qkv_rows;
    int slot_bytes, ring_slots, kv_splits, kv_block;
    int rpc_qkv, rpc_o, rpc_gateup, rpc_down, rpc_lm;
    int wbytes;     // bytes per streamed weight: 2 (BF16) or 1 (INT8 codes)
    int vec_bytes;  // shared-memory region for the input vector / attention scratch
    int res_off;    // in the vec region: residual rows of an O-proj / down tile
    int smem_bytes;
    int attn_mma;   // 1: some attention split can reach kConsumerWarps chunks, and the
                    // kernel instance carries the tensor-core owner form for them
    int kv8;        // 1: INT8 KV cache (every attention chunk on the tensor-core path)
    int kv_mp;      // INT8 cache: position stride (max_pos rounded up to 16)
};

// INT8 KV chunk: kv_block = 8192 / d positions (128 at d = 64, 64 at d = 128):
// key codes [kv_block][d], value codes transposed [d][kv_block], then the
// key and value scales, kv_block floats each.
TILES_HD int kv8_block(int d) { return 8192 / d; }
TILES_HD int kv8_chunk_bytes(int d) { return 2 * 8192 + 2 * kv8_block(d) * 4; }

TILES_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

TILES_HD int phase_of_op(int op) {
    switch (op) {
        case TILES_OP_QKV: return 0;
        case TILES_OP_ATTN: return 1;
        case TILES_OP_COMBINE: return 2;
        case TILES_OP_OPROJ: return 3;
        case TILES_OP_GATEUP: return 4;
        case TILES_OP_DOWN: return 5;
        case TILES_OP_LMHEAD: return 6;
        default: return -1;
    }
}

// Global phase index of (layer, kind) within one step; the LM head is last.
TILES_HD int phase_index(const Geom &g, int layer, int kind) {
    return kind == 6 ? kPhaseKinds * g.L : kPhaseKinds * layer + kind;
}

TILES_HD int phases_per_step(const Geom &g) { return kPhaseKinds * g.L + 1; }

// Rows (GEMV ops) or items (attention: kv head * splits + split; combine: q head).
TILES_HD int op_extent(const Geom &g, int op) {
    switch (op) {
        case TILES_OP_QKV: return g.qkv_rows;
        case TILES_OP_ATTN: return g.nkv * g.kv_splits;
        case TILES_OP_COMBINE: return 0;  // merged into the attention tiles (each merges 1/S)
        case TILES_OP_OPROJ: return g.H;
        case TILES_OP_GATEUP: return g.F;
        case TILES_OP_DOWN: return g.H;
        case TILES_OP_LMHEAD: return g.V;
        default: return 0;
    }
}

// Length (elements) of the input vector of a GEMV op.
TILES_HD int op_in_dim(const Geom &g, int op) {
    switch (op) {
        case TILES_OP_QKV: return g.H;
        case TILES_OP_OPROJ: return g.qd;
        case TILES_OP_GATEUP: return g.H;
        case TILES_OP_DOWN: return g.F;
        case TILES_OP_LMHEAD: return g.H;
        default: return 0;
    }
}

TILES_HD int op_mats(int op) { return op == TILES_OP_GATEUP ? 2 : 1; }

TILES_HD bool op_is_gemv(int op) {
    return op == TILES_OP_QKV || op == TILES_OP_OPROJ || op == TILES_OP_GATEUP ||
           op == TILES_OP_DOWN || op == TILES_OP_LMHEAD;
}

TILES_HD int op_rows_per_chunk(const Geom &g, int op) {
    switch (op) {
        case TILES_OP_QKV: return g.rpc_qkv;
        case TILES_OP_OPROJ: return g.rpc_o;
        case TILES_OP_GATEUP: return g.rpc_gateup;
        case TILES_OP_DOWN: return g.rpc_down;
        case TILES_OP_LMHEAD: return g.rpc_lm;
        default: return 0;
    }
}

// Split c of the n_pos positions 0..n_pos-1 covers KV blocks [*b0, *b1).
TILES_HD void attn_split_blocks(const Geom &g, int n_pos, int c, int *b0, int *b1) {
    int nb = ceil_div(n_pos, g.kv_block);
    *b0 = (int)(((long long)c * nb) / g.kv_splits);
    *b1 = (int)(((long long)(c + 1) * nb) / g.kv_splits);
}

// Number of ring chunks a task streams at context position P (0-based).
TILES_HD int task_chunks(const Geom &g, const tiles_task &t, int P) {
    if (op_is_gemv(t.op)) return ceil_div((int)(t.end - t.begin), op_rows_per_chunk(g, t.op));
    if (t.op == TILES_OP_ATTN) {
        int n = 0;
        for (uint32_t it = t.begin; it < t.end; ++it) {
            int b0, b1;
            attn_split_blocks(g, P + 1, (int)(it % (uint32_t)g.kv_splits), &b0, &b1);
            n += b1 - b0;
        }
        return n;
    }
    return 0;
}

// Bytes a task streams from HBM at position P (weights, or K/V of positions < P).
TILES_HD long long task_bytes(const Geom &g, const tiles_task &t, int P) {
    if (op_is_gemv(t.op))
        return (long long)(t.end - t.begin) * op_in_dim(g, t.op) * g.wbytes * op_mats(t.op);
    if (t.op == TILES_OP_ATTN) {
        long long n = 0;
        for (uint32_t it = t.begin; it < t.end; ++it) {
            int b0, b1;
            attn_split_blocks(g, P + 1, (int)(it % (uint32_t)g.kv_splits), &b0, &b1);
            int p0 = b0 * g.kv_block, p1 = b1 * g.kv_block;
            if (p1 > P) p1 = P;
            if (p1 > p0) n += (long long)(p1 - p0) * (g.kv8 ? 2 * g.d + 8 : g.d * 2 * 2);
        }
        return n;
    }
    return 0;
}

// Device copy of one layer's pointers. The streamed weights are rows of
// g.wbytes-byte elements: qkv = [Wq; Wk; Wv] as one [qd + 2 kvd][H] matrix and
// gu = Wg / Wu interleaved by row ([F][2][H]: gate row r, then up row r), both
// plan-packed so every ring chunk of those tiles is one contiguous bulk copy;
// o = Wo [H][qd], down = Wd [H][F]. With INT8 weights every streamed row has
// an FP32 scale (s_gu in the interleaved row order); with BF16 they are null.
struct LayerPtrs {
    const uint16_t *attn_norm, *q_norm, *k_norm, *ffn_norm;
    const uint8_t *qkv, *o, *gu, *down;
    const float *s_qkv, *s_o, *s_gu, *s_down;
};

// An opaque CUDA tensor map (CUtensorMap: 128 bytes, 128-byte aligned),
// declared here so the host planner compiles without the driver headers.
struct alignas(128) TensorMap {
    uint64_t opaque[16];
};

struct KernelParams {
    Geom g;
    float eps, attn_scale;
    int qk_norm;
    // schedule
    const tiles_task *tasks;
    const int32_t *offsets;
    int final_ctr;
    uint32_t final_mul;
    // weights
    const LayerPtrs *layers;
    const uint16_t *embed, *final_norm;   // BF16 embedding table (the lookup) and final gain
    const uint8_t *lm;                    // LM-head rows as streamed: the embedding, or its INT8 codes
    const float *lm_s;                    // INT8: their scales (null for BF16)
    const float *rope_cos, *rope_sin;  // [max_pos][d/2]
    // caches and scratch
    uint16_t *k_cache, *v_cache;
    // INT8 KV cache (kv8): key codes [Z][kv_mp][d], value codes [Z][d][kv_mp],
    // scales [Z][kv_mp], key shifts [Z][d] (Z = L n_kv)
    int8_t *kq8, *vq8;
    float *ks8, *vs8;
    const float *mu8;
    // tagged activations: (tag << 16) | bf16 for the residual stream x [H],
    // the SwiGLU output a [F] and the attention output o [nq d];
    // (tag << 32) | f32 bits for the Q/K/V rows and the split partials
    // [nq][S][2 + d] (m, l, o of each q head and split)
    uint32_t *xw, *aw, *ow;
    unsigned long long *qkvw, *partw;
    unsigned long long *keys;
    uint32_t *counters, *status;
    // run
    const int32_t *prompt;
    int n_prompt, step0, pos0, n_steps;
    int32_t *out_tokens;
    float *out_logits;
    unsigned long long timeout_ns;
    unsigned long long l2_prefetch_bytes;  // L2 lookahead of the weight stream per CTA (0: off)
    unsigned long long l2_prefetch_ns_per_4k;  // pacing of the prefetch warp (0: unpaced)
    int vec_off, ring_off, res_off;
    // optional per-task timeline: [cta][step < trace_steps][task][kTraceWords]
    unsigned long long *trace;
    int trace_steps, trace_tasks;
    // TMA descriptors (written per decode call; the kernel takes their
    // addresses in parameter space). BF16 cache: [0] K and [1] V as
    // [L * n_kv][max_pos][d], boxes of kv_block positions x 64 dims, 128-byte
    // swizzle. INT8 cache: [0] key codes (box kv_block x d), [1] value codes
    // (box d x kv_block), both swizzled by their row length (64 or 128
    // bytes); [2] key and [3] value scales (box kv_block).
    TensorMap kv_map[4];
};

// trace record words
constexpr int kTraceWords = 16;

// Attention chunks arrive as 128-byte-swizzled TMA tiles of whole KV blocks
// (a multiple of 16 positions) and are reduced on the tensor cores. A split of
// at least kConsumerWarps chunks gives each chunk to its slot's owner warp, in
// rounds of 2048 / d positions (32 at d = 64, 16 at d = 128, so the block must
// be a multiple of that; kernel instances compiled with the owner form only);
// a shorter split shares its chunks across all warps, one 16-position block
// per warp and round. Producer and consumers decide with the same rule.
TILES_HD bool attn_owner(const Geom &g, int n_chunks) { return g.attn_mma && n_chunks >= kConsumerWarps; }
// The kernel instance a plan runs: 0 shared-chunk attention only, 1 also the
// one-warp-per-chunk form for long splits, 2 INT8 KV cache.
TILES_HD int attn_kind(const Geom &g) { return g.kv8 ? 2 : g.attn_mma; }

enum { kTrWaitStart = 0, kTrWaitEnd, kTrTaskEnd, kTrProdFirst, kTrProdLast, kTrProdStall,
       kTrOpInfo, kTrPrologue, kTrFirstChunk, kTrPartials, kTrMergeIn };

}  // namespace tiles

// schedule object (host)
#include <string>
#include <vector>
struct tiles_schedule_s {
    tiles_model_desc desc;
    tiles_plan_opts opts;
    tiles::Geom geom;
    int n_ctas = 0;
    int scheduler = 0;
    int n_counters = 0;
    int final_ctr = 0;
    uint32_t final_mul = 0;
    std::vector<tiles_task> tasks;
    std::vector<int32_t> offsets;
};

namespace tiles {
// planner entry points used by the runtime
tiles_status_t resolve_geom(const tiles_model_desc &d, const tiles_plan_opts &o, int n_ctas,
                            int smem_limit, Geom *g, std::string *why);
tiles_status_t build_schedule(const tiles_model_desc &d, const tiles_plan_opts &o, int n_ctas,
                              int smem_limit, tiles_schedule_s *s, std::string *why);
tiles_status_t validate_schedule(const tiles_schedule_s &s, std::string *why);
tiles_plan_opts default_opts();
}  // namespace tiles
